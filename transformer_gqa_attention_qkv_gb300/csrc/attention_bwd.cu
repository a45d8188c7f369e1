// attention_bwd.cu -- backward of the causal grouped-query attention on
// tcgen05 (head_dim 64, 80, 96 and 128).
//
// With P = softmax(s), s = <q, k> / sqrt(d), o = P v and dO the gradient of
// the attention output (the derivatives of [T07] §4 step 6; K and V of a KV
// head receive the gradients of every query head of its group, [Part]):
//   dP = dO V^T,   D_t = <dO_t, O_t>,   dS = P o (dP - D),
//   dV = P^T dO,   dK = dS^T Q / sqrt(d),   dQ = dS K / sqrt(d).
// P is recomputed from Q, K and the forward's per-row log2-sum-exp, never
// stored.  Two kernels, so that no gradient needs atomics:
//   dkdv: one CTA per (sequence, KV head, 128-key block); it walks the query
//         tiles that see the block.  Keys sit in the MMA rows, so S^T = K Q^T
//         and dP^T = V dO^T land in TMEM with one key per lane; P^T and dS^T
//         are written back over them in 16-bit and are the TMEM A operands of
//         dV += P^T dO and dK += dS^T Q.  The G query heads of the group are
//         packed into the 128 query rows of a tile (as in the forward), so the
//         sum over the group's heads is part of the contraction.
//   dq:   one CTA per (sequence, KV head, query tile); it walks the key blocks
//         the tile sees: S = Q K^T, dP = dO V^T, dS in 16-bit over S, and
//         dQ += dS K.
// Both: warp 0 TMA, warp 1 MMA issue, and two warpgroups for the elementwise
// step, one TMEM lane (one key, or one query row) per thread.  Each streamed
// tile is processed in two halves of 64 rows with separate TMEM buffers, one
// warpgroup per half, so the tensor core computes one half while the other's
// P and dS are formed.  Q, K, V and dO are binary16 (head-major), so P and dS
// are binary16 as well.  Head widths 80 and 96 are staged as 128-wide rows
// whose columns past d the tensor copy fills with zeros: S and dP contract over
// the d real columns, the accumulating products run 128 wide (the zero columns
// give zero gradient columns) and only d columns are stored.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kRows = 128;      // query rows of a tile, keys of a block
constexpr int kHalf = 64;       // streamed rows of one pipeline half
constexpr int kThreads = 320;   // warp 0 TMA, warp 1 MMA, warps 2..9 two elementwise warpgroups

struct BwdParams {
    int B, S, Hq, Hkv, G, R, n_qt, n_kb, causal;
    float scale_log2;  // log2(e) / sqrt(d)
    float scale;       // 1 / sqrt(d)
    const float *lse;  // [B, Hq, S]
    const float *dsum; // [B, Hq, S]: D = <dO, O>
    float *dq;         // [B, Hq, S, d]
    float *dk, *dv;    // [B, Hkv, S, d]
    unsigned *err;
};

template <int D>
struct BSmem {
    static constexpr int NCH = (D + 63) / 64;     // 64-wide d chunks (80 and 96: two, the second part zero)
    static constexpr int DP = NCH * 64;           // the staged width
    static constexpr int CH = kRows * 128;        // 128 rows x 64 16-bit values (16 KB)
    static constexpr int TILE = NCH * CH;          // one 128-row tile of d values
    // dkdv: K, V kept; Q, dO rings of 2; lse/D rings of 2 x 2 x 128 floats
    // dq:   Q, dO kept;  K, V rings of 2; lse/D once
    static constexpr int A0 = 0;                   // K (dkdv) or Q (dq)
    static constexpr int A1 = A0 + TILE;           // V (dkdv) or dO (dq)
    static constexpr int RING = A1 + TILE;         // 2 stages x (2 tiles)
    static constexpr int ROWS = RING + 2 * 2 * TILE;  // 2 stages x (lse, D) x 128 floats
    static constexpr int BARS = ROWS + 2 * 2 * kRows * 4;
    static constexpr int NBARS = 10;
    static constexpr int TMEM_SLOT = BARS + NBARS * 8;
    static constexpr int COLS = TMEM_SLOT + 16;   // dkdv: position of each packed query row in its tile, -1: none
    static constexpr int TOTAL = COLS + kRows * 4;
    static constexpr int ALLOC = TOTAL + 1024;
};

// D = <dO, O> per (b, head, t): one warp per row.  dO head-major binary16,
// O token-major bf16 (the forward's attention output).
template <int D>
__global__ void __launch_bounds__(256) dsum_kernel(const uint16_t *dO, const uint16_t *O, float *dsum, int ld, int B,
                                                   int S, int Hq)
{
    const long row = (long)blockIdx.x * 8 + threadIdx.x / 32;  // (b*Hq + j)*S + t
    const int lane = threadIdx.x % 32;
    if (row >= (long)B * Hq * S) return;
    const long t = row % S, bj = row / S;
    const long j = bj % Hq, b = bj / Hq;
    const uint16_t *g = dO + row * D;
    const uint16_t *o = O + ((b * S + t) * Hq + j) * D;
    float acc = 0.0f;
#pragma unroll
    for (int c = lane * 2; c < D; c += 64) {
        const float2 gv = __half22float2(*reinterpret_cast<const __half2 *>(g + c));
        const uint32_t ov = *reinterpret_cast<const uint32_t *>(o + c);
        acc = fmaf(gv.x, bf16lo(ov), fmaf(gv.y, bf16hi(ov), acc));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) dsum[bj * ld + t] = acc;
}

// TMEM -> registers: 64 consecutive columns at ta and 64 at tb (32 lanes x
// 32 bits), both loads in flight together; the wait is part of the statement
// so no use of a or b is scheduled before the data has arrived.
DEVI void tmem_ld64x2(uint32_t ta, uint32_t tb, uint32_t (&a)[64], uint32_t (&b)[64])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%129];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        :
          "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
          "=r"(a[16]), "=r"(a[17]), "=r"(a[18]), "=r"(a[19]), "=r"(a[20]), "=r"(a[21]), "=r"(a[22]), "=r"(a[23]),
          "=r"(a[24]), "=r"(a[25]), "=r"(a[26]), "=r"(a[27]), "=r"(a[28]), "=r"(a[29]), "=r"(a[30]), "=r"(a[31]),
          "=r"(a[32]), "=r"(a[33]), "=r"(a[34]), "=r"(a[35]), "=r"(a[36]), "=r"(a[37]), "=r"(a[38]), "=r"(a[39]),
          "=r"(a[40]), "=r"(a[41]), "=r"(a[42]), "=r"(a[43]), "=r"(a[44]), "=r"(a[45]), "=r"(a[46]), "=r"(a[47]),
          "=r"(a[48]), "=r"(a[49]), "=r"(a[50]), "=r"(a[51]), "=r"(a[52]), "=r"(a[53]), "=r"(a[54]), "=r"(a[55]),
          "=r"(a[56]), "=r"(a[57]), "=r"(a[58]), "=r"(a[59]), "=r"(a[60]), "=r"(a[61]), "=r"(a[62]), "=r"(a[63]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
          "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15]),
          "=r"(b[16]), "=r"(b[17]), "=r"(b[18]), "=r"(b[19]), "=r"(b[20]), "=r"(b[21]), "=r"(b[22]), "=r"(b[23]),
          "=r"(b[24]), "=r"(b[25]), "=r"(b[26]), "=r"(b[27]), "=r"(b[28]), "=r"(b[29]), "=r"(b[30]), "=r"(b[31]),
          "=r"(b[32]), "=r"(b[33]), "=r"(b[34]), "=r"(b[35]), "=r"(b[36]), "=r"(b[37]), "=r"(b[38]), "=r"(b[39]),
          "=r"(b[40]), "=r"(b[41]), "=r"(b[42]), "=r"(b[43]), "=r"(b[44]), "=r"(b[45]), "=r"(b[46]), "=r"(b[47]),
          "=r"(b[48]), "=r"(b[49]), "=r"(b[50]), "=r"(b[51]), "=r"(b[52]), "=r"(b[53]), "=r"(b[54]), "=r"(b[55]),
          "=r"(b[56]), "=r"(b[57]), "=r"(b[58]), "=r"(b[59]), "=r"(b[60]), "=r"(b[61]), "=r"(b[62]), "=r"(b[63])
        : "r"(ta), "r"(tb)
        : "memory");
}

// P and dS for the 64 columns of one pipeline half in this thread's TMEM
// lane: S (or S^T) at tS, dP (or dP^T) at tdP.  DKDV: each column is a query
// row with its own log2-sum-exp and D (lse_c[i], dsum_c[i]); else the lane is
// the query row (lse_r, dsum_r).  Writes two binary16 values per column over
// columns this thread has already read: DKDV P over S and dS over dP (the A
// operands of dV += P^T dO and dK += dS^T Q); else dS over S (the A operand of
// dQ += dS K).  MASK: valid(i) says whether column i is a visible pair;
// invisible pairs get P = dS = 0.
template <bool DKDV, bool MASK, typename Valid>
DEVI void p_ds64(uint32_t tS, uint32_t tdP, float sl, const float *lse_c, const float *dsum_c, float lse_r,
                 float dsum_r, Valid valid)
{
    uint32_t s[64], gr[64];
    tmem_ld64x2(tS, tdP, s, gr);
    const float2 sl2 = make_float2(sl, sl);
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int i = 32 * hh + 2 * e;
            float2 nl, nd;
            if (DKDV) {
                const float2 l = *reinterpret_cast<const float2 *>(lse_c + i);
                const float2 dd = *reinterpret_cast<const float2 *>(dsum_c + i);
                nl = make_float2(-l.x, -l.y);
                nd = make_float2(-dd.x, -dd.y);
            } else {
                nl = make_float2(-lse_r, -lse_r);
                nd = make_float2(-dsum_r, -dsum_r);
            }
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[i]), __uint_as_float(s[i + 1])), sl2, nl);
            float2 p = make_float2(ex2(x.x), ex2(x.y));
            if (MASK) {
                if (!valid(i)) p.x = 0.0f;
                if (!valid(i + 1)) p.y = 0.0f;
            }
            const float2 ds =
                __fmul2_rn(p, __fadd2_rn(make_float2(__uint_as_float(gr[i]), __uint_as_float(gr[i + 1])), nd));
            pk[e] = pack_f16(p.x, p.y);
            dk[e] = pack_f16(ds.x, ds.y);
        }
        if (DKDV) {
            tmem_st16_nowait(tS + 16 * hh, pk);
            tmem_st16_nowait(tdP + 16 * hh, dk);
        } else {
            tmem_st16_nowait(tS + 16 * hh, dk);
        }
    }
    tmem_st_wait();
}

// One CTA of either backward kernel.
//   DKDV: (b, KV head g, 128-key block kb); keeps K, V; streams the Q / dO
//         tiles (with their lse / D rows) of the query tiles that see the block.
//   else: (b, KV head g, query tile); keeps Q, dO and the tile's lse / D;
//         streams the K / V blocks the tile sees.
// Each streamed item is taken in two halves of 64 rows, h = 0, 1, each with
// its own S / dP buffers in TMEM (columns [128h, 128h + 64) and
// [128h + 64, 128h + 128)) and its own warpgroup for the elementwise step
// (warps 2..5 for h = 0, 6..9 for h = 1), so the tensor core works on one half
// while the other half's P and dS are formed.  Accumulators (DP: d rounded up
// to 64): dV, dK at [256, 256 + DP), [256 + DP, 256 + 2 DP) (DKDV) or dQ at
// [256, 256 + DP).
// MMA order per item i: acc(i, 0), S(i + 1, 0), acc(i, 1), S(i + 1, 1), where
// S(i, h) is S and dP of half h and acc(i, h) the products that consume P and
// dS of half h.  The MMAs of one CTA run in issue order, so S(i + 1, h) reuses
// the columns acc(i, h) reads.
// PACKED: G*R = 128 (G a power of two), every row of a query tile a real
// query (the masks are index arithmetic); otherwise rows past G*R are padding.
template <int D, bool DKDV, bool PACKED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                    const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                    const BwdParams P)
{
    using L = BSmem<D>;
    constexpr int NCH = L::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *fix_full = bars, *ring_full = bars + 1, *ring_empty = bars + 3, *s_full = bars + 5, *p_full = bars + 7,
             *acc_done = bars + 9;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::TMEM_SLOT);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;

    const int bh = blockIdx.x % (P.B * P.Hkv), slot = blockIdx.x / (P.B * P.Hkv);
    const int b = bh / P.Hkv, g = bh % P.Hkv;
    const int qhead = b * P.Hq + g * P.G, kvhead = b * P.Hkv + g;
    // DKDV: heavy (early) key blocks first, they are seen by the most query
    // tiles; else heavy (late) query tiles first
    int u0 = 0, qt0 = 0, t0 = 0, n_it;
    if (DKDV) {
        u0 = slot * kRows;
        qt0 = P.causal ? u0 / P.R : 0;  // first query tile that sees a key of the block
        n_it = max(0, P.n_qt - qt0);
    } else {
        t0 = (P.n_qt - 1 - slot) * P.R;
        const int t_last = min(t0 + P.R, P.S) - 1;
        n_it = P.causal ? t_last / kRows + 1 : P.n_kb;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) mbar_init(bars + i, 1);
        mbar_init(p_full, 4);
        mbar_init(p_full + 1, 4);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmG);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    // A tile packs G heads x R positions = G*R <= 128 query rows.  dkdv: its
    // query rows are the columns of S^T and dP^T and are summed over in dV and
    // dK, so the ring's Q and dO rows and lse and D entries past G*R (never
    // written by the tensor copies) are zeroed once (finite S, dP and D there,
    // so P = 0 from the column table's mask gives dS = 0), and the column
    // table marks them.
    int *colpos = reinterpret_cast<int *>(smem + L::COLS);
    if (DKDV && !PACKED) {
        const int packed = P.G * P.R;
        for (int i = threadIdx.x; i < kRows; i += kThreads) colpos[i] = i < packed ? i - (i / P.R) * P.R : -1;
        const int pad = kRows - packed;
        float *rows_all = reinterpret_cast<float *>(smem + L::ROWS);  // [stage][lse, D][128]
        for (int idx = threadIdx.x; idx < 2 * 2 * pad; idx += kThreads)
            rows_all[(idx / pad) * kRows + packed + idx % pad] = 0.0f;
        for (int idx = threadIdx.x; idx < 2 * 2 * NCH * pad * 8; idx += kThreads) {
            int rest = idx / 8;
            const int unit = idx % 8, row = packed + rest % pad;
            rest /= pad;
            const int c = rest % NCH, tile = rest / NCH;  // tile: stage * 2 + (Q or dO)
            *reinterpret_cast<uint4 *>(smem + L::RING + tile * L::TILE + c * L::CH + row * 128 + unit * 16) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the tensor core reads these rows through the async proxy
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    float *rows0 = reinterpret_cast<float *>(smem + L::ROWS);

    if (warp == 0) {
        if (lane == 0) {
            // a query tile's copies bring its G*R packed rows (of Q, dO, lse and D) only
            const uint32_t packed = (uint32_t)(P.G * P.R);
            const uint32_t qtile = NCH * 128 * packed, qrows = 2 * packed * 4;
            mbar_arrive_expect_tx(fix_full, DKDV ? 2 * L::TILE : 2 * qtile + qrows);
            for (int c = 0; c < NCH; ++c) {
                if (DKDV) {
                    tma_load_3d(smem + L::A0 + c * L::CH, &tmK, c * 64, u0, kvhead, fix_full);
                    tma_load_3d(smem + L::A1 + c * L::CH, &tmV, c * 64, u0, kvhead, fix_full);
                } else {
                    tma_load_3d(smem + L::A0 + c * L::CH, &tmQ, c * 64, t0, qhead, fix_full);
                    tma_load_3d(smem + L::A1 + c * L::CH, &tmG, c * 64, t0, qhead, fix_full);
                }
            }
            if (!DKDV) {
                tma_load_2d(rows0, &tmL, t0, qhead, fix_full);
                tma_load_2d(rows0 + kRows, &tmD, t0, qhead, fix_full);
            }
            int it = 0;
            for (; it < n_it; ++it) {
                const int s = it & 1;
                if (!mbar_wait(ring_empty + s, ((it >> 1) & 1) ^ 1, err)) break;
                mbar_arrive_expect_tx(ring_full + s, DKDV ? 2 * qtile + qrows : 2 * L::TILE);
                uint8_t *st = smem + L::RING + s * 2 * L::TILE;
                if (DKDV) {
                    const int tt = (qt0 + it) * P.R;
                    for (int c = 0; c < NCH; ++c) {
                        tma_load_3d(st + c * L::CH, &tmQ, c * 64, tt, qhead, ring_full + s);
                        tma_load_3d(st + L::TILE + c * L::CH, &tmG, c * 64, tt, qhead, ring_full + s);
                    }
                    float *rows = rows0 + s * 2 * kRows;
                    tma_load_2d(rows, &tmL, tt, qhead, ring_full + s);
                    tma_load_2d(rows + kRows, &tmD, tt, qhead, ring_full + s);
                } else {
                    for (int c = 0; c < NCH; ++c) {
                        tma_load_3d(st + c * L::CH, &tmK, c * 64, it * kRows, kvhead, ring_full + s);
                        tma_load_3d(st + L::TILE + c * L::CH, &tmV, c * 64, it * kRows, kvhead, ring_full + s);
                    }
                }
            }
            // no copy may still be in flight when the CTA exits
            mbar_wait(fix_full, 0, err);
            for (int j = max(0, it - 2); j < it; ++j) mbar_wait(ring_full + (j & 1), (j >> 1) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(kRows, kHalf, 0, 0);  // 128 kept rows x 64 streamed rows
            constexpr uint32_t idesc_a = idesc_f16_f32(kRows, L::DP, 0, 1);  // 128 x DP, B MN-major (d contiguous)
            const uint32_t sA0 = smem_u32(smem + L::A0), sA1 = smem_u32(smem + L::A1);
            const uint32_t sRing = smem_u32(smem + L::RING);
            // S = A0 R0_h^T and dP = A1 R1_h^T for half h of item it: DKDV
            // S^T = K Q_h^T, dP^T = V dO_h^T; else S = Q K_h^T, dP = dO V_h^T
            auto issue_s = [&](int it, int h) {
                const uint32_t r0 = sRing + (it & 1) * 2 * L::TILE + h * kHalf * 128, r1 = r0 + L::TILE;
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        if (c * 64 + k * 16 >= D) continue;  // d real columns, 16 per step
                        umma_f16_ss(tmem + 128 * h, sw128_desc(sA0 + c * L::CH + 32 * k, 16, 1024),
                                    sw128_desc(r0 + c * L::CH + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                        umma_f16_ss(tmem + 128 * h + 64, sw128_desc(sA1 + c * L::CH + 32 * k, 16, 1024),
                                    sw128_desc(r1 + c * L::CH + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                    }
                umma_commit(s_full + h);
            };
            // the accumulating products of half h (16 streamed rows = 8 packed TMEM columns per step)
            auto issue_acc = [&](int it, int h) {
                const uint32_t r0 = sRing + (it & 1) * 2 * L::TILE + h * kHalf * 128, r1 = r0 + L::TILE;
#pragma unroll
                for (int k = 0; k < kHalf / 16; ++k) {
                    const uint32_t acc = (it | h | k) != 0;
                    if (DKDV) {
                        umma_f16_ts(tmem + 256, tmem + 128 * h + 8 * k, sw128_desc(r1 + k * 16 * 128, L::CH, 1024),
                                    idesc_a, acc);  // dV += P^T dO
                        umma_f16_ts(tmem + 256 + L::DP, tmem + 128 * h + 64 + 8 * k,
                                    sw128_desc(r0 + k * 16 * 128, L::CH, 1024), idesc_a, acc);  // dK += dS^T Q
                    } else {
                        umma_f16_ts(tmem + 256, tmem + 128 * h + 8 * k, sw128_desc(r0 + k * 16 * 128, L::CH, 1024),
                                    idesc_a, acc);  // dQ += dS K
                    }
                }
            };
            bool ok = mbar_wait(fix_full, 0, err) && n_it > 0 && mbar_wait(ring_full, 0, err);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(0, 1);
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const bool next = it + 1 < n_it;
                if (!mbar_wait(p_full, it & 1, err)) break;
                tc_fence_after();
                issue_acc(it, 0);
                if (next) {
                    if (!mbar_wait(ring_full + ((it + 1) & 1), ((it + 1) >> 1) & 1, err)) break;
                    tc_fence_after();
                    issue_s(it + 1, 0);
                }
                if (!mbar_wait(p_full + 1, it & 1, err)) break;
                tc_fence_after();
                issue_acc(it, 1);
                umma_commit(ring_empty + (it & 1));
                if (next) issue_s(it + 1, 1);
            }
            umma_commit(acc_done);
            mbar_wait(acc_done, 0, err);
        }
    } else {
        const int h = (warp - 2) >> 2;     // pipeline half of this warpgroup
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane; // TMEM lane: key u0 + r (DKDV) or packed query row r
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off + 128 * h, tdP = tS + 64;
        const float sl = P.scale_log2;
        const int u = u0 + r;
        const int hl = r / P.R, t = t0 + (PACKED ? (r & (P.R - 1)) : r - hl * P.R);
        const bool row_ok = (PACKED || hl < P.G) && t < P.S;  // dq: a query row of the tile
        // a wait's outcome is made warp-uniform, so that a timeout never
        // leaves part of a warp before a warp-collective TMEM access
        auto wait_all = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
        };
        bool ok = DKDV || wait_all(fix_full, 0);
        const float my_lse = DKDV ? 0.0f : rows0[r], my_d = DKDV ? 0.0f : rows0[kRows + r];
        for (int it = 0; ok && it < n_it; ++it) {
            if (!wait_all(s_full + h, it & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (DKDV) {
                const int s = it & 1, tt = (qt0 + it) * P.R;
                // the item's lse / D rows came with its Q / dO tiles
                if (!wait_all(ring_full + s, (it >> 1) & 1)) {
                    ok = false;
                    break;
                }
                const float *rows = rows0 + s * 2 * kRows + kHalf * h;
                // every (key, query) pair of the half visible: the whole block at
                // or before the first position of the tile, no ragged edge
                const bool full = PACKED && (!P.causal || u0 + kRows - 1 <= tt) && tt + P.R <= P.S &&
                                  u0 + kRows <= P.S;
                if (full) {
                    p_ds64<true, false>(tS, tdP, sl, rows, rows + kRows, 0.0f, 0.0f, [](int) { return true; });
                } else if (PACKED) {
                    // column i: packed query row 64h + i at position tt + ((64h + i) mod R)
                    const int rmask = P.R - 1;  // R = 128 / G is a power of two
                    auto valid = [&](int i) {
                        const int tq = tt + ((kHalf * h + i) & rmask);
                        return tq < P.S && u < P.S && (!P.causal || u <= tq);
                    };
                    p_ds64<true, true>(tS, tdP, sl, rows, rows + kRows, 0.0f, 0.0f, valid);
                } else {
                    // column i: packed query row 64h + i at position tt + ((64h + i) mod R), if any
                    auto valid = [&](int i) {
                        const int po = colpos[kHalf * h + i];
                        const int tq = tt + po;
                        return po >= 0 && tq < P.S && u < P.S && (!P.causal || u <= tq);
                    };
                    p_ds64<true, true>(tS, tdP, sl, rows, rows + kRows, 0.0f, 0.0f, valid);
                }
            } else {
                const int k0 = it * kRows + kHalf * h;  // key of column 0 of the half
                const bool full = (!P.causal || k0 + kHalf - 1 <= t0) && k0 + kHalf <= P.S && t0 + P.R <= P.S;
                if (full) {
                    p_ds64<false, false>(tS, tdP, sl, nullptr, nullptr, my_lse, my_d, [](int) { return true; });
                } else {
                    auto valid = [&](int i) {
                        const int uk = k0 + i;
                        return row_ok && uk < P.S && (!P.causal || uk <= t);
                    };
                    p_ds64<false, true>(tS, tdP, sl, nullptr, nullptr, my_lse, my_d, valid);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(p_full + h);
        }
        if (ok && wait_all(acc_done, 0)) {
            tc_fence_after();
            // DKDV: half 0 stores dV, half 1 dK; else each half stores DP/2 columns of dQ
            // (the d real ones of them).  tcgen05.ld is warp-collective: every lane loads,
            // only valid rows store.
            constexpr int NC = DKDV ? L::DP : L::DP / 2;
            const uint32_t tacc = tmem + lane_off + 256 + h * NC;
            float *dst;
            float sc;
            bool st_ok;
            if (DKDV) {
                dst = (h == 0 ? P.dv : P.dk) + ((size_t)kvhead * P.S + u) * D;
                sc = h == 0 ? 1.0f : P.scale;
                st_ok = u < P.S;
            } else {
                dst = P.dq + ((size_t)(qhead + hl) * P.S + t) * D + h * NC;
                sc = P.scale;
                st_ok = row_ok;
            }
            const int col0 = DKDV ? 0 : h * NC;  // d column of the first stored accumulator column
#pragma unroll 1
            for (int c = 0; c < NC; c += 32) {
                uint32_t a[32];
                tmem_ld32(tacc + c, a);
                const int nv = min(32, D - (col0 + c));  // real columns of this chunk (a multiple of 16)
                if (st_ok) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        if (4 * v < nv)
                            reinterpret_cast<float4 *>(dst + c)[v] =
                                make_float4(__uint_as_float(a[4 * v]) * sc, __uint_as_float(a[4 * v + 1]) * sc,
                                            __uint_as_float(a[4 * v + 2]) * sc, __uint_as_float(a[4 * v + 3]) * sc);
                }
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int D>
cudaError_t run_bwd(const AttnBwdProblem &p, unsigned *err, cudaStream_t stream)
{
    using L = BSmem<D>;
    // R positions of each of the G heads per tile, a multiple of 4 so that every
    // tile's first position is 16-byte aligned in the fp32 lse / D rows the
    // tensor copies read (G <= 32: R >= 4)
    const int G = p.Hq / p.Hkv, R = (kRows / G) & ~3;
    CUtensorMap tq, tg, tk, tv, tl, td;
    const uint64_t dq_[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.Hq};
    const uint64_t sq_[2] = {(uint64_t)D * 2, (uint64_t)p.S * D * 2};
    const uint32_t bq_[3] = {64, (uint32_t)R, (uint32_t)G};
    const uint64_t dk_[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.Hkv};
    const uint64_t sk_[2] = {(uint64_t)D * 2, (uint64_t)p.S * D * 2};
    const uint32_t bk_[3] = {64, (uint32_t)kRows, 1};
    const uint64_t dl_[2] = {(uint64_t)p.ld, (uint64_t)p.B * p.Hq};
    const uint64_t sl_[1] = {(uint64_t)p.ld * 4};
    const uint32_t bl_[2] = {(uint32_t)R, (uint32_t)G};
    if (encode_tmap(&tq, p.q, 3, dq_, sq_, bq_, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tg, p.dO, 3, dq_, sq_, bq_, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tk, p.k, 3, dk_, sk_, bk_, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tv, p.v, 3, dk_, sk_, bk_, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tl, p.lse, 2, dl_, sl_, bl_, false, 4) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&td, p.dsum, 2, dl_, sl_, bl_, false, 4) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    BwdParams a{};
    a.B = p.B;
    a.S = p.S;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.G = G;
    a.R = R;
    a.n_qt = (p.S + R - 1) / R;
    a.n_kb = (p.S + kRows - 1) / kRows;
    a.causal = p.causal;
    a.scale = 1.0f / sqrtf((float)D);
    a.scale_log2 = 1.4426950408889634f * a.scale;
    a.lse = p.lse;
    a.dsum = p.dsum;
    a.dq = p.dq;
    a.dk = p.dk;
    a.dv = p.dv;
    a.err = err;
    const long rows = (long)p.B * p.Hq * p.S;
    dsum_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p.dO, p.o, p.dsum, p.ld, p.B, p.S, p.Hq);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const bool packed = G * R == kRows;
    auto k1 = packed ? attn_bwd_kernel<D, true, true> : attn_bwd_kernel<D, true, false>;
    auto k2 = packed ? attn_bwd_kernel<D, false, true> : attn_bwd_kernel<D, false, false>;
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC)) != cudaSuccess) return e;
    k1<<<p.B * p.Hkv * a.n_kb, kThreads, L::ALLOC, stream>>>(tq, tk, tv, tg, tl, td, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k2<<<p.B * p.Hkv * a.n_qt, kThreads, L::ALLOC, stream>>>(tq, tk, tv, tg, tl, td, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_backward(const AttnBwdProblem &p, unsigned *err, cudaStream_t stream)
{
    const int G = p.Hkv > 0 ? p.Hq / p.Hkv : 0;
    if (G <= 0 || p.Hq % p.Hkv || G > 32 || p.ld % 4 || p.ld < p.S) return cudaErrorInvalidValue;
    if (p.d == 128) return run_bwd<128>(p, err, stream);
    if (p.d == 64) return run_bwd<64>(p, err, stream);
    if (p.d == 80) return run_bwd<80>(p, err, stream);
    if (p.d == 96) return run_bwd<96>(p, err, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gqa
