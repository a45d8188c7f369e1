// attention_bwd.cu -- backward of the causal grouped-query attention on
// tcgen05 (head_dim 64 and 128).
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
// Both: warp 0 TMA, warp 1 MMA issue, warps 2..5 the elementwise step with one
// TMEM lane (one key, or one query row) per thread.  Q, K, V and dO are
// binary16 (head-major), so P and dS are binary16 as well.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kRows = 128;      // query rows of a tile, keys of a block
constexpr int kThreads = 192;

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
    static constexpr int NCH = D / 64;
    static constexpr int CH = kRows * 128;        // 128 rows x 64 16-bit values (16 KB)
    static constexpr int TILE = NCH * CH;          // one 128-row tile of d values
    // dkdv: K, V once; Q, dO rings of 2; lse/D rings of 2 x 2 x 128 floats
    // dq:   Q, dO once;  K, V rings of 2; lse/D once
    static constexpr int A0 = 0;                   // K (dkdv) or Q (dq)
    static constexpr int A1 = A0 + TILE;           // V (dkdv) or dO (dq)
    static constexpr int RING = A1 + TILE;         // 2 stages x (2 tiles)
    static constexpr int ROWS = RING + 2 * 2 * TILE;  // 2 stages x (lse, D) x 128 floats
    static constexpr int BARS = ROWS + 2 * 2 * kRows * 4;
    static constexpr int NBARS = 8;
    static constexpr int TMEM_SLOT = BARS + NBARS * 8;
    static constexpr int TOTAL = TMEM_SLOT + 16;
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

// One elementwise pass over 64 columns of this thread's TMEM lane: reads S
// (or S^T) and dP (or dP^T) columns [c0, c0 + 64) and writes, two binary16
// values per column into columns [c0/2, c0/2 + 32):
//   DKDV: P over S and dS over dP (the A operands of dV += P^T dO, dK += dS^T Q)
//   else: dS over S (the A operand of dQ += dS K)
// The writes land on columns this thread has already read.  valid(c) says
// whether (lane, column c) is a visible pair; lse(c), dsum(c) give the
// log2-sum-exp and D of the query involved.
template <bool DKDV, typename Valid, typename Lse, typename Dsum>
DEVI void p_ds_half(uint32_t tS, uint32_t tdP, int c0, float sl, Valid valid, Lse lse, Dsum dsum)
{
    uint32_t s[64], g[64];
    tmem_ld32(tS + c0, *reinterpret_cast<uint32_t(*)[32]>(s));
    tmem_ld32(tS + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(s + 32));
    tmem_ld32(tdP + c0, *reinterpret_cast<uint32_t(*)[32]>(g));
    tmem_ld32(tdP + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(g + 32));
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            float p2[2], d2[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int i = 32 * h + 2 * e + k, c = c0 + i;
                const float p = valid(c) ? ex2(fmaf(__uint_as_float(s[i]), sl, -lse(c))) : 0.0f;
                p2[k] = p;
                d2[k] = p * (__uint_as_float(g[i]) - dsum(c));
            }
            pk[e] = pack_f16(p2[0], p2[1]);
            dk[e] = pack_f16(d2[0], d2[1]);
        }
        if (DKDV) {
            tmem_st16_nowait(tS + c0 / 2 + 16 * h, pk);
            tmem_st16_nowait(tdP + c0 / 2 + 16 * h, dk);
        } else {
            tmem_st16_nowait(tS + c0 / 2 + 16 * h, dk);
        }
    }
    tmem_st_wait();
}

// dK, dV for one (b, KV head g, 128-key block).
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                         const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                         const BwdParams P)
{
    using L = BSmem<D>;
    constexpr int NCH = L::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *kv_full = bars, *q_full = bars + 1, *q_empty = bars + 3, *s_full = bars + 5, *p_full = bars + 6,
             *acc_done = bars + 7;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::TMEM_SLOT);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;

    // heavy (early) key blocks first: they are seen by the most query tiles
    const int bh = blockIdx.x % (P.B * P.Hkv);
    const int kb = blockIdx.x / (P.B * P.Hkv);
    const int b = bh / P.Hkv, g = bh % P.Hkv;
    const int u0 = kb * kRows;
    const int qt0 = P.causal ? u0 / P.R : 0;        // first query tile that sees a key of the block
    const int nq = max(0, P.n_qt - qt0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) mbar_init(bars + i, 1);
        mbar_init(p_full, 4);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmG);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM: S^T / P^T [0, 128), dP^T / dS^T [128, 256), dV [256, 256 + D), dK [256 + D, 256 + 2D)

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(kv_full, 2 * L::TILE);
            for (int c = 0; c < NCH; ++c) {
                tma_load_3d(smem + L::A0 + c * L::CH, &tmK, c * 64, u0, b * P.Hkv + g, kv_full);
                tma_load_3d(smem + L::A1 + c * L::CH, &tmV, c * 64, u0, b * P.Hkv + g, kv_full);
            }
            int i = 0;
            for (; i < nq; ++i) {
                const int s = i & 1, t0 = (qt0 + i) * P.R;
                if (!mbar_wait(q_empty + s, ((i >> 1) & 1) ^ 1, err)) break;
                mbar_arrive_expect_tx(q_full + s, 2 * L::TILE + 2 * kRows * 4);
                uint8_t *st = smem + L::RING + s * 2 * L::TILE;
                for (int c = 0; c < NCH; ++c) {
                    tma_load_3d(st + c * L::CH, &tmQ, c * 64, t0, b * P.Hq + g * P.G, q_full + s);
                    tma_load_3d(st + L::TILE + c * L::CH, &tmG, c * 64, t0, b * P.Hq + g * P.G, q_full + s);
                }
                float *rows = reinterpret_cast<float *>(smem + L::ROWS) + s * 2 * kRows;
                tma_load_2d(rows, &tmL, t0, b * P.Hq + g * P.G, q_full + s);
                tma_load_2d(rows + kRows, &tmD, t0, b * P.Hq + g * P.G, q_full + s);
            }
            mbar_wait(kv_full, 0, err);
            for (int j = max(0, i - 2); j < i; ++j) mbar_wait(q_full + (j & 1), (j >> 1) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(kRows, kRows, 0, 0);   // 128 keys x 128 query rows
            constexpr uint32_t idesc_g = idesc_f16_f32(kRows, D, 0, 1);       // 128 keys x d, B MN-major
            const uint32_t sK = smem_u32(smem + L::A0), sV = smem_u32(smem + L::A1);
            const uint32_t tST = tmem, tdPT = tmem + 128, tdV = tmem + 256, tdK = tmem + 256 + D;
            bool ok = mbar_wait(kv_full, 0, err);
            for (int i = 0; ok && i < nq; ++i) {
                const int s = i & 1;
                if (!mbar_wait(q_full + s, (i >> 1) & 1, err)) break;
                tc_fence_after();
                const uint32_t sQ = smem_u32(smem + L::RING + s * 2 * L::TILE), sG = sQ + L::TILE;
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        umma_f16_ss(tST, sw128_desc(sK + c * L::CH + 32 * k, 16, 1024),
                                    sw128_desc(sQ + c * L::CH + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                        umma_f16_ss(tdPT, sw128_desc(sV + c * L::CH + 32 * k, 16, 1024),
                                    sw128_desc(sG + c * L::CH + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                    }
                umma_commit(s_full);
                if (!mbar_wait(p_full, i & 1, err)) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kRows / 16; ++k) {  // 16 query rows = 8 packed TMEM columns
                    umma_f16_ts(tdV, tST + 8 * k, sw128_desc(sG + k * 16 * 128, L::CH, 1024), idesc_g, (i | k) != 0);
                    umma_f16_ts(tdK, tdPT + 8 * k, sw128_desc(sQ + k * 16 * 128, L::CH, 1024), idesc_g, (i | k) != 0);
                }
                umma_commit(q_empty + s);
            }
            umma_commit(acc_done);
            mbar_wait(acc_done, 0, err);
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;        // key u0 + r
        const int u = u0 + r;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tST = tmem + lane_off, tdPT = tST + 128;
        const float sl = P.scale_log2;
        bool ok = true;
        for (int i = 0; i < nq; ++i) {
            const int s = i & 1, t0 = (qt0 + i) * P.R;
            if (!mbar_wait(s_full, i & 1, err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float *rows = reinterpret_cast<const float *>(smem + L::ROWS) + s * 2 * kRows;
            // column c = packed query row: head g*G + c/R at position t0 + c%R
            auto valid = [&](int c) {
                const int hl = c / P.R, t = t0 + (c - hl * P.R);
                return hl < P.G && t < P.S && u < P.S && (!P.causal || u <= t);
            };
            auto lse = [&](int c) { return rows[c]; };
            auto dsum = [&](int c) { return rows[kRows + c]; };
            p_ds_half<true>(tST, tdPT, 0, sl, valid, lse, dsum);
            p_ds_half<true>(tST, tdPT, 64, sl, valid, lse, dsum);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && mbar_wait(acc_done, 0, err)) {
            tc_fence_after();
            // tcgen05.ld is warp-collective: every lane loads, only keys < S store
            float *dv = P.dv + ((size_t)(b * P.Hkv + g) * P.S + u) * D;
            float *dk = P.dk + ((size_t)(b * P.Hkv + g) * P.S + u) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t a[32], k[32];
                tmem_ld32(tmem + lane_off + 256 + c, a);
                tmem_ld32(tmem + lane_off + 256 + D + c, k);
                if (u < P.S) {
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        reinterpret_cast<float4 *>(dv + c)[v] =
                            make_float4(__uint_as_float(a[4 * v]), __uint_as_float(a[4 * v + 1]),
                                        __uint_as_float(a[4 * v + 2]), __uint_as_float(a[4 * v + 3]));
                        reinterpret_cast<float4 *>(dk + c)[v] =
                            make_float4(__uint_as_float(k[4 * v]) * P.scale, __uint_as_float(k[4 * v + 1]) * P.scale,
                                        __uint_as_float(k[4 * v + 2]) * P.scale,
                                        __uint_as_float(k[4 * v + 3]) * P.scale);
                    }
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

// dQ for one (b, KV head g, query tile).
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmG,
                       const __grid_constant__ CUtensorMap tmL, const __grid_constant__ CUtensorMap tmD,
                       const BwdParams P)
{
    using L = BSmem<D>;
    constexpr int NCH = L::NCH;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *q_full = bars, *kv_full = bars + 1, *kv_empty = bars + 3, *s_full = bars + 5, *p_full = bars + 6,
             *acc_done = bars + 7;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::TMEM_SLOT);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;

    // heavy (late) query tiles first
    const int bh = blockIdx.x % (P.B * P.Hkv);
    const int qt = P.n_qt - 1 - blockIdx.x / (P.B * P.Hkv);
    const int b = bh / P.Hkv, g = bh % P.Hkv;
    const int t0 = qt * P.R;
    const int t_last = min(t0 + P.R, P.S) - 1;
    const int nk = P.causal ? t_last / kRows + 1 : P.n_kb;

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) mbar_init(bars + i, 1);
        mbar_init(p_full, 4);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmG);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM: S / dS [0, 128), dP [128, 256), dQ [256, 256 + D)
    float *rows = reinterpret_cast<float *>(smem + L::ROWS);  // lse [128], D [128]

    if (warp == 0) {
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, 2 * L::TILE + 2 * kRows * 4);
            for (int c = 0; c < NCH; ++c) {
                tma_load_3d(smem + L::A0 + c * L::CH, &tmQ, c * 64, t0, b * P.Hq + g * P.G, q_full);
                tma_load_3d(smem + L::A1 + c * L::CH, &tmG, c * 64, t0, b * P.Hq + g * P.G, q_full);
            }
            tma_load_2d(rows, &tmL, t0, b * P.Hq + g * P.G, q_full);
            tma_load_2d(rows + kRows, &tmD, t0, b * P.Hq + g * P.G, q_full);
            int j = 0;
            for (; j < nk; ++j) {
                const int s = j & 1;
                if (!mbar_wait(kv_empty + s, ((j >> 1) & 1) ^ 1, err)) break;
                mbar_arrive_expect_tx(kv_full + s, 2 * L::TILE);
                uint8_t *st = smem + L::RING + s * 2 * L::TILE;
                for (int c = 0; c < NCH; ++c) {
                    tma_load_3d(st + c * L::CH, &tmK, c * 64, j * kRows, b * P.Hkv + g, kv_full + s);
                    tma_load_3d(st + L::TILE + c * L::CH, &tmV, c * 64, j * kRows, b * P.Hkv + g, kv_full + s);
                }
            }
            mbar_wait(q_full, 0, err);
            for (int i = max(0, j - 2); i < j; ++i) mbar_wait(kv_full + (i & 1), (i >> 1) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(kRows, kRows, 0, 0);
            constexpr uint32_t idesc_q = idesc_f16_f32(kRows, D, 0, 1);   // dS K: B = K tile, d contiguous
            const uint32_t sQ = smem_u32(smem + L::A0), sG = smem_u32(smem + L::A1);
            const uint32_t tS = tmem, tdP = tmem + 128, tdQ = tmem + 256;
            bool ok = mbar_wait(q_full, 0, err);
            for (int j = 0; ok && j < nk; ++j) {
                const int s = j & 1;
                if (!mbar_wait(kv_full + s, (j >> 1) & 1, err)) break;
                tc_fence_after();
                const uint32_t sK = smem_u32(smem + L::RING + s * 2 * L::TILE), sV = sK + L::TILE;
#pragma unroll
                for (int c = 0; c < NCH; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        umma_f16_ss(tS, sw128_desc(sQ + c * L::CH + 32 * k, 16, 1024),
                                    sw128_desc(sK + c * L::CH + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                        umma_f16_ss(tdP, sw128_desc(sG + c * L::CH + 32 * k, 16, 1024),
                                    sw128_desc(sV + c * L::CH + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                    }
                umma_commit(s_full);
                if (!mbar_wait(p_full, j & 1, err)) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kRows / 16; ++k)  // 16 keys = 8 packed TMEM columns of dS
                    umma_f16_ts(tdQ, tS + 8 * k, sw128_desc(sK + k * 16 * 128, L::CH, 1024), idesc_q, (j | k) != 0);
                umma_commit(kv_empty + s);
            }
            umma_commit(acc_done);
            mbar_wait(acc_done, 0, err);
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;        // packed query row
        const int hl = r / P.R, t = t0 + (r - hl * P.R);
        const bool row_ok = hl < P.G && t < P.S;
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off, tdP = tS + 128;
        const float sl = P.scale_log2;
        bool ok = mbar_wait(q_full, 0, err);
        const float my_lse = rows[r], my_d = rows[kRows + r];
        for (int j = 0; ok && j < nk; ++j) {
            if (!mbar_wait(s_full, j & 1, err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = j * kRows;
            auto valid = [&](int c) {
                const int u = k0 + c;
                return row_ok && u < P.S && (!P.causal || u <= t);
            };
            auto lse = [&](int) { return my_lse; };
            auto dsum = [&](int) { return my_d; };
            p_ds_half<false>(tS, tdP, 0, sl, valid, lse, dsum);
            p_ds_half<false>(tS, tdP, 64, sl, valid, lse, dsum);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && mbar_wait(acc_done, 0, err)) {
            tc_fence_after();
            float *dq = P.dq + ((size_t)(b * P.Hq + g * P.G + hl) * P.S + t) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t a[32];
                tmem_ld32(tmem + lane_off + 256 + c, a);
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        reinterpret_cast<float4 *>(dq + c)[v] =
                            make_float4(__uint_as_float(a[4 * v]) * P.scale, __uint_as_float(a[4 * v + 1]) * P.scale,
                                        __uint_as_float(a[4 * v + 2]) * P.scale,
                                        __uint_as_float(a[4 * v + 3]) * P.scale);
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
    const int G = p.Hq / p.Hkv, R = kRows / G;
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
    auto k1 = attn_bwd_dkdv_kernel<D>;
    auto k2 = attn_bwd_dq_kernel<D>;
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
    if (p.Hkv <= 0 || p.Hq % p.Hkv || p.Hq / p.Hkv > 32 || p.ld % 4 || p.ld < p.S) return cudaErrorInvalidValue;
    if (p.d == 128) return run_bwd<128>(p, err, stream);
    if (p.d == 64) return run_bwd<64>(p, err, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gqa
