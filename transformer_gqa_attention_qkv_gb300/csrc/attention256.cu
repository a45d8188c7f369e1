// attention256.cu -- causal grouped-query flash attention on tcgen05 for
// head_dim 256 (prefill, and prefill into a KV cache).
//
// Computes the same function as attention.cu ([T07] §4 step 6; [NeoX]
// "Scaling and RoPE": scale head_dim^-0.5; "Attention output flattening"):
//   attn[b, t, j*256:(j+1)*256] = softmax_u( <q, k_u> / 16 ) v_u   over u <= t
// for head widths like the Gemma-3 example of [NeoX] ("Background": hidden
// 640, four query heads, an explicit head_dim of 256).
//
// Why a kernel of its own: an O accumulator 256 columns wide leaves room in
// TMEM (512 columns) for one 128-row query tile only, so the two-tile
// ping-pong of the narrower heads does not fit.  Instead one query tile
// keeps two S buffers: while the softmax warps turn S(j) into P(j), the
// tensor core computes S(j+1), then PV(j), then S(j+2) into the buffer P(j)
// came from (MMAs issued by one thread run in order, so S(j+2) overwrites
// P(j) only after PV(j) has read it).
//
//   TMEM    S buffer 0 [0, 64), S buffer 1 [64, 128), O [128, 384)
//   smem    Q 64 KB (4 swizzled 64-wide d chunks), a 3-stage K ring and a
//           2-stage V ring of 64-key tiles (32 KB each): 224 KB
//   warp 0  TMA: Q once, then K(j), V(j-1), K(j+1), V(j), ... (the order the
//           tensor core needs them)
//   warp 1  MMA issue
//   warps 2..5  softmax, one thread per row (tcgen05.ld 32x32b gives a
//           thread its row); P in 16-bit over the first 32 columns of S; O is
//           rescaled only past a 2^8 growth of the running max, after the
//           previous PV has completed (an mbarrier committed after each PV).
//
//
// G query heads of one KV group share the 128 MMA rows (floor(128/G)
// positions each), so every K/V tile is brought in once for all of them.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

// TMEM -> registers, 32 lanes x 32 bits, 64 consecutive columns, then wait;
// *mx is this thread's maximum over the 64 values (a reducing load).
__device__ __forceinline__ void tmem_ld64_max(uint32_t taddr, uint32_t (&r)[64], float &mx)
{
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x64.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, %64, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), 
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), 
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), 
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), 
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), 
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), 
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), 
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), 
          "=f"(mx)
        : "r"(taddr)
        : "memory");
}


constexpr int kD = 256;
constexpr int kRows = 128;       // MMA M: packed query rows
constexpr int kKeys = 64;        // keys per K/V tile
constexpr int kNch = kD / 64;    // 64-wide d chunks (one 128-byte swizzle row each)
constexpr int kKst = 3;          // K ring depth
constexpr int kVst = 2;          // V ring depth
constexpr int kThreads = 192;    // TMA, MMA, 4 softmax warps
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Params256 {
    int B, S, Hq, Hkv, G, R, n_qblk, causal;
    int kv_seq;
    const int *kv_start;
    float scale_log2;
    uint16_t *out;
    unsigned *err;
};

struct Smem256 {
    static constexpr int QCH = kRows * 128;            // 16 KB: 128 rows x 64 16-bit values
    static constexpr int KCH = kKeys * 128;            // 8 KB: 64 keys x 64 16-bit values
    static constexpr int Q = 0;
    static constexpr int K = Q + kNch * QCH;
    static constexpr int V = K + kKst * kNch * KCH;
    static constexpr int BARS = V + kVst * kNch * KCH;  // 224 KB of tiles
    // q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done, o_done, drain
    static constexpr int NBARS = 1 + 2 * kKst + 2 * kVst + 2 + 2 + 3;
    static constexpr int TMEM_SLOT = BARS + NBARS * 8;
    static constexpr int TOTAL = TMEM_SLOT + 16;
    static constexpr int ALLOC = TOTAL + 1024;
};
static_assert(Smem256::ALLOC <= 232448, "shared memory per CTA");

// Q, K, V and P are binary16 in the MMAs.  CACHED: the queries follow
// kv_start[b] cached keys (K and V: the binary16 copy of a bf16 cache that
// cache_widen_kernel makes); otherwise the keys are the S query positions.
template <bool CACHED>
__global__ void __launch_bounds__(kThreads, 1)
    attn256_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Params256 P)
{
    using L = Smem256;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *q_full = bars;
    uint64_t *k_full = q_full + 1;
    uint64_t *k_empty = k_full + kKst;
    uint64_t *v_full = k_empty + kKst;
    uint64_t *v_empty = v_full + kVst;
    uint64_t *s_full = v_empty + kVst;
    uint64_t *p_full = s_full + 2;
    uint64_t *pv_done = p_full + 2;
    uint64_t *o_done = pv_done + 1;
    uint64_t *drain = o_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::TMEM_SLOT);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;

    // heavy (late) query blocks first
    const int item = blockIdx.x;
    const int bh = item % (P.B * P.Hkv);
    const int qblk = P.n_qblk - 1 - item / (P.B * P.Hkv);
    const int b = bh / P.Hkv, g = bh % P.Hkv;
    const int t0 = qblk * P.R;
    const int t_last = min(t0 + P.R, P.S) - 1;
    int p0 = 0;
    bool bad = false;
    if constexpr (CACHED) {
        p0 = P.kv_start[b];
        bad = p0 < 0 || p0 + P.S > P.kv_seq;
        if (bad) {
            if (threadIdx.x == 0) atomicOr(P.err, kErrIndex);
            p0 = 0;
        }
    }
    const int n_kv = bad ? 0 : (P.causal ? ((p0 + t_last) / kKeys + 1) : (p0 + P.S + kKeys - 1) / kKeys);

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) mbar_init(bars + i, 1);
        mbar_init(p_full, 4);  // one arrival per softmax warp
        mbar_init(p_full + 1, 4);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            auto load_k = [&](int j) {
                const int s = j % kKst;
                if (!mbar_wait(k_empty + s, ((j / kKst) & 1) ^ 1, err)) return false;
                mbar_arrive_expect_tx(k_full + s, kNch * L::KCH);
                for (int c = 0; c < kNch; ++c)
                    tma_load_3d(smem + L::K + (s * kNch + c) * L::KCH, &tmK, c * 64, j * kKeys, b * P.Hkv + g,
                                k_full + s);
                return true;
            };
            auto load_v = [&](int j) {
                const int s = j % kVst;
                if (!mbar_wait(v_empty + s, ((j / kVst) & 1) ^ 1, err)) return false;
                mbar_arrive_expect_tx(v_full + s, kNch * L::KCH);
                for (int c = 0; c < kNch; ++c)
                    tma_load_3d(smem + L::V + (s * kNch + c) * L::KCH, &tmV, c * 64, j * kKeys, b * P.Hkv + g,
                                v_full + s);
                return true;
            };
            mbar_arrive_expect_tx(q_full, kNch * 64 * 2 * P.R * P.G);
            for (int c = 0; c < kNch; ++c)
                tma_load_3d(smem + L::Q + c * L::QCH, &tmQ, c * 64, t0, b * P.Hq + g * P.G, q_full);
            int nk = 0, nv = 0;  // tiles issued
            if (n_kv > 0) {
                ok = load_k(0);
                if (ok) nk = 1;
            }
            for (int j = 1; ok && j < n_kv; ++j) {
                ok = load_k(j);
                if (ok) nk = j + 1;
                if (ok) ok = load_v(j - 1);
                if (ok) nv = j;
            }
            if (ok && n_kv > 0 && load_v(n_kv - 1)) nv = n_kv;
            // every issued copy has landed before the CTA may exit
            mbar_wait(q_full, 0, err);
            for (int j = max(0, nk - kKst); j < nk; ++j) mbar_wait(k_full + j % kKst, (j / kKst) & 1, err);
            for (int j = max(0, nv - kVst); j < nv; ++j) mbar_wait(v_full + j % kVst, (j / kVst) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(kRows, kKeys, 0, 0);
            constexpr uint32_t idesc_o = idesc_f16_f32(kRows, kD, 0, 1);
            const uint32_t sQ = smem_u32(smem + L::Q);
            auto issue_s = [&](int buf, int j) {  // S(j) = Q K(j)^T into S buffer buf
                const uint32_t sK = smem_u32(smem + L::K + (j % kKst) * kNch * L::KCH);
#pragma unroll
                for (int c = 0; c < kNch; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f16_ss(tmem + 64 * buf, sw128_desc(sQ + c * L::QCH + 32 * k, 16, 1024),
                                    sw128_desc(sK + c * L::KCH + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                umma_commit(k_empty + j % kKst);
                umma_commit(s_full + buf);
            };
            bool ok = (!CACHED || n_kv > 0) && mbar_wait(q_full, 0, err) && mbar_wait(k_full, 0, err);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                if (n_kv > 1) {
                    ok = mbar_wait(k_full + 1, 0, err);
                    if (ok) {
                        tc_fence_after();
                        issue_s(1, 1);
                    }
                }
            }
            const uint32_t tO = tmem + 128;
            for (int j = 0; ok && j < n_kv; ++j) {
                const int buf = j & 1;
                if (!mbar_wait(p_full + buf, (j >> 1) & 1, err) ||
                    !mbar_wait(v_full + j % kVst, (j / kVst) & 1, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sV = smem_u32(smem + L::V + (j % kVst) * kNch * L::KCH);
#pragma unroll
                for (int k = 0; k < kKeys / 16; ++k)  // 16 keys = 8 packed TMEM columns of P
                    umma_f16_ts(tO, tmem + 64 * buf + 8 * k, sw128_desc(sV + k * 16 * 128, L::KCH, 1024), idesc_o,
                                (j | k) != 0);
                umma_commit(v_empty + j % kVst);
                umma_commit(pv_done);
                if (j + 2 < n_kv) {
                    if (!mbar_wait(k_full + (j + 2) % kKst, ((j + 2) / kKst) & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(buf, j + 2);
                }
            }
            if (ok && n_kv > 0) umma_commit(o_done);
            umma_commit(drain);
            mbar_wait(drain, 0, err);
        }
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int r = quarter * 32 + lane;
        const int hl = r / P.R, tl = r - hl * P.R;
        const bool in_pack = hl < P.G;
        const int t = t0 + tl;
        const bool row_ok = in_pack && t < P.S;
        const int lim = !in_pack ? -1 : (P.causal ? p0 + min(t, P.S - 1) : p0 + P.S - 1);
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + 128;
        const float sl = P.scale_log2;
        float m_i = -INFINITY, l_i = 0.0f;

        for (int j = 0; j < n_kv; ++j) {
            const int buf = j & 1;
            if (!mbar_wait(s_full + buf, (j >> 1) & 1, err)) break;
            tc_fence_after();
            const uint32_t tS = tmem + lane_off + 64 * buf;
            const int u0 = j * kKeys;
            // the S row and its maximum from one reducing TMEM load
            static_assert(kKeys == 64, "one 64-column load");
            uint32_t v[kKeys];
            float mx;
            tmem_ld64_max(tS, v, mx);
            if (u0 + kKeys - 1 > lim) {  // diagonal or ragged tile: mask keys past lim, max of the rest
#pragma unroll
                for (int e = 0; e < kKeys; ++e)
                    if (u0 + e > lim) v[e] = __float_as_uint(-INFINITY);
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kKeys; e += 8)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mx4[k] = fmax3(mx4[k], __uint_as_float(v[e + 2 * k]), __uint_as_float(v[e + 2 * k + 1]));
                mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
            }
            const float m_cand = fmaxf(m_i, mx * sl);
            float m_new = m_i, alpha = 1.0f;
            if (m_cand > m_i + kRescaleThreshold) {
                m_new = m_cand;
                alpha = ex2(m_i - m_new);  // 0 on the first tile
            }
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(-m_use, -m_use);
            float2 rs2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
            for (int c = 0; c < kKeys / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(v[32 * c + 2 * e]), __uint_as_float(v[32 * c + 2 * e + 1])), sl2,
                        nm2);
                    const float2 p = make_float2(ex2(x.x), ex2(x.y));
                    rs2[e & 1] = __fadd2_rn(rs2[e & 1], p);
                    pk[e] = pack_f16(p.x, p.y);
                }
                tmem_st16_nowait(tS + 16 * c, pk);
            }
            tmem_st_wait();
            const float rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
            l_i = l_i * alpha + rs;
            m_i = m_new;
            // O holds PV(0..j-1) once PV(j-1) has completed (PV(j) waits for this P)
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                if (!mbar_wait(pv_done, (j - 1) & 1, err)) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kD; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tO + c, o);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full + buf);
        }
        if (CACHED && n_kv == 0) {  // rejected offset (reported): zero rows, nothing else ran
            if (row_ok) {
                uint4 *d4 = reinterpret_cast<uint4 *>(P.out + ((size_t)(b * P.S + t) * P.Hq + g * P.G + hl) * kD);
                for (int c = 0; c < kD / 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
            }
        } else if (mbar_wait(o_done, 0, err)) {
            tc_fence_after();
            const float inv_l = (l_i > 0.0f) ? 1.0f / l_i : 0.0f;
            uint16_t *dst = P.out + ((size_t)(b * P.S + t) * P.Hq + g * P.G + hl) * kD;
#pragma unroll 1
            for (int c = 0; c < kD; c += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c, o);
                if (row_ok) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            w[k] = pack_bf16(__uint_as_float(o[8 * i + 2 * k]) * inv_l,
                                             __uint_as_float(o[8 * i + 2 * k + 1]) * inv_l);
                        d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
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

// ------------------------------------------------------------ CTA pairs
// The same attention on 2-CTA clusters (.cta_group::2).  A pair takes two
// consecutive query blocks of one (b, KV head); its MMAs have M = 256 (each
// CTA's 128 packed rows) and read each B operand half from each CTA's shared
// memory, so S tiles are 128 keys wide (N = 128, the tensor core's full rate;
// 64-wide products run at ~60% of it) while each CTA still stages only 32 KB
// per K or V tile:
//   S(j) = Q K(j)^T   N = 128 keys: CTA r stages keys [64r, 64r + 64) of the
//                     tile, all 256 d; each CTA's TMEM receives its rows x 128
//   O += P(j) V(j)    N = 256 d: CTA r stages d [128r, 128r + 128) of all 128
//                     keys (MN-major); A = P from each CTA's TMEM
// The even CTA's thread issues every MMA once both CTAs' operands are in place:
// the tensor copies of both CTAs count their bytes on the even CTA's full
// barriers, both CTAs' softmax warps arrive on its P barriers, and each MMA
// commit arrives on the barrier at the same offset in both CTAs.  The keys
// walked are those of the pair's later block (the earlier block masks the
// keys past its rows).
//
//   TMEM (each CTA)  S buffer 0 [0, 128), S buffer 1 [128, 256), O [256, 512)
//   smem (each CTA)  Q 64 KB, a 3-stage K ring and a 2-stage V ring (32 KB
//                    stages): 224 KB
constexpr int kPKeys = 128;  // keys per tile of the pair
constexpr int kPKst = 3;
constexpr int kPVst = 2;

struct SmemPair {
    static constexpr int QCH = kRows * 128;            // 16 KB: 128 rows x 64 16-bit values
    static constexpr int BOX = 64 * 128;               // 8 KB: 64 keys x 64 16-bit values
    static constexpr int KST = kNch * BOX;             // 32 KB: this CTA's 64 keys x 256 d
    static constexpr int VCH = kPKeys * 128;           // 16 KB: 128 keys x 64 d
    static constexpr int VST = 2 * VCH;                // 32 KB: 128 keys x this CTA's 128 d
    static constexpr int Q = 0;
    static constexpr int K = Q + kNch * QCH;
    static constexpr int V = K + kPKst * KST;
    static constexpr int BARS = V + kPVst * VST;       // 224 KB of tiles
    // q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done, o_done, drain
    static constexpr int NBARS = 1 + 2 * kPKst + 2 * kPVst + 2 + 2 + 3;
    static constexpr int TMEM_SLOT = BARS + NBARS * 8;
    static constexpr int TOTAL = TMEM_SLOT + 16;
    static constexpr int ALLOC = TOTAL + 1024;
};
static_assert(SmemPair::ALLOC <= 232448, "shared memory per CTA");

template <bool CACHED>
__global__ void __launch_bounds__(kThreads, 1)
    attn256_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const Params256 P)
{
    using L = SmemPair;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *q_full = bars;
    uint64_t *k_full = q_full + 1;
    uint64_t *k_empty = k_full + kPKst;
    uint64_t *v_full = k_empty + kPKst;
    uint64_t *v_empty = v_full + kPVst;
    uint64_t *s_full = v_empty + kPVst;
    uint64_t *p_full = s_full + 2;
    uint64_t *pv_done = p_full + 2;
    uint64_t *o_done = pv_done + 1;
    uint64_t *drain = o_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::TMEM_SLOT);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;
    const uint32_t rank = cluster_rank();  // 0: the CTA that issues the MMAs

    // heavy (late) query blocks first; the pair's blocks are consecutive
    const int pair = (int)blockIdx.x / 2;
    const int n_qp = (P.n_qblk + 1) / 2;
    const int bh = pair % (P.B * P.Hkv);
    const int qp = n_qp - 1 - pair / (P.B * P.Hkv);
    const int b = bh / P.Hkv, g = bh % P.Hkv;
    const int t0 = (2 * qp + (int)rank) * P.R;           // >= S for the odd CTA of a last odd block: no rows
    const int t_last = min((2 * qp + 2) * P.R, P.S) - 1;  // the pair's last position
    int p0 = 0;
    bool bad = false;
    if constexpr (CACHED) {
        p0 = P.kv_start[b];
        bad = p0 < 0 || p0 + P.S > P.kv_seq;
        if (bad) {
            if (threadIdx.x == 0 && rank == 0) atomicOr(P.err, kErrIndex);
            p0 = 0;
        }
    }
    const int n_kv = bad ? 0 : (P.causal ? ((p0 + t_last) / kPKeys + 1) : (p0 + P.S + kPKeys - 1) / kPKeys);

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) mbar_init(bars + i, 1);
        mbar_init(p_full, 8);  // the softmax warps of both CTAs
        mbar_init(p_full + 1, 8);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, 512);
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any copy or arrival reaches them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto lead = [&](uint64_t *bar) { return cluster_map(smem_u32(bar), 0); };  // the even CTA's barrier

    if (warp == 0) {
        if (lane == 0) {
            bool ok = true;
            auto arm = [&](uint64_t *bar, uint32_t bytes) {
                if (rank == 0) mbar_arrive_expect_tx(bar, 2 * bytes);  // both CTAs' copies
            };
            auto load_k = [&](int j) {
                const int s = j % kPKst;
                if (!mbar_wait<true>(k_empty + s, ((j / kPKst) & 1) ^ 1, err)) return false;
                arm(k_full + s, L::KST);
                for (int c = 0; c < kNch; ++c)
                    tma_load_3d_pair(smem + L::K + s * L::KST + c * L::BOX, &tmK, c * 64,
                                     j * kPKeys + (int)rank * 64, b * P.Hkv + g, lead(k_full + s));
                return true;
            };
            auto load_v = [&](int j) {
                const int s = j % kPVst;
                if (!mbar_wait<true>(v_empty + s, ((j / kPVst) & 1) ^ 1, err)) return false;
                arm(v_full + s, L::VST);
                for (int c = 0; c < 2; ++c)
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d_pair(smem + L::V + s * L::VST + c * L::VCH + h * L::BOX, &tmV,
                                         ((int)rank * 2 + c) * 64, j * kPKeys + h * 64, b * P.Hkv + g,
                                         lead(v_full + s));
                return true;
            };
            arm(q_full, kNch * 64 * 2 * P.R * P.G);
            for (int c = 0; c < kNch; ++c)
                tma_load_3d_pair(smem + L::Q + c * L::QCH, &tmQ, c * 64, t0, b * P.Hq + g * P.G, lead(q_full));
            int nk = 0, nv = 0;  // tiles issued
            if (n_kv > 0) {
                ok = load_k(0);
                if (ok) nk = 1;
            }
            for (int j = 1; ok && j < n_kv; ++j) {
                ok = load_k(j);
                if (ok) nk = j + 1;
                if (ok) ok = load_v(j - 1);
                if (ok) nv = j;
            }
            if (ok && n_kv > 0 && load_v(n_kv - 1)) nv = n_kv;
            // every issued copy of both CTAs has landed before the pair may exit
            // (the full barriers count both CTAs' bytes; the odd CTA waits for the
            // even one at the final cluster barrier)
            if (rank == 0) {
                mbar_wait<true>(q_full, 0, err);
                for (int j = max(0, nk - kPKst); j < nk; ++j)
                    mbar_wait<true>(k_full + j % kPKst, (j / kPKst) & 1, err);
                for (int j = max(0, nv - kPVst); j < nv; ++j)
                    mbar_wait<true>(v_full + j % kPVst, (j / kPVst) & 1, err);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(2 * kRows, kPKeys, 0, 0);
            constexpr uint32_t idesc_o = idesc_f16_f32(2 * kRows, kD, 0, 1);
            constexpr uint16_t kBoth = 3;
            const uint32_t sQ = smem_u32(smem + L::Q);
            auto issue_s = [&](int buf, int j) {  // S(j) = Q K(j)^T into S buffer buf of both CTAs
                const uint32_t sK = smem_u32(smem + L::K + (j % kPKst) * L::KST);
#pragma unroll
                for (int c = 0; c < kNch; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f16_ss_pair(tmem + kPKeys * buf, sw128_desc(sQ + c * L::QCH + 32 * k, 16, 1024),
                                         sw128_desc(sK + c * L::BOX + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                umma_commit_pair(k_empty + j % kPKst, kBoth);
                umma_commit_pair(s_full + buf, kBoth);
            };
            bool ok = (!CACHED || n_kv > 0) && mbar_wait<true>(q_full, 0, err) && mbar_wait<true>(k_full, 0, err);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                if (n_kv > 1) {
                    ok = mbar_wait<true>(k_full + 1, 0, err);
                    if (ok) {
                        tc_fence_after();
                        issue_s(1, 1);
                    }
                }
            }
            const uint32_t tO = tmem + 256;
            for (int j = 0; ok && j < n_kv; ++j) {
                const int buf = j & 1;
                if (!mbar_wait<true>(p_full + buf, (j >> 1) & 1, err) ||
                    !mbar_wait<true>(v_full + j % kPVst, (j / kPVst) & 1, err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sV = smem_u32(smem + L::V + (j % kPVst) * L::VST);
#pragma unroll
                for (int k = 0; k < kPKeys / 16; ++k)  // 16 keys = 8 packed TMEM columns of P
                    umma_f16_ts_pair(tO, tmem + kPKeys * buf + 8 * k, sw128_desc(sV + k * 16 * 128, L::VCH, 1024),
                                     idesc_o, (j | k) != 0);
                umma_commit_pair(v_empty + j % kPVst, kBoth);
                umma_commit_pair(pv_done, kBoth);
                if (j + 2 < n_kv) {
                    if (!mbar_wait<true>(k_full + (j + 2) % kPKst, ((j + 2) / kPKst) & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(buf, j + 2);
                }
            }
            if (ok && n_kv > 0) umma_commit_pair(o_done, kBoth);
            umma_commit_pair(drain, 1);
            mbar_wait(drain, 0, err);
        }
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int r = quarter * 32 + lane;
        const int hl = r / P.R, tl = r - hl * P.R;
        const bool in_pack = hl < P.G;
        const int t = t0 + tl;
        const bool row_ok = in_pack && t < P.S;
        const int lim = !in_pack ? -1 : (P.causal ? p0 + min(t, P.S - 1) : p0 + P.S - 1);
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_off + 256;
        const float sl = P.scale_log2;
        float m_i = -INFINITY, l_i = 0.0f;

        for (int j = 0; j < n_kv; ++j) {
            const int buf = j & 1;
            if (!mbar_wait<true>(s_full + buf, (j >> 1) & 1, err)) break;
            tc_fence_after();
            const uint32_t tS = tmem + lane_off + kPKeys * buf;
            const int u0 = j * kPKeys;
            // the S row (two 64-column reducing loads) and its maximum
            uint32_t va[64], vb[64];
            float mxa, mxb;
            tmem_ld64_max(tS, va, mxa);
            tmem_ld64_max(tS + 64, vb, mxb);
            float mx = fmaxf(mxa, mxb);
            if (u0 + kPKeys - 1 > lim) {  // diagonal or ragged tile: mask keys past lim, max of the rest
#pragma unroll
                for (int e = 0; e < 64; ++e) {
                    if (u0 + e > lim) va[e] = __float_as_uint(-INFINITY);
                    if (u0 + 64 + e > lim) vb[e] = __float_as_uint(-INFINITY);
                }
                float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 64; e += 4)
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        mx4[k] = fmax3(mx4[k], __uint_as_float(va[e + 2 * k]), __uint_as_float(va[e + 2 * k + 1]));
                        mx4[2 + k] =
                            fmax3(mx4[2 + k], __uint_as_float(vb[e + 2 * k]), __uint_as_float(vb[e + 2 * k + 1]));
                    }
                mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
            }
            const float m_cand = fmaxf(m_i, mx * sl);
            float m_new = m_i, alpha = 1.0f;
            if (m_cand > m_i + kRescaleThreshold) {
                m_new = m_cand;
                alpha = ex2(m_i - m_new);  // 0 on the first tile
            }
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(-m_use, -m_use);
            float2 rs2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
            for (int c = 0; c < kPKeys / 32; ++c) {
                const uint32_t *v = c < 2 ? va + 32 * c : vb + 32 * (c - 2);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1])), sl2, nm2);
                    const float2 p = make_float2(ex2(x.x), ex2(x.y));
                    rs2[e & 1] = __fadd2_rn(rs2[e & 1], p);
                    pk[e] = pack_f16(p.x, p.y);
                }
                tmem_st16_nowait(tS + 16 * c, pk);
            }
            tmem_st_wait();
            const float rs = (rs2[0].x + rs2[0].y) + (rs2[1].x + rs2[1].y);
            l_i = l_i * alpha + rs;
            m_i = m_new;
            // O holds PV(0..j-1) once PV(j-1) has completed (PV(j) waits for this P)
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
                if (!mbar_wait<true>(pv_done, (j - 1) & 1, err)) break;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kD; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + c, o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tO + c, o);
                }
            }
            tc_fence_before();
            __syncwarp();
            // P (and any rescaled O) is in TMEM: the arrival carries no memory writes
            if (lane == 0) mbar_arrive_cluster_relaxed(lead(p_full + buf));
        }
        if (CACHED && n_kv == 0) {  // rejected offset (reported): zero rows, nothing else ran
            if (row_ok) {
                uint4 *d4 = reinterpret_cast<uint4 *>(P.out + ((size_t)(b * P.S + t) * P.Hq + g * P.G + hl) * kD);
                for (int c = 0; c < kD / 8; ++c) d4[c] = make_uint4(0, 0, 0, 0);
            }
        } else if (mbar_wait<true>(o_done, 0, err)) {
            tc_fence_after();
            const float inv_l = (l_i > 0.0f) ? 1.0f / l_i : 0.0f;
            uint16_t *dst = P.out + ((size_t)(b * P.S + t) * P.Hq + g * P.G + hl) * kD;
#pragma unroll 1
            for (int c = 0; c < kD; c += 32) {
                uint32_t o[32];
                tmem_ld32(tO + c, o);
                if (row_ok) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t w[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            w[k] = pack_bf16(__uint_as_float(o[8 * i + 2 * k]) * inv_l,
                                             __uint_as_float(o[8 * i + 2 * k + 1]) * inv_l);
                        d4[i] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }
    __syncthreads();
    cluster_sync();  // no CTA leaves while the other's copies, MMAs or arrivals may still reach it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

template <bool CACHED>
cudaError_t run_attn256(const AttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    const int G = p.Hq / p.Hkv;
    const int R = kRows / G;
    CUtensorMap tq, tk, tv;
    // Q viewed as [B*Hq, S, 256]; box {64, R, G}: the G heads of one group, R positions each
    const uint64_t dq[3] = {(uint64_t)kD, (uint64_t)p.S, (uint64_t)p.B * p.Hq};
    const uint64_t sq[2] = {(uint64_t)kD * 2, (uint64_t)p.S * kD * 2};
    const uint32_t bq[3] = {64, (uint32_t)R, (uint32_t)G};
    // K, V viewed as [B*Hkv, kv_seq, 256]; box {64, 64 keys, 1}
    const uint64_t dk[3] = {(uint64_t)kD, (uint64_t)p.kv_seq, (uint64_t)p.B * p.Hkv};
    const uint64_t sk[2] = {(uint64_t)kD * 2, (uint64_t)p.kv_seq * kD * 2};
    const uint32_t bk[3] = {64, (uint32_t)kKeys, 1};
    if (encode_tmap(&tq, p.q, 3, dq, sq, bq, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tk, p.k, 3, dk, sk, bk, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tv, p.v, 3, dk, sk, bk, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    Params256 a{};
    a.B = p.B;
    a.S = p.S;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.G = G;
    a.R = R;
    a.n_qblk = (p.S + R - 1) / R;
    a.causal = p.causal;
    a.kv_seq = p.kv_seq;
    a.kv_start = p.kv_start;
    a.scale_log2 = 1.4426950408889634f / 16.0f;  // log2(e) / sqrt(256)
    a.out = p.out;
    a.err = err;

    // CTA pairs when enabled and the cluster shape can be placed, else one CTA per block
    if (cta_pairs_enabled()) {
        auto kern = attn256_pair_kernel<CACHED>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SmemPair::ALLOC);
        if (e != cudaSuccess) return e;
        int clusters = 0;
        LaunchCfg probe(dim3(2), dim3(kThreads), SmemPair::ALLOC, stream, false, 2);
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &probe.cfg) == cudaSuccess && clusters >= 1) {
            const long long grid = 2LL * ((a.n_qblk + 1) / 2) * p.B * p.Hkv;
            if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
            LaunchCfg lc(dim3((unsigned)grid), dim3(kThreads), SmemPair::ALLOC, stream, false, 2);
            e = cudaLaunchKernelEx(&lc.cfg, kern, tq, tk, tv, a);
            if (e != cudaSuccess) return e;
            return cudaGetLastError();
        }
        cudaGetLastError();
    }
    auto kern = attn256_kernel<CACHED>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Smem256::ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<p.B * p.Hkv * a.n_qblk, kThreads, Smem256::ALLOC, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention256(const AttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    if (p.d != kD || p.Hkv <= 0 || p.Hq % p.Hkv || p.Hq / p.Hkv > kRows) return cudaErrorInvalidValue;
    return p.cached ? run_attn256<true>(p, err, stream) : run_attn256<false>(p, err, stream);
}

}  // namespace gqa
