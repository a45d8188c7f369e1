// attention.cu -- causal grouped-query flash attention on tcgen05 (prefill).
//
// Computes, for query head j, KV head g = j / G (G = Hq/Hkv), query position t:
//   attn[b, t, j*d:(j+1)*d] = softmax_u( <q, k_u> / sqrt(d) ) v_u   over u <= t
// ([T07] §4 step 6 in fp32; [NeoX] "Scaling and RoPE" scale head_dim^-0.5;
//  [NeoX] "Attention output flattening": output width Hq*d).
//
// One CTA handles one (sequence b, KV head g, block of R = 128/G positions)
// work item.  The G query heads of the group are packed into the MMA's M
// dimension: row r of the 128-row tile is head g*G + r/R at position
// t0 + r%R.  Each K/V tile (128 keys) is therefore brought into shared memory
// once by TMA and used by every query head of the group in a single MMA.
//
//   warp 0      TMA: Q tile once, then K and V tiles into a 2-deep ring
//   warp 1      MMA: S = Q K^T (TMEM), then O += P V (TMEM)
//   warps 2..5  softmax: one thread per row (tcgen05.ld 32x32b gives a thread
//               a whole row, so row max and row sum need no shuffles); online
//               softmax in fp32 with exp2; P to shared memory as binary16;
//               O rescaled in TMEM only when the running max grows by more
//               than 2^8; final O / l written as bf16.
//
// Q, K and V arrive as binary16: with QK-norm their rows are bounded by
// sqrt(d) * max|w|, and binary16 keeps 3 more mantissa bits than bf16, which
// halves the rounding error that storage adds to the scores and outputs.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kRows = 128;      // MMA M: packed query rows per tile
constexpr int kKeys = 128;      // keys per K/V tile
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only past a 256x growth

struct AttnParams {
    int B, S, Hq, Hkv, G, R, n_qblk, causal, num_items;
    float scale_log2;  // log2(e) / sqrt(d)
    uint16_t *out;
    unsigned *err;
};

template <int D>
struct ASmem {
    static constexpr int CHUNK = kRows * 128;             // 128 rows x 64 16-bit = 16 KB
    static constexpr int NCH = D / 64;                    // d chunks per row
    static constexpr int Q = 0;
    static constexpr int K = Q + NCH * CHUNK;             // 2 stages
    static constexpr int V = K + 2 * NCH * CHUNK;         // 2 stages
    static constexpr int P = V + 2 * NCH * CHUNK;         // 2 key chunks
    static constexpr int BARS = P + 2 * CHUNK;
    static constexpr int NBARS = 1 + 2 + 2 + 2 + 3 + 1;   // q, k[2], v[2], kv_empty[2], s, p, o, drain
    static constexpr int TMEM_SLOT = BARS + NBARS * 8;
    static constexpr int TOTAL = TMEM_SLOT + 16;
    static constexpr int ALLOC = TOTAL + 1024;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnParams P)
{
    using L = ASmem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *q_full = bars;
    uint64_t *k_full = bars + 1;
    uint64_t *v_full = bars + 3;
    uint64_t *kv_empty = bars + 5;
    uint64_t *s_full = bars + 7;
    uint64_t *p_full = bars + 8;
    uint64_t *o_done = bars + 9;
    uint64_t *drain = bars + 10;
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
    const int n_kv = P.causal ? (t_last / kKeys + 1) : (P.S + kKeys - 1) / kKeys;

    if (threadIdx.x == 0) {
        for (int i = 0; i < L::NBARS; ++i) mbar_init(bars + i, 1);
        mbar_init(p_full, 4);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 256);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem;        // S: columns [0, 128)
    const uint32_t tO = tmem + 128;  // O: columns [128, 128 + D)

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t q_bytes = L::NCH * 64 * 2 * P.R * P.G;
            mbar_arrive_expect_tx(q_full, q_bytes);
            for (int c = 0; c < L::NCH; ++c)
                tma_load_3d(smem + L::Q + c * L::CHUNK, &tmQ, c * 64, t0, b * P.Hq + g * P.G, q_full);
            int j = 0;
            for (; j < n_kv; ++j) {
                const int s = j & 1;
                if (!mbar_wait(kv_empty + s, ((j >> 1) & 1) ^ 1, err)) break;
                mbar_arrive_expect_tx(k_full + s, L::NCH * L::CHUNK);
                for (int c = 0; c < L::NCH; ++c)
                    tma_load_3d(smem + L::K + (s * L::NCH + c) * L::CHUNK, &tmK, c * 64, j * kKeys, b * P.Hkv + g,
                                k_full + s);
                mbar_arrive_expect_tx(v_full + s, L::NCH * L::CHUNK);
                for (int c = 0; c < L::NCH; ++c)
                    tma_load_3d(smem + L::V + (s * L::NCH + c) * L::CHUNK, &tmV, c * 64, j * kKeys, b * P.Hkv + g,
                                v_full + s);
            }
            mbar_wait(q_full, 0, err);
            for (int i = max(0, j - 2); i < j; ++i) {
                mbar_wait(k_full + (i & 1), (i >> 1) & 1, err);
                mbar_wait(v_full + (i & 1), (i >> 1) & 1, err);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16_f32(kRows, kKeys, 0, 0);  // Q, K: binary16, K-major (over d)
            constexpr uint32_t idesc_o = idesc_f16_f32(kRows, D, 0, 1);      // P K-major, V MN-major (d contiguous)
            const uint32_t sQ = smem_u32(smem + L::Q);
            const uint32_t sP = smem_u32(smem + L::P);
            auto issue_s = [&](int j) {
                const int s = j & 1;
                const uint32_t sK = smem_u32(smem + L::K + s * L::NCH * L::CHUNK);
#pragma unroll
                for (int c = 0; c < L::NCH; ++c)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_f16_ss(tS, sw128_desc(sQ + c * L::CHUNK + 32 * k, 16, 1024),
                                     sw128_desc(sK + c * L::CHUNK + 32 * k, 16, 1024), idesc_s, (c | k) != 0);
                umma_commit(s_full);
            };
            bool ok = mbar_wait(q_full, 0, err) && mbar_wait(k_full, 0, err);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int s = j & 1;
                if (!mbar_wait(p_full, j & 1, err)) break;
                tc_fence_after();
                if (j + 1 < n_kv) {
                    if (!mbar_wait(k_full + ((j + 1) & 1), ((j + 1) >> 1) & 1, err)) break;
                    tc_fence_after();
                    issue_s(j + 1);
                }
                if (!mbar_wait(v_full + s, (j >> 1) & 1, err)) break;
                tc_fence_after();
                const uint32_t sV = smem_u32(smem + L::V + s * L::NCH * L::CHUNK);
#pragma unroll
                for (int k = 0; k < kKeys / 16; ++k)
                    umma_f16_ss(tO, sw128_desc(sP + (k >> 2) * L::CHUNK + 32 * (k & 3), 16, 1024),
                                 sw128_desc(sV + k * 16 * 128, L::CHUNK, 1024), idesc_o, (j | k) != 0);
                umma_commit(o_done);
                umma_commit(kv_empty + s);
            }
            umma_commit(drain);
            mbar_wait(drain, 0, err);
        }
    } else {
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;  // tile row = TMEM lane
        const int hl = r / P.R, tl = r - hl * P.R;
        const bool in_pack = hl < P.G;
        const int t = t0 + tl;
        const bool row_ok = in_pack && t < P.S;
        const int t_vis = in_pack ? t : -1;  // last visible key for a causal row
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        uint8_t *prow = smem + L::P + r * 128;
        float m_i = -INFINITY, l_i = 0.0f;

        for (int j = 0; j < n_kv; ++j) {
            if (!mbar_wait(s_full, j & 1, err)) break;
            tc_fence_after();
            float sv[kKeys];
#pragma unroll
            for (int c = 0; c < kKeys; c += 32) {
                uint32_t rr[32];
                tmem_ld32(tS + lane_off + c, rr);
#pragma unroll
                for (int i = 0; i < 32; ++i) sv[c + i] = __uint_as_float(rr[i]);
            }
            const int u0 = j * kKeys;
            const int lim = P.causal ? min(t_vis, P.S - 1) : (in_pack ? P.S - 1 : -1);  // keys u <= lim visible
            float mx = -INFINITY;
            if (u0 + kKeys - 1 > lim) {
#pragma unroll
                for (int c = 0; c < kKeys; ++c)
                    if (u0 + c > lim) sv[c] = -INFINITY;
            }
#pragma unroll
            for (int c = 0; c < kKeys; ++c) mx = fmaxf(mx, sv[c]);
            const float m_cand = fmaxf(m_i, mx * P.scale_log2);
            float m_new = m_i, alpha = 1.0f;
            if (m_cand > m_i + kRescaleThreshold) {
                m_new = m_cand;
                alpha = ex2(m_i - m_new);  // 0 on the first tile
            }
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            float rs = 0.0f;
            uint32_t pk[kKeys / 2];
#pragma unroll
            for (int c = 0; c < kKeys; c += 2) {
                const float p0 = ex2(fmaf(sv[c], P.scale_log2, -m_use));
                const float p1 = ex2(fmaf(sv[c + 1], P.scale_log2, -m_use));
                rs += p0 + p1;
                pk[c / 2] = pack_f16(p0, p1);  // p <= 2^8: inside the binary16 range
            }
            l_i = l_i * alpha + rs;
            m_i = m_new;
            // PV(j-1) must be done before P is overwritten and before O is rescaled
            if (j > 0) {
                if (!mbar_wait(o_done, (j - 1) & 1, err)) break;
                tc_fence_after();
            }
#pragma unroll
            for (int kc = 0; kc < 2; ++kc)
#pragma unroll
                for (int gi = 0; gi < 8; ++gi) {
                    const int q16 = kc * 32 + gi * 4;
                    *reinterpret_cast<uint4 *>(prow + kc * L::CHUNK + ((gi ^ (r & 7)) << 4)) =
                        make_uint4(pk[q16], pk[q16 + 1], pk[q16 + 2], pk[q16 + 3]);
                }
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t o[32];
                    tmem_ld32(tO + lane_off + c, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(tO + lane_off + c, o);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (mbar_wait(o_done, (n_kv - 1) & 1, err)) {
            tc_fence_after();
            const float inv_l = (l_i > 0.0f) ? 1.0f / l_i : 0.0f;
            const int head = g * P.G + hl;
            uint16_t *dst = P.out + ((size_t)(b * P.S + t) * P.Hq + head) * D;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
                uint32_t o[32];
                tmem_ld32(tO + lane_off + c, o);
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
        tmem_dealloc(tmem, 256);
    }
}

template <int D>
cudaError_t run_attn(const AttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    using L = ASmem<D>;
    const int G = p.Hq / p.Hkv;
    const int R = kRows / G;
    CUtensorMap tq, tk, tv;
    // Q viewed as [B*Hq, S, D]; box {64, R, G}: the G heads of one group, R positions each
    const uint64_t dq[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.Hq};
    const uint64_t sq[2] = {(uint64_t)D * 2, (uint64_t)p.S * D * 2};
    const uint32_t bq[3] = {64, (uint32_t)R, (uint32_t)G};
    const uint64_t dk[3] = {(uint64_t)D, (uint64_t)p.S, (uint64_t)p.B * p.Hkv};
    const uint64_t sk[2] = {(uint64_t)D * 2, (uint64_t)p.S * D * 2};
    const uint32_t bk[3] = {64, (uint32_t)kKeys, 1};
    if (encode_tmap(&tq, p.q, 3, dq, sq, bq, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tk, p.k, 3, dk, sk, bk, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tv, p.v, 3, dk, sk, bk, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    AttnParams a{};
    a.B = p.B;
    a.S = p.S;
    a.Hq = p.Hq;
    a.Hkv = p.Hkv;
    a.G = G;
    a.R = R;
    a.n_qblk = (p.S + R - 1) / R;
    a.causal = p.causal;
    a.num_items = p.B * p.Hkv * a.n_qblk;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    a.out = p.out;
    a.err = err;
    auto kern = attn_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    kern<<<a.num_items, kThreads, L::ALLOC, stream>>>(tq, tk, tv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttentionProblem &p, unsigned *err, int num_sms, cudaStream_t stream)
{
    (void)num_sms;
    if (p.Hkv <= 0 || p.Hq % p.Hkv) return cudaErrorInvalidValue;
    const int G = p.Hq / p.Hkv;
    if (G > kRows) return cudaErrorInvalidValue;
    if (p.d == 128) return run_attn<128>(p, err, stream);
    if (p.d == 64) return run_attn<64>(p, err, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gqa
