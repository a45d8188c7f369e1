// decode.cu -- split-KV grouped-query attention for one new token per
// sequence over a bf16 KV cache ([T07] §4 steps 5-6: the cache returns the
// whole history and the new query attends to all of it).
//
// The step reads every cached key and value once and does ~4 flops per byte,
// so it is bound by HBM bandwidth, not by math: it runs on the CUDA cores.
//
// Pass 1 (decode_split_kernel): one CTA per (sequence b, KV head g, split s)
// streams keys [s*chunk, (s+1)*chunk) of that KV head exactly once and serves
// all G query heads of the group from each load.  Inside a warp, LPK = d/8
// lanes share one key (16 bytes each, so a warp load instruction reads whole
// 256-byte rows), partial dot products are reduced with xor-shuffles, and
// softmax runs online per block of keys in the exp2 domain.  The four warps'
// (max, sum, unnormalised output) are merged in shared memory and written as
// one fp32 partial.
//
// Pass 2 (decode_combine_kernel): per (b, g), merge the splits by their
// log-sum-exp weights and write attn[b, j*d + c] in bf16.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kWarps = 4;
constexpr int kUnroll = 4;  // key steps in flight per lane

// Partial record per (b, g, split): for each of the G heads, m (log2 domain),
// l, then o[d].
DEVI size_t part_index(int b, int g, int s, int splits, int Hkv) { return ((size_t)(b * Hkv + g) * splits + s); }

DEVI uint4 ld_stream(const uint16_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <int D, int G>
__global__ void __launch_bounds__(kWarps * 32)
    decode_split_kernel(const DecodeAttentionProblem P, float scale_log2, unsigned *err)
{
    constexpr int LPK = D / 8;       // lanes per key
    constexpr int KPS = 32 / LPK;    // keys per warp step
    constexpr int REC = G * (D + 2); // floats per partial record
    const int splits = P.splits;
    const int s = blockIdx.x % splits;
    const int bg = blockIdx.x / splits;
    const int b = bg / P.Hkv, g = bg % P.Hkv;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub = lane / LPK;      // which key of the step this lane works on
    const int dl = lane % LPK;       // which 8-element slice of d

    __shared__ float red[kWarps][G][D + 2];

    int len = P.len[b] + P.len_bias;
    if (len < 1 || len > P.Lmax) {
        if (threadIdx.x == 0) atomicOr(err, kErrIndex);
        len = 0;
    }
    const int chunk = (len + splits - 1) / splits;
    const int k_begin = min(len, s * chunk), k_end = min(len, k_begin + chunk);

    // query slices of the G heads, fp32, pre-scaled into the exp2 domain
    float q[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const uint4 v = *reinterpret_cast<const uint4 *>(P.q + ((size_t)(b * P.Hq + g * G + h) * D + dl * 8));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {  // q is binary16
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
            q[h][2 * k] = f.x * scale_log2;
            q[h][2 * k + 1] = f.y * scale_log2;
        }
    }
    float m[G], l[G], o[G][8];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) o[h][c] = 0.0f;
    }

    const size_t head_base = (size_t)(b * P.Hkv + g) * P.Lmax * D;
    const uint16_t *kbase = P.k_cache + head_base + dl * 8;
    const uint16_t *vbase = P.v_cache + head_base + dl * 8;

    // this warp's share of the split: interleaved blocks of KPS*kUnroll keys
    constexpr int BLK = KPS * kUnroll;
    for (int u0 = k_begin + warp * BLK; u0 < k_end; u0 += kWarps * BLK) {
        uint4 kv[kUnroll], vv[kUnroll];
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            const int u = u0 + i * KPS + sub;
            if (u < k_end) {
                kv[i] = ld_stream(kbase + (size_t)u * D);
                vv[i] = ld_stream(vbase + (size_t)u * D);
            } else {
                kv[i] = make_uint4(0, 0, 0, 0);
                vv[i] = make_uint4(0, 0, 0, 0);
            }
        }
        float sc[kUnroll][G];
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            const uint32_t w[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
            float kf[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                kf[2 * k] = bf16lo(w[k]);
                kf[2 * k + 1] = bf16hi(w[k]);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float acc = 0.0f;
#pragma unroll
                for (int c = 0; c < 8; ++c) acc = fmaf(q[h][c], kf[c], acc);
#pragma unroll
                for (int off = LPK / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                const int u = u0 + i * KPS + sub;
                sc[i][h] = (u < k_end) ? acc : -INFINITY;
            }
        }
        // online softmax over this block: a lane sees the KPS*kUnroll keys of
        // its own key slot; the block max is taken across the warp
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) mx = fmaxf(mx, sc[i][h]);
#pragma unroll
            for (int off = LPK; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m[h], mx);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float alpha = ex2(m[h] - m_use);
            m[h] = m_new;
            float ps = 0.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) o[h][c] *= alpha;
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                const float p = ex2(sc[i][h] - m_use);
                ps += p;
                const uint32_t w[4] = {vv[i].x, vv[i].y, vv[i].z, vv[i].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    o[h][2 * k] = fmaf(p, bf16lo(w[k]), o[h][2 * k]);
                    o[h][2 * k + 1] = fmaf(p, bf16hi(w[k]), o[h][2 * k + 1]);
                }
            }
            // every lane of a key slot holds the same ps: l is per slot, like o
            l[h] = l[h] * alpha + ps;
        }
    }
    // reduce across the KPS key slots of the warp: o and l are per-slot partial
    // sums with a common (warp-wide) max, so they simply add
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) {
#pragma unroll
            for (int c = 0; c < 8; ++c) o[h][c] += __shfl_xor_sync(0xffffffffu, o[h][c], off);
            l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
        }
    }
    if (sub == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
#pragma unroll
            for (int c = 0; c < 8; ++c) red[warp][h][dl * 8 + c] = o[h][c];
            if (dl == 0) {
                red[warp][h][D] = m[h];
                red[warp][h][D + 1] = l[h];
            }
        }
    }
    __syncthreads();
    // merge the warps and write this split's partial record
    float *rec = P.partials + part_index(b, g, s, splits, P.Hkv) * REC;
    for (int idx = threadIdx.x; idx < G * D; idx += kWarps * 32) {
        const int h = idx / D, c = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[w][h][D]);
        const float Mu = (M == -INFINITY) ? 0.0f : M;
        float acc = 0.0f, lsum = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float sc = ex2(red[w][h][D] - Mu);
            acc = fmaf(sc, red[w][h][c], acc);
            lsum = fmaf(sc, red[w][h][D + 1], lsum);
        }
        rec[h * (D + 2) + c] = acc;
        if (c == 0) {
            rec[h * (D + 2) + D] = M;
            rec[h * (D + 2) + D + 1] = lsum;
        }
    }
}

// One CTA per (b, g): merge the splits and write bf16 attn.
template <int D, int G>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeAttentionProblem P)
{
    constexpr int REC = G * (D + 2);
    const int bg = blockIdx.x;
    const int b = bg / P.Hkv, g = bg % P.Hkv;
    const float *recs = P.partials + (size_t)bg * P.splits * REC;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int h = idx / D, c = idx % D;
        float M = -INFINITY;
        for (int s = 0; s < P.splits; ++s) M = fmaxf(M, recs[s * REC + h * (D + 2) + D]);
        const float Mu = (M == -INFINITY) ? 0.0f : M;
        float acc = 0.0f, lsum = 0.0f;
        for (int s = 0; s < P.splits; ++s) {
            const float *r = recs + s * REC + h * (D + 2);
            const float w = ex2(r[D] - Mu);
            acc = fmaf(w, r[c], acc);
            lsum = fmaf(w, r[D + 1], lsum);
        }
        const float out = lsum > 0.0f ? acc / lsum : 0.0f;
        const __nv_bfloat16 ob = __float2bfloat16_rn(out);
        P.out[(size_t)b * P.Hq * D + (size_t)(g * G + h) * D + c] = *reinterpret_cast<const uint16_t *>(&ob);
    }
}

template <int D, int G>
cudaError_t run_decode(const DecodeAttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    const int grid1 = p.B * p.Hkv * p.splits;
    decode_split_kernel<D, G><<<grid1, kWarps * 32, 0, stream>>>(p, scale_log2, err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    decode_combine_kernel<D, G><<<p.B * p.Hkv, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t run_decode_d(const DecodeAttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    switch (p.Hq / p.Hkv) {
    case 1: return run_decode<D, 1>(p, err, stream);
    case 2: return run_decode<D, 2>(p, err, stream);
    case 4: return run_decode<D, 4>(p, err, stream);
    case 8: return run_decode<D, 8>(p, err, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int decode_choose_splits(int B, int Hkv, int Lmax, int num_sms)
{
    // about 512 keys per split; more splits (down to 64 keys each) when that
    // would leave fewer than ~16 CTAs per SM
    const int units = B * Hkv;
    int s = (Lmax + 511) / 512;
    const int want = (num_sms * 16 + units - 1) / units;
    const int max_by_len = (Lmax + 63) / 64;
    if (s < want) s = want < max_by_len ? want : max_by_len;
    return s < 1 ? 1 : s;
}

size_t decode_partials_floats(int B, int Hq, int splits, int d)
{
    return (size_t)B * Hq * splits * (d + 2);
}

cudaError_t launch_decode_attention(const DecodeAttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    if (p.d == 128) return run_decode_d<128>(p, err, stream);
    if (p.d == 64) return run_decode_d<64>(p, err, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gqa
