// decode.cu -- split-KV grouped-query attention for one new token per
// sequence over a bf16 KV cache ([T07] §4 steps 5-6: the cache returns the
// whole history and the new query attends to all of it).
//
// The step reads every cached key and value once (2.1 GB for 64 sequences of
// 8193 tokens) and does ~4 flops per byte: it is bound by HBM bandwidth.  The
// design keeps ~150 KB per SM in flight and spends as few instructions per
// key as possible.
//
// Pass 1 (decode_split_kernel), persistent, one CTA per SM.  Work item =
// (sequence b, KV head g, split s): a contiguous range of that head's keys.
//   warp 0      TMA: the item's keys and values in chunks of 64 keys
//               (128-byte swizzled tiles), into a shared-memory ring, across
//               items without pausing;
//   warps 1..4  16 keys of every chunk each.  The G query heads of the group
//               sharing each K/V row are a genuine G x d by d x keys product,
//               computed with warp-level mma.sync m16n8k16 (heads in the M
//               rows, padded to 16): S = Q K^T with K fragments read by
//               ldmatrix from the swizzled tile; the binary16 query is split
//               into bf16 high and low parts (two MMAs) so no query precision
//               is lost; online softmax in the S accumulator registers; the
//               probabilities are already laid out as the A fragment of
//               O += P V, with V fragments from ldmatrix.trans.
//   At the end of an item the four warps' (max, sum, unnormalised output)
//   are merged in shared memory into one fp32 partial record.
// Pass 2 (decode_combine_kernel): per (b, g), merge the splits by their
// log-sum-exp weights and write attn[b, j*d + c] in bf16.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kChunk = 64;     // keys per staged chunk
constexpr int kWarps = 4;      // consumer warps, 16 keys of each chunk each
constexpr int kThreads = 32 * (1 + kWarps);

template <int D>
struct DSmem {
    static constexpr int NCH = D / 64;            // 64-wide d halves
    static constexpr int BOX = kChunk * 128;       // one 64-key x 64-d swizzled box (8 KB)
    static constexpr int CB = NCH * BOX;           // one K (or V) chunk
    static constexpr int STAGES = D == 128 ? 6 : 12;
    static constexpr int K = 0;
    static constexpr int V = STAGES * CB;
    static constexpr int RED = 2 * STAGES * CB;    // [kWarps][8][D + 2] floats
    static constexpr int BARS = RED + kWarps * 8 * (D + 2) * 4;
    static constexpr int TOTAL = BARS + 2 * STAGES * 8;
    static constexpr int ALLOC = TOTAL + 1024;
};

DEVI void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kWarps * 32) : "memory"); }

// Key range of one work item.
struct ItemRange {
    int b, g, s, begin, end;  // keys [begin, end)
};

DEVI ItemRange item_range(const DecodeAttentionProblem &P, int item, unsigned *err, bool report)
{
    ItemRange r;
    const int bg = item / P.splits;
    r.s = item - bg * P.splits;
    r.b = bg / P.Hkv;
    r.g = bg - r.b * P.Hkv;
    int len = P.len[r.b] + P.len_bias;
    if (len < 1 || len > P.Lmax) {
        if (report) atomicOr(err, kErrIndex);
        len = 0;
    }
    const int chunks = (len + kChunk - 1) / kChunk;
    const int per = (chunks + P.splits - 1) / P.splits;
    const int c0 = min(chunks, r.s * per), c1 = min(chunks, c0 + per);
    r.begin = c0 * kChunk;
    r.end = min(c1 * kChunk, len);
    if (r.end < r.begin) r.end = r.begin;
    return r;
}

// Byte offset of (key, d) inside a chunk stored as NCH swizzled 64-key x 64-d
// boxes: 128-byte rows, 16-byte units XOR-ed with the row's low 3 bits.
template <int D>
DEVI uint32_t swz(int key, int dcol)
{
    return (uint32_t)((dcol >> 6) * DSmem<D>::BOX + key * 128 + ((((dcol & 63) >> 3) ^ (key & 7)) << 4));
}

DEVI uint32_t bf16x2_bits(float lo, float hi) { return pack_bf16(lo, hi); }

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeAttentionProblem P, float scale_log2, int n_items, unsigned *err)
{
    using L = DSmem<D>;
    constexpr int ST = L::STAGES;
    constexpr int KS = D / 16;   // k-steps of the QK product
    constexpr int NT = D / 8;    // n-tiles of the PV product
    constexpr int REC = G * (D + 2);
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *empty = full + ST;
    float *red = reinterpret_cast<float *>(smem + L::RED);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kWarps);
        }
        fence_mbar_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    __syncthreads();

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < n_items; item += gridDim.x) {
                const ItemRange r = item_range(P, item, err, true);
                const int z = r.b * P.Hkv + r.g;
                for (int u0 = r.begin; u0 < r.end; u0 += kChunk, ++it) {
                    const int s = it % ST;
                    if (!mbar_wait(empty + s, ((it / ST) & 1) ^ 1, err)) {
                        ok = false;
                        break;
                    }
                    // whole boxes are transferred (rows past Lmax read as zero)
                    mbar_arrive_expect_tx(full + s, 2 * L::CB);
                    for (int c = 0; c < L::NCH; ++c) {
                        tma_load_3d(smem + L::K + s * L::CB + c * L::BOX, &tmK, c * 64, u0, z, full + s);
                        tma_load_3d(smem + L::V + s * L::CB + c * L::BOX, &tmV, c * 64, u0, z, full + s);
                    }
                }
            }
            for (int j = max(0, it - ST); j < it; ++j) mbar_wait(full + j % ST, (j / ST) & 1, err);
        }
        return;  // the producer takes no part in the consumer barriers below
    }

    const int cw = warp - 1;            // consumer warp: keys [16 cw, 16 cw + 16) of each chunk
    const int grp = lane >> 2, tig = lane & 3;
    const bool row_valid = grp < G;     // MMA row grp = query head g*G + grp
    // ldmatrix row addresses (relative to a chunk): lane i serves row i%8 of matrix i/8
    const int mi = lane >> 3, mr = lane & 7;
    const int qk_key = cw * 16 + (mi >> 1) * 8 + mr, qk_dofs = (mi & 1) * 8;  // K: (keys, d) blocks
    const int pv_key = cw * 16 + (mi & 1) * 8 + mr, pv_dofs = (mi >> 1) * 8;  // V: transposed blocks

    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const ItemRange r = item_range(P, item, err, false);
        // A fragments of Q (rows = heads of the group, binary16 split into bf16 hi + lo)
        uint32_t qh[KS][2], ql[KS][2];
        {
            const uint16_t *qrow = P.q + ((size_t)(r.b * P.Hq + r.g * G + (row_valid ? grp : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float2 f = make_float2(0.0f, 0.0f);
                    if (row_valid)
                        f = __half22float2(*reinterpret_cast<const __half2 *>(qrow + ks * 16 + half * 8 + 2 * tig));
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(f.x, f.y);
                    const float2 hf = __bfloat1622float2(hi);
                    qh[ks][half] = *reinterpret_cast<const uint32_t *>(&hi);
                    ql[ks][half] = bf16x2_bits(f.x - hf.x, f.y - hf.y);
                }
        }
        float o[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
        float m_run = -INFINITY, l_run = 0.0f;  // for row grp (scaled log2 domain)

        for (int u0 = r.begin; u0 < r.end; u0 += kChunk, ++it) {
            const int s = it % ST;
            if (!mbar_wait(full + s, (it / ST) & 1, err)) break;
            const uint32_t kb = smem_u32(smem + L::K + s * L::CB);
            const uint32_t vb = smem_u32(smem + L::V + s * L::CB);
            // Value rows past the item's last key may hold anything (slots past
            // the sequence are not initialised); 0 * NaN would poison O, so the
            // rows this warp reads are zeroed.  Masked scores need no such care.
            if (u0 + kChunk > r.end) {
                const int first = max(r.end - u0, cw * 16);
                uint4 *vrow = reinterpret_cast<uint4 *>(smem + L::V + s * L::CB);
                for (int idx = lane; idx < (cw * 16 + 16 - first) * L::NCH * 8; idx += 32) {
                    const int key = first + idx / (L::NCH * 8), rem = idx % (L::NCH * 8);
                    vrow[((rem >> 3) * L::BOX + key * 128) / 16 + (rem & 7)] = make_uint4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            // S[heads x 16 keys] = Q K^T
            float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t b00, b01, b10, b11;
                ldsm_x4(kb + swz<D>(qk_key, ks * 16 + qk_dofs), b00, b01, b10, b11);
                mma_bf16_16816(sc[0], qh[ks][0], 0u, qh[ks][1], 0u, b00, b01);
                mma_bf16_16816(sc[1], qh[ks][0], 0u, qh[ks][1], 0u, b10, b11);
                mma_bf16_16816(sc[0], ql[ks][0], 0u, ql[ks][1], 0u, b00, b01);
                mma_bf16_16816(sc[1], ql[ks][0], 0u, ql[ks][1], 0u, b10, b11);
            }
            // mask keys beyond the item and take the row max over this warp's 16 keys
            const int kbase = u0 + cw * 16 + 2 * tig;
            float v[4] = {sc[0][0], sc[0][1], sc[1][0], sc[1][1]};  // keys kbase, +1, +8, +9
            const int koff[4] = {0, 1, 8, 9};
            float mx = -INFINITY;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[e] = (kbase + koff[e] < r.end) ? v[e] * scale_log2 : -INFINITY;
                mx = fmaxf(mx, v[e]);
            }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run, mx);
            const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
            const float alpha = ex2(m_run - m_use);
            m_run = m_new;
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) p[e] = (v[e] == -INFINITY) ? 0.0f : ex2(v[e] - m_use);
            l_run = l_run * alpha + (p[0] + p[1] + p[2] + p[3]);
            // P as the A fragment of O += P V (rows 8..15 are padding), split
            // into bf16 high and low parts so P keeps ~16 mantissa bits
            uint32_t a0h = 0u, a2h = 0u, a0l = 0u, a2l = 0u;
            if (row_valid) {
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(p[0], p[1]);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(p[2], p[3]);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                a0h = *reinterpret_cast<const uint32_t *>(&h01);
                a2h = *reinterpret_cast<const uint32_t *>(&h23);
                a0l = bf16x2_bits(p[0] - f01.x, p[1] - f01.y);
                a2l = bf16x2_bits(p[2] - f23.x, p[3] - f23.y);
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= alpha;
                o[n][1] *= alpha;
            }
#pragma unroll
            for (int nb = 0; nb < NT / 2; ++nb) {
                uint32_t b0a, b1a, b0b, b1b;
                ldsm_x4_trans(vb + swz<D>(pv_key, nb * 16 + pv_dofs), b0a, b1a, b0b, b1b);
                mma_bf16_16816(o[2 * nb], a0h, 0u, a2h, 0u, b0a, b1a);
                mma_bf16_16816(o[2 * nb + 1], a0h, 0u, a2h, 0u, b0b, b1b);
                mma_bf16_16816(o[2 * nb], a0l, 0u, a2l, 0u, b0a, b1a);
                mma_bf16_16816(o[2 * nb + 1], a0l, 0u, a2l, 0u, b0b, b1b);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
        }
        // row sum over the four lanes of a row; the max is already row-uniform
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
        float *rw = red + cw * 8 * (D + 2);
        if (row_valid) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                rw[grp * (D + 2) + 8 * n + 2 * tig] = o[n][0];
                rw[grp * (D + 2) + 8 * n + 2 * tig + 1] = o[n][1];
            }
            if (tig == 0) {
                rw[grp * (D + 2) + D] = m_run;
                rw[grp * (D + 2) + D + 1] = l_run;
            }
        }
        consumer_sync();
        float *rec = P.partials + (size_t)item * REC;
        for (int idx = threadIdx.x - 32; idx < G * D; idx += kWarps * 32) {
            const int h = idx / D, c = idx - h * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red[(w * 8 + h) * (D + 2) + D]);
            const float Mu = (M == -INFINITY) ? 0.0f : M;
            float acc = 0.0f, lsum = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float* rr = red + (w * 8 + h) * (D + 2);
                const float f = ex2(rr[D] - Mu);
                acc = fmaf(f, rr[c], acc);
                lsum = fmaf(f, rr[D + 1], lsum);
            }
            rec[h * (D + 2) + c] = acc;
            if (c == 0) {
                rec[h * (D + 2) + D] = M;
                rec[h * (D + 2) + D + 1] = lsum;
            }
        }
        consumer_sync();  // red is reused by the next item
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
    using L = DSmem<D>;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    const int n_items = p.B * p.Hkv * p.splits;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // caches viewed as [B*Hkv, Lmax, D]; box {64, 64 keys, 1}, 128-byte swizzle
    CUtensorMap tk, tv;
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.Lmax, (uint64_t)p.B * p.Hkv};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)p.Lmax * D * 2};
    const uint32_t box[3] = {64, (uint32_t)kChunk, 1};
    if (encode_tmap(&tk, p.k_cache, 3, dims, strides, box, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tv, p.v_cache, 3, dims, strides, box, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = decode_split_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    const int grid = n_items < sms ? n_items : sms;
    kern<<<grid, kThreads, L::ALLOC, stream>>>(tk, tv, p, scale_log2, n_items, err);
    e = cudaGetLastError();
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
    // Items = B*Hkv*splits are spread over num_sms persistent CTAs.  Pick the
    // split count that balances them best, with at least 4 chunks of keys per
    // item (the per-item merge costs about as much as one chunk).
    const int units = B * Hkv;
    const int chunks = (Lmax + kChunk - 1) / kChunk;
    const int max_s = chunks / 4 > 1 ? chunks / 4 : 1;
    int best = 1;
    double best_cost = 1e30;
    for (int s = 1; s <= max_s && s <= 256; ++s) {
        const long items = (long)units * s;
        const long waves = (items + num_sms - 1) / num_sms;
        const double per = (double)((chunks + s - 1) / s);        // chunks per item
        const double cost = waves * (per + 1.0);                  // + the item's merge
        if (cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
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
