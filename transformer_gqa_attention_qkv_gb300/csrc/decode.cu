// decode.cu -- split-KV grouped-query attention for one new token per
// sequence over a KV cache of bf16 values or of FP8 E4M3 codes with
// per-tensor scales ([T07] §4 steps 5-6: the cache returns the whole history
// and the new query attends to all of it; "Head Dimension" article §5.2: an
// FP8 K/V cache).
//
// The step reads every cached key and value once (2.1 GB for 64 sequences of
// 8193 tokens in bf16, half that in E4M3) and does ~4 flops per bf16 byte: it
// is bound by HBM bandwidth.  The design keeps ~150-190 KB per SM in flight
// and spends as few instructions per key as possible.
//
// Pass 1 (decode_split_kernel), persistent, one CTA per SM.  Work item =
// (sequence b, KV head g, split s): a contiguous range of that head's keys.
//   warp 0      TMA: the item's keys and values in chunks of 64 keys
//               (128-byte swizzled tiles), into a shared-memory ring, across
//               items without pausing;
//   warps 1..   consumer warps in groups of four.  The groups take the staged
//               chunks in turn (one group for bf16 caches; two for E4M3
//               caches, whose chunks carry half the bytes and would otherwise
//               leave the SM waiting on instruction latency); each warp of a
//               group takes 16 keys of its group's chunks.  The G query heads
//               sharing each K/V row are a genuine G x d by d x keys product,
//               computed with warp-level mma.sync m16n8k16 (heads in the M
//               rows, padded to 16): S = Q K^T with K fragments read by
//               ldmatrix from the swizzled tile; for bf16 caches the binary16
//               query is split into bf16 high and low parts (two MMAs) so no
//               query precision is lost; online softmax in the S accumulator
//               registers; the probabilities are already laid out as the A
//               fragment of O += P V, with V fragments from ldmatrix.trans.
//   At the end of an item the warps' (max, sum, unnormalised output) are
//   merged in shared memory into one fp32 partial record.
// Pass 2 (decode_combine_kernel): per (b, g), merge the splits by their
// log-sum-exp weights and write attn[b, j*d + c] in bf16.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kChunk = 64;     // keys per staged chunk
constexpr int kGroup = 4;      // consumer warps per chunk, 16 keys each

// F8: the caches hold one-byte E4M3 codes, so a 128-wide row is one 128-byte
// swizzled box row and a chunk is half the bytes (twice the stages in flight).
// CW consumer warps: CW / kGroup groups of four take the staged chunks in turn.
template <int D, bool F8 = false, int CW = kGroup>
struct DSmem {
    static constexpr int NCH = F8 ? 1 : D / 64;   // 128-byte boxes per row: 64-wide d halves, or all 128 codes
    static constexpr int BOX = kChunk * 128;       // one 64-key x 128-byte swizzled box (8 KB)
    static constexpr int CB = NCH * BOX;           // one K (or V) chunk
    // a multiple of the group count: stage s then always serves group s % (CW / kGroup),
    // so a group waiting for a stage's next fill has consumed its previous one
    static constexpr int STAGES = F8 ? 12 : (D == 128 ? 6 : 12);
    static constexpr int K = 0;
    static constexpr int V = STAGES * CB;
    static constexpr int RED = 2 * STAGES * CB;    // [CW][8][D + 2] floats
    static constexpr int BARS = RED + CW * 8 * (D + 2) * 4;
    static constexpr int TOTAL = BARS + 2 * STAGES * 8;
    static constexpr int ALLOC = TOTAL + 1024;
};

template <int CW>
DEVI void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory"); }

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

// Byte offset of code (key, byte) inside an E4M3 chunk of 128-byte rows.
DEVI uint32_t swz8(int key, int byte)
{
    return (uint32_t)(key * 128 + ((((byte >> 4) ^ (key & 7))) << 4) + (byte & 15));
}

DEVI uint32_t bf16x2_bits(float lo, float hi) { return pack_bf16(lo, hi); }

// F8 = false: bf16 caches, bf16 MMAs with the query and P split into high
// and low bf16 parts.  F8 = true: E4M3 caches, binary16 MMAs (E4M3 widens
// exactly to binary16, the binary16 query needs no split, P is split into
// binary16 high and low parts).  In the F8 path the 16 d-values of one
// k-step reach the K fragment in the order ldmatrix delivers 4-byte groups:
// MMA k-index 2t+e holds d = 4t+e and k-index 2t+8+e holds d = 4t+2+e
// (t = lane % 4); the query fragment uses the same order, which leaves the
// dot product unchanged.  V fragments come from a transposed ldmatrix whose
// 4 bytes (keys k, k+1 x d-values c, c+1) a byte permute splits into an
// even-d and an odd-d n-tile: output columns arrive interleaved and are put
// back in order when written to shared memory.
template <int D, int G, bool F8, int CW>
__global__ void __launch_bounds__(32 * (1 + CW), 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeAttentionProblem P, float scale_log2, int n_items, unsigned *err)
{
    static_assert(!F8 || D == 128, "E4M3 caches: 128-wide heads");
    static_assert(CW % kGroup == 0, "whole groups of four consumer warps");
    constexpr int NG = CW / kGroup;  // chunk it goes to group it % NG
    using L = DSmem<D, F8, CW>;
    static_assert(L::STAGES % NG == 0, "each ring stage must belong to one group (phase parity)");
    static_assert(L::ALLOC <= 232448, "shared memory per CTA");
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
    grid_dep_launch();  // the combine kernel may be scheduled meanwhile
    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kGroup);  // the four warps of the group that reads the stage
        }
        fence_mbar_init();
    }
    if (threadIdx.x == 32) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    __syncthreads();
    grid_dep_wait();  // q and the new cache entries come from the previous kernel

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

    const int cwi = warp - 1;           // consumer warp index (partials slot)
    const int grpi = cwi / kGroup;      // its group: chunks it with it % NG == grpi
    const int cw = cwi % kGroup;        // keys [16 cw, 16 cw + 16) of each of its chunks
    const int grp = lane >> 2, tig = lane & 3;
    const bool row_valid = grp < G;     // MMA row grp = query head g*G + grp
    // ldmatrix row addresses (relative to a chunk): lane i serves row i%8 of matrix i/8
    const int mi = lane >> 3, mr = lane & 7;
    const int qk_key = cw * 16 + (mi >> 1) * 8 + mr, qk_dofs = (mi & 1) * 8;  // K: (keys, d) blocks
    const int pv_key = cw * 16 + (mi & 1) * 8 + mr, pv_dofs = (mi >> 1) * 8;  // V: transposed blocks
    // E4M3: matrix mi covers keys 8*(mi&1).. of the warp and 16-byte block mi>>1 of the pair
    const int f8_key = cw * 16 + (mi & 1) * 8 + mr, f8_blk = mi >> 1;

    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const ItemRange r = item_range(P, item, err, false);
        // A fragments of Q (rows = heads of the group, binary16 split into bf16 hi + lo)
        uint32_t qh[KS][2], ql[KS][2];
        if constexpr (F8) {  // binary16 as it is, d in the fragment order described above
            const uint16_t *qrow = P.q + ((size_t)(r.b * P.Hq + r.g * G + (row_valid ? grp : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint2 v = make_uint2(0u, 0u);
                if (row_valid) v = *reinterpret_cast<const uint2 *>(qrow + ks * 16 + 4 * tig);
                qh[ks][0] = v.x;
                qh[ks][1] = v.y;
                ql[ks][0] = ql[ks][1] = 0u;
            }
        } else {
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
            if (NG > 1 && it % NG != grpi) continue;  // another group's chunk
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
            if constexpr (F8) {
                // four independent accumulators (n-tile x k-step parity) halve the MMA chains
                float sc2[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
                for (int kp = 0; kp < KS / 2; ++kp) {  // two k-steps (32 codes) per ldmatrix
                    uint32_t rk[4];  // (keys 0-7, k-step 2kp), (8-15, 2kp), (0-7, 2kp+1), (8-15, 2kp+1)
                    ldsm_x4(kb + swz8(f8_key, (2 * kp + f8_blk) * 16), rk[0], rk[1], rk[2], rk[3]);
                    uint32_t bk[4][2];
#pragma unroll
                    for (int m = 0; m < 4; ++m) e4m3x4_to_f16x4(rk[m], bk[m][0], bk[m][1]);
                    mma_f16_16816(sc[0], qh[2 * kp][0], 0u, qh[2 * kp][1], 0u, bk[0][0], bk[0][1]);
                    mma_f16_16816(sc[1], qh[2 * kp][0], 0u, qh[2 * kp][1], 0u, bk[1][0], bk[1][1]);
                    mma_f16_16816(sc2[0], qh[2 * kp + 1][0], 0u, qh[2 * kp + 1][1], 0u, bk[2][0], bk[2][1]);
                    mma_f16_16816(sc2[1], qh[2 * kp + 1][0], 0u, qh[2 * kp + 1][1], 0u, bk[3][0], bk[3][1]);
                }
#pragma unroll
                for (int n = 0; n < 2; ++n) {
                    sc[n][0] += sc2[n][0];
                    sc[n][1] += sc2[n][1];
                }
            } else {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t b00, b01, b10, b11;
                    ldsm_x4(kb + swz<D>(qk_key, ks * 16 + qk_dofs), b00, b01, b10, b11);
                    mma_bf16_16816(sc[0], qh[ks][0], 0u, qh[ks][1], 0u, b00, b01);
                    mma_bf16_16816(sc[1], qh[ks][0], 0u, qh[ks][1], 0u, b10, b11);
                    mma_bf16_16816(sc[0], ql[ks][0], 0u, ql[ks][1], 0u, b00, b01);
                    mma_bf16_16816(sc[1], ql[ks][0], 0u, ql[ks][1], 0u, b10, b11);
                }
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
            // F8: the running max moves only when a score passes it by more than
            // 2^8 (P then stays <= 2^8, exact in binary16's range), so O is
            // rescaled rarely; bf16: every time the max grows
            float m_new = fmaxf(m_run, mx);
            if (F8 && !(mx > m_run + 8.0f)) m_new = m_run;
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
            if (F8 && row_valid) {  // binary16 (11-bit significand), one MMA per tile
                a0h = pack_f16(p[0], p[1]);
                a2h = pack_f16(p[2], p[3]);
            } else if (row_valid) {
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(p[0], p[1]);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(p[2], p[3]);
                const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                a0h = *reinterpret_cast<const uint32_t *>(&h01);
                a2h = *reinterpret_cast<const uint32_t *>(&h23);
                a0l = bf16x2_bits(p[0] - f01.x, p[1] - f01.y);
                a2l = bf16x2_bits(p[2] - f23.x, p[3] - f23.y);
            }
            if (!F8 || __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    o[n][0] *= alpha;
                    o[n][1] *= alpha;
                }
            }
            if constexpr (F8) {
#pragma unroll
                for (int j2 = 0; j2 < D / 32; ++j2) {  // two 16-wide d blocks per ldmatrix
                    uint32_t rv[4];  // (keys 0-7, block 2j2), (8-15, 2j2), (0-7, 2j2+1), (8-15, 2j2+1)
                    ldsm_x4_trans(vb + swz8(f8_key, (2 * j2 + f8_blk) * 16), rv[0], rv[1], rv[2], rv[3]);
                    uint32_t bv[4][2];  // n-tiles 4 j2 .. 4 j2 + 3: (even d, odd d) of blocks 2 j2, 2 j2 + 1
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        // bytes (k c, k c+1, k+1 c, k+1 c+1) -> (k c, k+1 c | k c+1, k+1 c+1)
                        const uint32_t lo = prmt(rv[2 * x], 0u, 0x3120u), hi = prmt(rv[2 * x + 1], 0u, 0x3120u);
                        e4m3x4_to_f16x4(lo, bv[2 * x][0], bv[2 * x + 1][0]);
                        e4m3x4_to_f16x4(hi, bv[2 * x][1], bv[2 * x + 1][1]);
                    }
#pragma unroll
                    for (int n = 0; n < 4; ++n) mma_f16_16816(o[4 * j2 + n], a0h, 0u, a2h, 0u, bv[n][0], bv[n][1]);
                }
            } else {
#pragma unroll
                for (int nb = 0; nb < NT / 2; ++nb) {
                    uint32_t b0a, b1a, b0b, b1b;
                    ldsm_x4_trans(vb + swz<D>(pv_key, nb * 16 + pv_dofs), b0a, b1a, b0b, b1b);
                    mma_bf16_16816(o[2 * nb], a0h, 0u, a2h, 0u, b0a, b1a);
                    mma_bf16_16816(o[2 * nb + 1], a0h, 0u, a2h, 0u, b0b, b1b);
                    mma_bf16_16816(o[2 * nb], a0l, 0u, a2l, 0u, b0a, b1a);
                    mma_bf16_16816(o[2 * nb + 1], a0l, 0u, a2l, 0u, b0b, b1b);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
        }
        // row sum over the four lanes of a row; the max is already row-uniform
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
        float *rw = red + cwi * 8 * (D + 2);
        if (row_valid) {
            if constexpr (F8) {  // n-tile 2j: d = 16j + 4t + {0, 2}; n-tile 2j+1: d = 16j + 4t + {1, 3}
#pragma unroll
                for (int j = 0; j < NT / 2; ++j) {
                    float *dst = rw + grp * (D + 2) + 16 * j + 4 * tig;
                    dst[0] = o[2 * j][0];
                    dst[1] = o[2 * j + 1][0];
                    dst[2] = o[2 * j][1];
                    dst[3] = o[2 * j + 1][1];
                }
            } else {
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    rw[grp * (D + 2) + 8 * n + 2 * tig] = o[n][0];
                    rw[grp * (D + 2) + 8 * n + 2 * tig + 1] = o[n][1];
                }
            }
            if (tig == 0) {
                rw[grp * (D + 2) + D] = m_run;
                rw[grp * (D + 2) + D + 1] = l_run;
            }
        }
        consumer_sync<CW>();
        float *rec = P.partials + (size_t)item * REC;
        for (int idx = threadIdx.x - 32; idx < G * D; idx += CW * 32) {
            const int h = idx / D, c = idx - h * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < CW; ++w) M = fmaxf(M, red[(w * 8 + h) * (D + 2) + D]);
            const float Mu = (M == -INFINITY) ? 0.0f : M;
            float acc = 0.0f, lsum = 0.0f;
#pragma unroll
            for (int w = 0; w < CW; ++w) {
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
        consumer_sync<CW>();  // red is reused by the next item
    }
}

// One CTA per (b, g): merge the splits and write bf16 attn.
template <int D, int G>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeAttentionProblem P)
{
    constexpr int REC = G * (D + 2);
    grid_dep_launch();
    grid_dep_wait();  // the split kernel's partial records
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
        const float out = lsum > 0.0f ? acc / lsum * (P.fp8 ? P.v_scale : 1.0f) : 0.0f;
        const __nv_bfloat16 ob = __float2bfloat16_rn(out);
        P.out[(size_t)b * P.Hq * D + (size_t)(g * G + h) * D + c] = *reinterpret_cast<const uint16_t *>(&ob);
    }
}

template <int D, int G, bool F8, int CW = (F8 ? 8 : 4)>
cudaError_t run_decode(const DecodeAttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    using L = DSmem<D, F8, CW>;
    // E4M3 keys are code * k_scale: the scale joins the softmax scale
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D) * (F8 ? p.k_scale : 1.0f);
    const int n_items = p.B * p.Hkv * p.splits;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // caches viewed as [B*Hkv, Lmax, D]; box {128 bytes, 64 keys, 1}, 128-byte swizzle
    CUtensorMap tk, tv;
    const int eb = F8 ? 1 : 2;
    const uint64_t dims[3] = {(uint64_t)D, (uint64_t)p.Lmax, (uint64_t)p.B * p.Hkv};
    const uint64_t strides[2] = {(uint64_t)D * eb, (uint64_t)p.Lmax * D * eb};
    const uint32_t box[3] = {(uint32_t)(128 / eb), (uint32_t)kChunk, 1};
    if (encode_tmap(&tk, p.k_cache, 3, dims, strides, box, true, eb) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tv, p.v_cache, 3, dims, strides, box, true, eb) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = decode_split_kernel<D, G, F8, CW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    const int grid = n_items < sms ? n_items : sms;
    {
        LaunchCfg lc(dim3(grid), dim3(32 * (1 + CW)), L::ALLOC, stream, p.pdl != 0);
        e = cudaLaunchKernelEx(&lc.cfg, kern, tk, tv, p, scale_log2, n_items, err);
        if (e != cudaSuccess) return e;
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the combine follows the split kernel as its programmatic dependent
    LaunchCfg lc(dim3(p.B * p.Hkv), dim3(128), 0, stream, true);
    e = cudaLaunchKernelEx(&lc.cfg, decode_combine_kernel<D, G>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int D, bool F8>
cudaError_t run_decode_d(const DecodeAttentionProblem &p, unsigned *err, cudaStream_t stream)
{
    switch (p.Hq / p.Hkv) {
    case 1: return run_decode<D, 1, F8>(p, err, stream);
    case 2: return run_decode<D, 2, F8>(p, err, stream);
    case 4: return run_decode<D, 4, F8>(p, err, stream);
    case 8: return run_decode<D, 8, F8>(p, err, stream);
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
    if (p.fp8) return p.d == 128 ? run_decode_d<128, true>(p, err, stream) : cudaErrorInvalidValue;
    if (p.d == 128) return run_decode_d<128, false>(p, err, stream);
    if (p.d == 64) return run_decode_d<64, false>(p, err, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gqa
