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
// (sequence b, KV head g, split s, head sub-group): a contiguous range of that
// head's keys for up to GM of the query heads that share it.
//   warp 0      TMA: the item's keys and values in chunks of 64 keys
//               (128-byte swizzled tiles), into a shared-memory ring, across
//               items without pausing;
//   warps 1..   consumer warps in groups of four.  The groups take the staged
//               chunks in turn (one group for bf16 caches; three for E4M3
//               caches, whose chunks carry half the bytes and would otherwise
//               leave the SM waiting on instruction latency); each warp of a
//               group takes 16 keys of its group's chunks.  The query heads
//               sharing each K/V row make it a genuine heads x d by d x keys
//               product, computed with warp-level mma.sync m16n8k16:
//     bf16 caches, groups of up to 8 heads (GM = 8): transposed products,
//               S^T = K Q^T (16 keys in the MMA rows, the heads in its 8
//               columns) and O^T = V^T P^T (d in the rows), K the A fragment
//               straight from ldmatrix, V^T from ldmatrix.trans, P^T reaching
//               the B-fragment layout by an 8x8 transpose (movmatrix); the
//               binary16 query and P are split into bf16 high and low parts
//               (two MMAs each) so no precision is lost;
//     bf16 caches, 9 to 16 heads (GM = 16): heads in the MMA's 16 rows,
//               S = Q K^T, online softmax in the S accumulator registers,
//               whose layout is already the A fragment of O += P V (q and P
//               split the same way), V fragments from ldmatrix.trans;
//     E4M3 caches: the transposed products of the first form (up to GM = 8
//               heads); E4M3 widens exactly to binary16, so the MMAs are
//               binary16 and the query needs no split.  Rows of 64, 80 or 96
//               codes are staged as 128 codes (the tensor copy fills the rest
//               with zeros, the query is zero-padded alike, and the partial
//               records keep the real width); rows of 256 codes are two
//               128-byte boxes, taken by one group of consumer warps.
//   Online softmax in the accumulator registers in every form.
//   At the end of an item the warps' (max, sum, unnormalised output) are
//   merged in shared memory into one fp32 partial record.
// A group of more than GM query heads is taken as vsub sub-groups of G / vsub
// heads each; the sub-groups of one key range are consecutive work items, so
// they run at the same time on neighbouring SMs and the second read of each
// chunk comes from L2.
// Pass 2 (decode_combine_kernel): per (b, sub-group), merge the splits by
// their log-sum-exp weights and write attn[b, j*d + c] in bf16.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kChunk = 64;     // keys per staged chunk
constexpr int kGroup = 4;      // consumer warps per chunk, 16 keys each

// F8: the caches hold one-byte E4M3 codes, so a 128-wide row is one 128-byte
// swizzled box row and a chunk is half the bytes (twice the stages in flight).
// bf16 rows are NCH boxes of 64 values; at head widths 80 and 96 the second
// box is zero-filled past d by the tensor copy (dims end at d), and the
// products run over the d real columns only.
// CW consumer warps: CW / kGroup groups of four take the staged chunks in turn.
// GM: query heads per work item (rows of the per-warp partials).
template <int D, int GM, bool F8 = false, int CW = kGroup>
struct DSmem {
    static constexpr int NCH = F8 ? D / 128 : (D + 63) / 64;  // 128-byte boxes per row: 64-wide d chunks, or 128 codes
    static constexpr int BOX = kChunk * 128;       // one 64-key x 128-byte swizzled box (8 KB)
    static constexpr int CB = NCH * BOX;           // one K (or V) chunk
    // a multiple of the group count: stage s then always serves group s % (CW / kGroup),
    // so a group waiting for a stage's next fill has consumed its previous one
    static constexpr int STAGES = F8 ? (NCH == 2 ? 6 : CW == 12 ? 9 : 12) : (NCH == 4 ? 3 : NCH == 2 ? 6 : 12);
    static constexpr int K = 0;
    static constexpr int V = STAGES * CB;
    static constexpr int RED = 2 * STAGES * CB;    // [CW][GM][D + 2] floats
    static constexpr int BARS = RED + CW * GM * (D + 2) * 4;
    static constexpr int TOTAL = BARS + 2 * STAGES * 8;
    static constexpr int ALLOC = TOTAL + 1024;
};

template <int CW>
DEVI void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(CW * 32) : "memory"); }

// One work item: keys [begin, end) of cache head g of sequence b, for the
// query heads vg*Gv .. vg*Gv + Gv - 1 (vg = g*vsub + sub); its partial record
// is number rec.
struct ItemRange {
    int b, g, vg, rec, begin, end;
};

DEVI ItemRange item_range(const DecodeAttentionProblem &P, int item, unsigned *err, bool report)
{
    ItemRange r;
    const int vsub = P.vsub;
    const int sub = item % vsub;
    const int t = item / vsub;
    const int s = t % P.splits;
    const int bg = t / P.splits;
    r.b = bg / P.Hkv;
    r.g = bg - r.b * P.Hkv;
    r.vg = r.g * vsub + sub;
    r.rec = (bg * vsub + sub) * P.splits + s;
    int len = P.len[r.b] + P.len_bias;
    if (len < 1 || len > P.Lmax) {
        if (report) atomicOr(err, kErrIndex);
        len = 0;
    }
    const int chunks = (len + kChunk - 1) / kChunk;
    const int per = (chunks + P.splits - 1) / P.splits;
    const int c0 = min(chunks, s * per), c1 = min(chunks, c0 + per);
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
    return (uint32_t)((dcol >> 6) * DSmem<D, 8>::BOX + key * 128 + ((((dcol & 63) >> 3) ^ (key & 7)) << 4));
}

// Byte offset of code (key, byte) inside an E4M3 chunk of 128-byte rows.
DEVI uint32_t swz8(int key, int byte)
{
    return (uint32_t)(key * 128 + ((((byte >> 4) ^ (key & 7))) << 4) + (byte & 15));
}

// Byte offset of 16-byte block blk (codes 16 blk ..) of key `key` inside an
// E4M3 chunk stored as 128-byte boxes (rows of 256 codes take two).
DEVI uint32_t f8_off(int key, int blk)
{
    return (uint32_t)((blk >> 3) * (kChunk * 128)) + swz8(key, (blk & 7) * 16);
}

DEVI uint32_t bf16x2_bits(float lo, float hi) { return pack_bf16(lo, hi); }

// Transpose of an 8x8 matrix of 16-bit elements held as the warp's A/C
// fragment rows (lane: row lane/4, elements 2(lane%4), +1).
DEVI uint32_t movmatrix_t(uint32_t x)
{
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// bf16 high part of (lo, hi) and the bf16 of what it leaves over.
DEVI void split_bf16(float lo, float hi, uint32_t &h, uint32_t &l)
{
    const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    const float2 f = __bfloat1622float2(b);
    h = *reinterpret_cast<const uint32_t *>(&b);
    l = bf16x2_bits(lo - f.x, hi - f.y);
}

// Value rows past the item's last key may hold anything (slots past the
// sequence are not initialised); 0 * NaN would poison O, so the rows of this
// warp's 16 keys at or past `end` are zeroed.  Masked scores need no such care.
template <int NCH>
DEVI void zero_v_tail(uint8_t *vchunk, int u0, int end, int cw, int lane)
{
    const int first = max(end - u0, cw * 16);
    uint4 *vrow = reinterpret_cast<uint4 *>(vchunk);
    for (int idx = lane; idx < (cw * 16 + 16 - first) * NCH * 8; idx += 32) {
        const int key = first + idx / (NCH * 8), rem = idx % (NCH * 8);
        vrow[((rem >> 3) * (kChunk * 128) + key * 128) / 16 + (rem & 7)] = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
}

// One step of the online softmax for the four scores a lane holds of one
// query row (keys kbase, +1, +8, +9; scaled to log2 units, masked ones
// -inf): the row max over the four lanes of the row, the rescale factor of the
// running sums and the probabilities.  lazy: the running max moves only when a
// score passes it by more than 2^8 (P then stays <= 2^8), so O is rescaled
// rarely; otherwise it moves whenever the max grows.
template <bool LAZY>
DEVI void softmax_step(const float (&v)[4], float &m_run, float &l_run, float &alpha, float (&p)[4])
{
    float mx = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    float m_new = fmaxf(m_run, mx);
    if (LAZY && !(mx > m_run + 8.0f)) m_new = m_run;
    const float m_use = (m_new == -INFINITY) ? 0.0f : m_new;
    alpha = ex2(m_run - m_use);
    m_run = m_new;
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = (v[e] == -INFINITY) ? 0.0f : ex2(v[e] - m_use);
    l_run = l_run * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
}

// Merge of the consumer warps' per-head (o, max, sum) rows in `red` into the
// item's partial record: o = sum_w 2^(m_w - M) o_w, l likewise, M = max_w m_w.
// Records hold the DR real columns of each head (DR < D: rows staged wider,
// with zero columns past DR).
template <int D, int GM, int CW, int DR = D>
DEVI void write_record(const float *red, float *rec, int Gv)
{
    for (int idx = threadIdx.x - 32; idx < Gv * DR; idx += CW * 32) {
        const int h = idx / DR, c = idx - h * DR;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < CW; ++w) M = fmaxf(M, red[(w * GM + h) * (D + 2) + D]);
        const float Mu = (M == -INFINITY) ? 0.0f : M;
        float acc = 0.0f, lsum = 0.0f;
#pragma unroll
        for (int w = 0; w < CW; ++w) {
            const float *rr = red + (w * GM + h) * (D + 2);
            const float f = ex2(rr[D] - Mu);
            acc = fmaf(f, rr[c], acc);
            lsum = fmaf(f, rr[D + 1], lsum);
        }
        rec[h * (DR + 2) + c] = acc;
        if (c == 0) {
            rec[h * (DR + 2) + DR] = M;
            rec[h * (DR + 2) + DR + 1] = lsum;
        }
    }
}

// Consumer warps over bf16 caches: heads in the MMA rows (row grp: head grp,
// row grp + 8: head grp + 8 when GM = 16), bf16 MMAs with the query and P
// split into high and low bf16 parts.
template <int D, int GM, int CW>
DEVI void consume_bf16(const DecodeAttentionProblem &P, uint8_t *smem, uint64_t *full, uint64_t *empty, float *red,
                       float scale_log2, int n_items, unsigned *err)
{
    using L = DSmem<D, GM, false, CW>;
    static_assert(CW == kGroup, "bf16 caches: one group of four consumer warps");
    static_assert(GM == 8 || GM == 16, "8 or 16 heads per item");
    constexpr bool TWO = GM > 8;  // MMA rows 8..15 carry heads 8..15
    constexpr int ST = L::STAGES;
    constexpr int KS = D / 16;    // k-steps of the QK product
    constexpr int NT = D / 8;     // n-tiles of the PV product
    const int Gv = P.Hq / P.Hkv / P.vsub;
    const int lane = threadIdx.x % 32;
    const int cw = threadIdx.x / 32 - 1;  // keys [16 cw, 16 cw + 16) of each chunk
    const int grp = lane >> 2, tig = lane & 3;
    const bool va = grp < Gv, vb = TWO && grp + 8 < Gv;
    // ldmatrix row addresses (relative to a chunk): lane i serves row i%8 of matrix i/8
    const int mi = lane >> 3, mr = lane & 7;
    const int qk_key = cw * 16 + (mi >> 1) * 8 + mr, qk_dofs = (mi & 1) * 8;  // K: (keys, d) blocks
    const int pv_key = cw * 16 + (mi & 1) * 8 + mr, pv_dofs = (mi >> 1) * 8;  // V: transposed blocks

    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const ItemRange r = item_range(P, item, err, false);
        const uint16_t *qbase = P.q + (size_t)(r.b * P.Hq + r.vg * Gv) * D;
        // A fragments of Q: [0] row grp, k 2t..; [1] row grp+8, k 2t..; [2] row grp, k 2t+8..;
        // [3] row grp+8, k 2t+8.. (binary16 split into bf16 hi + lo)
        uint32_t qh[KS][4], ql[KS][4];
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float2 f = make_float2(0.0f, 0.0f);
                if (va) f = __half22float2(*reinterpret_cast<const __half2 *>(qbase + grp * D + ks * 16 + half * 8 + 2 * tig));
                split_bf16(f.x, f.y, qh[ks][2 * half], ql[ks][2 * half]);
                qh[ks][2 * half + 1] = ql[ks][2 * half + 1] = 0u;
                if (TWO && vb) {
                    f = __half22float2(
                        *reinterpret_cast<const __half2 *>(qbase + (grp + 8) * D + ks * 16 + half * 8 + 2 * tig));
                    split_bf16(f.x, f.y, qh[ks][2 * half + 1], ql[ks][2 * half + 1]);
                }
            }
        float o[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.0f;
        float mA = -INFINITY, lA = 0.0f, mB = -INFINITY, lB = 0.0f;  // rows grp, grp + 8

        for (int u0 = r.begin; u0 < r.end; u0 += kChunk, ++it) {
            const int s = it % ST;
            if (!mbar_wait(full + s, (it / ST) & 1, err)) break;
            const uint32_t kb = smem_u32(smem + L::K + s * L::CB);
            const uint32_t vbase = smem_u32(smem + L::V + s * L::CB);
            if (u0 + kChunk > r.end) zero_v_tail<L::NCH>(smem + L::V + s * L::CB, u0, r.end, cw, lane);
            // S[heads x 16 keys] = Q K^T
            float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t b00, b01, b10, b11;
                ldsm_x4(kb + swz<D>(qk_key, ks * 16 + qk_dofs), b00, b01, b10, b11);
                mma_bf16_16816(sc[0], qh[ks][0], qh[ks][1], qh[ks][2], qh[ks][3], b00, b01);
                mma_bf16_16816(sc[1], qh[ks][0], qh[ks][1], qh[ks][2], qh[ks][3], b10, b11);
                mma_bf16_16816(sc[0], ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3], b00, b01);
                mma_bf16_16816(sc[1], ql[ks][0], ql[ks][1], ql[ks][2], ql[ks][3], b10, b11);
            }
            // this lane's keys: kbase, +1 (n-tile 0) and kbase + 8, +9 (n-tile 1)
            const int kbase = u0 + cw * 16 + 2 * tig;
            const bool k0 = kbase < r.end, k1 = kbase + 1 < r.end, k8 = kbase + 8 < r.end, k9 = kbase + 9 < r.end;
            const float vA[4] = {k0 ? sc[0][0] * scale_log2 : -INFINITY, k1 ? sc[0][1] * scale_log2 : -INFINITY,
                                 k8 ? sc[1][0] * scale_log2 : -INFINITY, k9 ? sc[1][1] * scale_log2 : -INFINITY};
            float pA[4], aA;
            softmax_step<false>(vA, mA, lA, aA, pA);
            // P as the A fragment of O += P V, split into bf16 high and low parts
            uint32_t a0h = 0u, a2h = 0u, a0l = 0u, a2l = 0u, a1h = 0u, a3h = 0u, a1l = 0u, a3l = 0u;
            if (va) {
                split_bf16(pA[0], pA[1], a0h, a0l);
                split_bf16(pA[2], pA[3], a2h, a2l);
            }
            float aB = 1.0f;
            if constexpr (TWO) {
                const float vB[4] = {k0 ? sc[0][2] * scale_log2 : -INFINITY, k1 ? sc[0][3] * scale_log2 : -INFINITY,
                                     k8 ? sc[1][2] * scale_log2 : -INFINITY, k9 ? sc[1][3] * scale_log2 : -INFINITY};
                float pB[4];
                softmax_step<false>(vB, mB, lB, aB, pB);
                if (vb) {
                    split_bf16(pB[0], pB[1], a1h, a1l);
                    split_bf16(pB[2], pB[3], a3h, a3l);
                }
            }
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                o[n][0] *= aA;
                o[n][1] *= aA;
                if (TWO) {
                    o[n][2] *= aB;
                    o[n][3] *= aB;
                }
            }
#pragma unroll
            for (int nb = 0; nb < NT / 2; ++nb) {
                uint32_t b0a, b1a, b0b, b1b;
                ldsm_x4_trans(vbase + swz<D>(pv_key, nb * 16 + pv_dofs), b0a, b1a, b0b, b1b);
                mma_bf16_16816(o[2 * nb], a0h, a1h, a2h, a3h, b0a, b1a);
                mma_bf16_16816(o[2 * nb + 1], a0h, a1h, a2h, a3h, b0b, b1b);
                mma_bf16_16816(o[2 * nb], a0l, a1l, a2l, a3l, b0a, b1a);
                mma_bf16_16816(o[2 * nb + 1], a0l, a1l, a2l, a3l, b0b, b1b);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
        }
        // row sums over the four lanes of a row; the maxima are already row-uniform
        lA += __shfl_xor_sync(0xffffffffu, lA, 1);
        lA += __shfl_xor_sync(0xffffffffu, lA, 2);
        lB += __shfl_xor_sync(0xffffffffu, lB, 1);
        lB += __shfl_xor_sync(0xffffffffu, lB, 2);
        float *rw = red + cw * GM * (D + 2);
        if (va) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                rw[grp * (D + 2) + 8 * n + 2 * tig] = o[n][0];
                rw[grp * (D + 2) + 8 * n + 2 * tig + 1] = o[n][1];
            }
            if (tig == 0) {
                rw[grp * (D + 2) + D] = mA;
                rw[grp * (D + 2) + D + 1] = lA;
            }
        }
        if (TWO && vb) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                rw[(grp + 8) * (D + 2) + 8 * n + 2 * tig] = o[n][2];
                rw[(grp + 8) * (D + 2) + 8 * n + 2 * tig + 1] = o[n][3];
            }
            if (tig == 0) {
                rw[(grp + 8) * (D + 2) + D] = mB;
                rw[(grp + 8) * (D + 2) + D + 1] = lB;
            }
        }
        consumer_sync<CW>();
        write_record<D, GM, CW>(red, P.partials + (size_t)r.rec * Gv * (D + 2), Gv);
        consumer_sync<CW>();  // red is reused by the next item
    }
}

// Consumer warps over bf16 caches for groups of up to 8 heads, transposed
// products: S^T = K Q^T (16 keys in the MMA rows, the heads in its 8 columns)
// and O^T = V^T P^T (16 values of d in the rows), so one m16n8k16 covers 16
// keys x 8 heads and O takes D/16 x 4 registers (heads-in-rows needs twice
// both).  K is the A fragment straight from ldmatrix; V^T from ldmatrix.trans;
// the binary16 query (the B fragment of S^T) and P (the B fragment of O^T,
// reached through an 8x8 movmatrix transpose) are split into bf16 high and low
// parts, two MMAs each, so no precision is lost.  A lane holds the scores of
// keys grp and grp + 8 for heads 2 tig and 2 tig + 1.
template <int D, int CW>
DEVI void consume_bf16_t(const DecodeAttentionProblem &P, uint8_t *smem, uint64_t *full, uint64_t *empty,
                         float *red, float scale_log2, int n_items, unsigned *err)
{
    constexpr int GM = 8;
    using L = DSmem<D, GM, false, CW>;
    static_assert(CW == kGroup, "bf16 caches: one group of four consumer warps");
    static_assert(D % 16 == 0, "16-wide k-steps and d blocks");
    constexpr int ST = L::STAGES;
    constexpr int KS = D / 16;  // k-steps of S^T, and 16-row d blocks of O^T
    const int Gv = P.Hq / P.Hkv / P.vsub;
    const int lane = threadIdx.x % 32;
    const int cw = threadIdx.x / 32 - 1;  // keys [16 cw, 16 cw + 16) of each chunk
    const int grp = lane >> 2, tig = lane & 3;
    const bool head_valid = grp < Gv;     // B-fragment column grp = query head vg*Gv + grp
    // ldmatrix: matrix mi covers keys 8*(mi&1).. and d block (mi>>1) (K, the A fragment),
    // and keys 8*(mi>>1).. of d block (mi&1) (V, read transposed as the A fragment of O^T)
    const int mi = lane >> 3, mr = lane & 7;
    const int k_key = cw * 16 + (mi & 1) * 8 + mr, k_dofs = (mi >> 1) * 8;
    const int v_key = cw * 16 + (mi >> 1) * 8 + mr, v_dofs = (mi & 1) * 8;

    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const ItemRange r = item_range(P, item, err, false);
        // B fragments of Q^T: [0] d 2t, 2t+1 and [1] d 2t+8, 2t+9 of k-step ks, head grp
        uint32_t qh[KS][2], ql[KS][2];
        const uint16_t *qrow = P.q + (size_t)(r.b * P.Hq + r.vg * Gv + (head_valid ? grp : 0)) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float2 f = make_float2(0.0f, 0.0f);
                if (head_valid) f = __half22float2(*reinterpret_cast<const __half2 *>(qrow + ks * 16 + half * 8 + 2 * tig));
                split_bf16(f.x, f.y, qh[ks][half], ql[ks][half]);
            }
        float o[KS][4];  // d block b: c0/c1 d = 16b + grp (heads 2t, 2t+1), c2/c3 d = 16b + grp + 8
#pragma unroll
        for (int b = 0; b < KS; ++b) o[b][0] = o[b][1] = o[b][2] = o[b][3] = 0.0f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // heads 2 tig, 2 tig + 1

        for (int u0 = r.begin; u0 < r.end; u0 += kChunk, ++it) {
            const int s = it % ST;
            if (!mbar_wait(full + s, (it / ST) & 1, err)) break;
            const uint32_t kb = smem_u32(smem + L::K + s * L::CB);
            const uint32_t vb = smem_u32(smem + L::V + s * L::CB);
            if (u0 + kChunk > r.end) zero_v_tail<L::NCH>(smem + L::V + s * L::CB, u0, r.end, cw, lane);
            // S^T [16 keys x 8 heads], two accumulators (k-step parity)
            float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kb + swz<D>(k_key, ks * 16 + k_dofs), a0, a1, a2, a3);
                mma_bf16_16816(sc[ks & 1], a0, a1, a2, a3, qh[ks][0], qh[ks][1]);
                mma_bf16_16816(sc[ks & 1], a0, a1, a2, a3, ql[ks][0], ql[ks][1]);
            }
            const int ka = u0 + cw * 16 + grp;  // this lane's keys: ka, ka + 8
            const float v0 = (ka < r.end) ? (sc[0][0] + sc[1][0]) * scale_log2 : -INFINITY;      // head 2t
            const float v1 = (ka < r.end) ? (sc[0][1] + sc[1][1]) * scale_log2 : -INFINITY;      // head 2t+1
            const float v2 = (ka + 8 < r.end) ? (sc[0][2] + sc[1][2]) * scale_log2 : -INFINITY;  // head 2t
            const float v3 = (ka + 8 < r.end) ? (sc[0][3] + sc[1][3]) * scale_log2 : -INFINITY;  // head 2t+1
            float x0 = fmaxf(v0, v2), x1 = fmaxf(v1, v3);
#pragma unroll
            for (int sh = 4; sh <= 16; sh <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, sh));
                x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, sh));
            }
            // the running max moves only past a 2^8 growth, so O is rescaled rarely
            const float n0 = (x0 > m0 + 8.0f) ? fmaxf(m0, x0) : m0;
            const float n1 = (x1 > m1 + 8.0f) ? fmaxf(m1, x1) : m1;
            const float u0m = (n0 == -INFINITY) ? 0.0f : n0, u1m = (n1 == -INFINITY) ? 0.0f : n1;
            const float a0s = ex2(m0 - u0m), a1s = ex2(m1 - u1m);
            m0 = n0;
            m1 = n1;
            const float p0 = (v0 == -INFINITY) ? 0.0f : ex2(v0 - u0m);
            const float p1 = (v1 == -INFINITY) ? 0.0f : ex2(v1 - u1m);
            const float p2 = (v2 == -INFINITY) ? 0.0f : ex2(v2 - u0m);
            const float p3 = (v3 == -INFINITY) ? 0.0f : ex2(v3 - u1m);
            l0 = l0 * a0s + (p0 + p2);
            l1 = l1 * a1s + (p1 + p3);
            // P^T as the B fragment (high and low bf16 parts): transpose the (key x head) 8x8 blocks
            uint32_t h01, l01, h23, l23;
            split_bf16(p0, p1, h01, l01);
            split_bf16(p2, p3, h23, l23);
            const uint32_t pbh0 = movmatrix_t(h01), pbh1 = movmatrix_t(h23);
            const uint32_t pbl0 = movmatrix_t(l01), pbl1 = movmatrix_t(l23);
            if (__any_sync(0xffffffffu, a0s != 1.0f || a1s != 1.0f)) {
#pragma unroll
                for (int b = 0; b < KS; ++b) {
                    o[b][0] *= a0s;
                    o[b][1] *= a1s;
                    o[b][2] *= a0s;
                    o[b][3] *= a1s;
                }
            }
#pragma unroll
            for (int b = 0; b < KS; ++b) {
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(vb + swz<D>(v_key, b * 16 + v_dofs), a0, a1, a2, a3);
                mma_bf16_16816(o[b], a0, a1, a2, a3, pbh0, pbh1);
                mma_bf16_16816(o[b], a0, a1, a2, a3, pbl0, pbl1);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
        }
        // sums over the eight lanes of a head column; the max is already uniform there
#pragma unroll
        for (int sh = 4; sh <= 16; sh <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
            l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
        }
        float *rw = red + cw * GM * (D + 2);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * tig + e;
            if (h < Gv) {
                float *dst = rw + h * (D + 2);
#pragma unroll
                for (int b = 0; b < KS; ++b) {
                    dst[16 * b + grp] = o[b][e];
                    dst[16 * b + grp + 8] = o[b][2 + e];
                }
                if (grp == 0) {
                    dst[D] = e ? m1 : m0;
                    dst[D + 1] = e ? l1 : l0;
                }
            }
        }
        consumer_sync<CW>();
        write_record<D, GM, CW>(red, P.partials + (size_t)r.rec * Gv * (D + 2), Gv);
        consumer_sync<CW>();  // red is reused by the next item
    }
}

// Consumer warps over E4M3 caches: transposed products with the group's heads
// in the MMA's 8 columns (GM = 8), binary16 MMAs.  In the S^T product the 16
// d-values of one k-step reach the K (A) fragment in the order ldmatrix
// delivers 4-byte groups: MMA k-index 2t+e holds d = 4t+e and k-index 2t+8+e
// holds d = 4t+2+e (t = lane % 4); the query (B) fragment uses the same order,
// which leaves the dot product unchanged.  V fragments come from a transposed
// ldmatrix whose 4 bytes (keys k, k+1 x d-values c, c+1) a byte permute splits
// into an even-d and an odd-d half: rows of O^T arrive interleaved (m-tile b
// holds d = 16b + 2grp and 16b + 2grp + 1) and are put back in order when
// written to shared memory.  P stays <= 2^8 (lazy running max), exact in
// binary16's range, so O is rescaled rarely.
template <int D, int CW, int DR = D>
DEVI void consume_f8(const DecodeAttentionProblem &P, uint8_t *smem, uint64_t *full, uint64_t *empty, float *red,
                     float scale_log2, int n_items, unsigned *err)
{
    constexpr int GM = 8;
    using L = DSmem<D, GM, true, CW>;
    static_assert(D == 128 || D == 256, "E4M3 caches: rows of one or two 128-code boxes");
    static_assert(DR <= D && DR % 16 == 0, "real head width");
    constexpr int NG = CW / kGroup;  // chunk it goes to group it % NG
    static_assert(L::STAGES % NG == 0, "each ring stage must belong to one group (phase parity)");
    constexpr int ST = L::STAGES;
    constexpr int KS = D / 16;
    const int Gv = P.Hq / P.Hkv / P.vsub;
    const int lane = threadIdx.x % 32;
    const int cwi = threadIdx.x / 32 - 1;  // consumer warp index (partials slot)
    const int grpi = cwi / kGroup;         // its group: chunks it with it % NG == grpi
    const int cw = cwi % kGroup;           // keys [16 cw, 16 cw + 16) of each of its chunks
    const int grp = lane >> 2, tig = lane & 3;
    const bool head_valid = grp < Gv;      // B-fragment column grp = query head vg*Gv + grp
    // matrix mi of an ldmatrix covers keys 8*(mi&1).. of the warp and 16-byte block mi>>1 of the pair
    const int mi = lane >> 3, mr = lane & 7;
    const int f8_key = cw * 16 + (mi & 1) * 8 + mr, f8_blk = mi >> 1;

    int it = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
        const ItemRange r = item_range(P, item, err, false);
        // B fragments of Q^T, d in the order described above
        uint32_t qb[KS][2];
        const uint16_t *qrow = P.q + (size_t)(r.b * P.Hq + r.vg * Gv + (head_valid ? grp : 0)) * DR;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint2 v = make_uint2(0u, 0u);  // zero past the real width (the staged codes there are zero too)
            if (head_valid && ks * 16 < DR) v = *reinterpret_cast<const uint2 *>(qrow + ks * 16 + 4 * tig);
            qb[ks][0] = v.x;
            qb[ks][1] = v.y;
        }
        float o[D / 16][4];  // m-tile b: rows d = 16b + 2grp (c0, c1) and 16b + 2grp + 1 (c2, c3)
#pragma unroll
        for (int b = 0; b < D / 16; ++b) o[b][0] = o[b][1] = o[b][2] = o[b][3] = 0.0f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;  // heads 2 tig, 2 tig + 1

        for (int u0 = r.begin; u0 < r.end; u0 += kChunk, ++it) {
            if (NG > 1 && it % NG != grpi) continue;  // another group's chunk
            const int s = it % ST;
            if (!mbar_wait(full + s, (it / ST) & 1, err)) break;
            const uint32_t kb = smem_u32(smem + L::K + s * L::CB);
            const uint32_t vb = smem_u32(smem + L::V + s * L::CB);
            if (u0 + kChunk > r.end) zero_v_tail<L::NCH>(smem + L::V + s * L::CB, u0, r.end, cw, lane);
            // S^T [16 keys x 8 heads], two accumulators (k-step parity)
            float sc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
                uint32_t rk[4];  // (keys 0-7, block 2kp), (8-15, 2kp), (0-7, 2kp+1), (8-15, 2kp+1)
                ldsm_x4(kb + f8_off(f8_key, 2 * kp + f8_blk), rk[0], rk[1], rk[2], rk[3]);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    uint32_t lo0, hi0, lo1, hi1;
                    e4m3x4_to_f16x4(rk[2 * j], lo0, hi0);
                    e4m3x4_to_f16x4(rk[2 * j + 1], lo1, hi1);
                    mma_f16_16816(sc[j], lo0, lo1, hi0, hi1, qb[2 * kp + j][0], qb[2 * kp + j][1]);
                }
            }
            const int ka = u0 + cw * 16 + grp;  // this lane's keys: ka, ka + 8
            const float v0 = (ka < r.end) ? (sc[0][0] + sc[1][0]) * scale_log2 : -INFINITY;      // head 2t
            const float v1 = (ka < r.end) ? (sc[0][1] + sc[1][1]) * scale_log2 : -INFINITY;      // head 2t+1
            const float v2 = (ka + 8 < r.end) ? (sc[0][2] + sc[1][2]) * scale_log2 : -INFINITY;  // head 2t
            const float v3 = (ka + 8 < r.end) ? (sc[0][3] + sc[1][3]) * scale_log2 : -INFINITY;  // head 2t+1
            float x0 = fmaxf(v0, v2), x1 = fmaxf(v1, v3);
#pragma unroll
            for (int sh = 4; sh <= 16; sh <<= 1) {
                x0 = fmaxf(x0, __shfl_xor_sync(0xffffffffu, x0, sh));
                x1 = fmaxf(x1, __shfl_xor_sync(0xffffffffu, x1, sh));
            }
            // the running max moves only past a 2^8 growth (P <= 2^8 in binary16)
            const float n0 = (x0 > m0 + 8.0f) ? fmaxf(m0, x0) : m0;
            const float n1 = (x1 > m1 + 8.0f) ? fmaxf(m1, x1) : m1;
            const float u0m = (n0 == -INFINITY) ? 0.0f : n0, u1m = (n1 == -INFINITY) ? 0.0f : n1;
            const float a0 = ex2(m0 - u0m), a1 = ex2(m1 - u1m);
            m0 = n0;
            m1 = n1;
            const float p0 = (v0 == -INFINITY) ? 0.0f : ex2(v0 - u0m);
            const float p1 = (v1 == -INFINITY) ? 0.0f : ex2(v1 - u1m);
            const float p2 = (v2 == -INFINITY) ? 0.0f : ex2(v2 - u0m);
            const float p3 = (v3 == -INFINITY) ? 0.0f : ex2(v3 - u1m);
            l0 = l0 * a0 + (p0 + p2);
            l1 = l1 * a1 + (p1 + p3);
            // P^T as the B fragment: transpose the (key x head) 8x8 blocks
            const uint32_t pb0 = movmatrix_t(pack_f16(p0, p1)), pb1 = movmatrix_t(pack_f16(p2, p3));
            if (__any_sync(0xffffffffu, a0 != 1.0f || a1 != 1.0f)) {
#pragma unroll
                for (int b = 0; b < D / 16; ++b) {
                    o[b][0] *= a0;
                    o[b][1] *= a1;
                    o[b][2] *= a0;
                    o[b][3] *= a1;
                }
            }
#pragma unroll
            for (int j2 = 0; j2 < D / 32; ++j2) {
                uint32_t rv[4];  // (keys 0-7, block 2j2), (8-15, 2j2), (0-7, 2j2+1), (8-15, 2j2+1)
                ldsm_x4_trans(vb + f8_off(f8_key, 2 * j2 + f8_blk), rv[0], rv[1], rv[2], rv[3]);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    // bytes (k c, k c+1, k+1 c, k+1 c+1) -> (k c, k+1 c | k c+1, k+1 c+1)
                    uint32_t lo0, hi0, lo1, hi1;
                    e4m3x4_to_f16x4(prmt(rv[2 * x], 0u, 0x3120u), lo0, hi0);
                    e4m3x4_to_f16x4(prmt(rv[2 * x + 1], 0u, 0x3120u), lo1, hi1);
                    mma_f16_16816(o[2 * j2 + x], lo0, hi0, lo1, hi1, pb0, pb1);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + s);
        }
        // sums over the eight lanes of a head column; the max is already uniform there
#pragma unroll
        for (int sh = 4; sh <= 16; sh <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, sh);
            l1 += __shfl_xor_sync(0xffffffffu, l1, sh);
        }
        float *rw = red + cwi * GM * (D + 2);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * tig + e;
            if (h < Gv) {
                float *dst = rw + h * (D + 2);
#pragma unroll
                for (int b = 0; b < D / 16; ++b) {
                    dst[16 * b + 2 * grp] = o[b][e];
                    dst[16 * b + 2 * grp + 1] = o[b][2 + e];
                }
                if (grp == 0) {
                    dst[D] = e ? m1 : m0;
                    dst[D + 1] = e ? l1 : l0;
                }
            }
        }
        consumer_sync<CW>();
        write_record<D, GM, CW, DR>(red, P.partials + (size_t)r.rec * Gv * (DR + 2), Gv);
        consumer_sync<CW>();  // red is reused by the next item
    }
}

template <int D, int GM, bool F8, int CW, int DR>
__global__ void __launch_bounds__(32 * (1 + CW), 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecodeAttentionProblem P, float scale_log2, int n_items, unsigned *err)
{
    static_assert(CW % kGroup == 0, "whole groups of four consumer warps");
    using L = DSmem<D, GM, F8, CW>;
    static_assert(L::ALLOC <= 232448, "shared memory per CTA");
    constexpr int ST = L::STAGES;
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
                    for (int c = 0; c < L::NCH; ++c) {  // 128-byte boxes: 64 bf16 values or 128 codes
                        const int x = c * (F8 ? 128 : 64);
                        tma_load_3d(smem + L::K + s * L::CB + c * L::BOX, &tmK, x, u0, z, full + s);
                        tma_load_3d(smem + L::V + s * L::CB + c * L::BOX, &tmV, x, u0, z, full + s);
                    }
                }
            }
            for (int j = max(0, it - ST); j < it; ++j) mbar_wait(full + j % ST, (j / ST) & 1, err);
        }
        return;  // the producer takes no part in the consumer barriers below
    }
    if constexpr (F8)
        consume_f8<D, CW, DR>(P, smem, full, empty, red, scale_log2, n_items, err);
    else if constexpr (GM == 8)
        consume_bf16_t<D, CW>(P, smem, full, empty, red, scale_log2, n_items, err);
    else
        consume_bf16<D, GM, CW>(P, smem, full, empty, red, scale_log2, n_items, err);
}

// One CTA per (b, head sub-group): merge the splits and write bf16 attn.  The
// splits' maxima and sums are read first (one round of independent loads),
// each head's weights 2^(m_s - M) / sum_s 2^(m_s - M) l_s formed once in
// shared memory, then every output element is one pass of independent loads
// over the splits (a per-element max-then-sum would chain two dependent
// memory reads per element).
constexpr int kCombineThreads = 256;
constexpr int kCombineMaxW = 16 * 256;  // weights: heads of a sub-group x splits

template <int D>
__global__ void __launch_bounds__(kCombineThreads) decode_combine_kernel(const DecodeAttentionProblem P)
{
    __shared__ float s_w[kCombineMaxW];  // [h][split]: m, then the normalised weight
    __shared__ float s_l[kCombineMaxW];  // [h][split]: l
    const int Gv = P.Hq / P.Hkv / P.vsub;
    const int REC = Gv * (D + 2);
    const int NS = P.splits;
    grid_dep_launch();
    grid_dep_wait();  // the split kernel's partial records
    const int bvg = blockIdx.x;
    const int nvg = P.Hkv * P.vsub;
    const int b = bvg / nvg, vg = bvg - b * nvg;
    const float *recs = P.partials + (size_t)bvg * NS * REC;
    for (int i = threadIdx.x; i < Gv * NS; i += kCombineThreads) {
        const int h = i / NS, s = i - h * NS;
        const float *r = recs + (size_t)s * REC + h * (D + 2);
        s_w[i] = r[D];
        s_l[i] = r[D + 1];
    }
    __syncthreads();
    for (int h = threadIdx.x; h < Gv; h += kCombineThreads) {
        float M = -INFINITY;
        for (int s = 0; s < NS; ++s) M = fmaxf(M, s_w[h * NS + s]);
        const float Mu = (M == -INFINITY) ? 0.0f : M;
        float L = 0.0f;
        for (int s = 0; s < NS; ++s) {
            const float w = ex2(s_w[h * NS + s] - Mu);
            s_w[h * NS + s] = w;
            L = fmaf(w, s_l[h * NS + s], L);
        }
        const float inv = L > 0.0f ? (P.fp8 ? P.v_scale : 1.0f) / L : 0.0f;
        for (int s = 0; s < NS; ++s) s_w[h * NS + s] *= inv;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < Gv * D; idx += kCombineThreads) {
        const int h = idx / D, c = idx - h * D;
        const float *r = recs + h * (D + 2) + c;
        float acc = 0.0f;
        for (int s = 0; s < NS; ++s) acc = fmaf(s_w[h * NS + s], r[(size_t)s * REC], acc);
        const __nv_bfloat16 ob = __float2bfloat16_rn(acc);
        P.out[(size_t)b * P.Hq * D + (size_t)(vg * Gv + h) * D + c] = *reinterpret_cast<const uint16_t *>(&ob);
    }
}

// D: the staged row width; DR: the head's real width (E4M3 rows narrower than
// 128 codes are staged 128 wide, the tensor copy filling codes past DR with
// zeros).
template <int D, int GM, bool F8, int CW = (F8 ? 12 : 4), int DR = D>
cudaError_t run_decode(const DecodeAttentionProblem &p0, unsigned *err, cudaStream_t stream)
{
    static_assert(F8 || DR == D, "bf16 caches are staged at their own width");
    using L = DSmem<D, GM, F8, CW>;
    DecodeAttentionProblem p = p0;
    p.vsub = decode_head_subgroups(p.Hq / p.Hkv, GM);
    // E4M3 keys are code * k_scale: the scale joins the softmax scale
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)DR) * (F8 ? p.k_scale : 1.0f);
    const int n_items = p.B * p.Hkv * p.vsub * p.splits;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // caches viewed as [B*Hkv, Lmax, D]; box {128 bytes, 64 keys, 1}, 128-byte swizzle
    CUtensorMap tk, tv;
    const int eb = F8 ? 1 : 2;
    const uint64_t dims[3] = {(uint64_t)DR, (uint64_t)p.Lmax, (uint64_t)p.B * p.Hkv};
    const uint64_t strides[2] = {(uint64_t)DR * eb, (uint64_t)p.Lmax * DR * eb};
    const uint32_t box[3] = {(uint32_t)(128 / eb), (uint32_t)kChunk, 1};
    if (encode_tmap(&tk, p.k_cache, 3, dims, strides, box, true, eb) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tv, p.v_cache, 3, dims, strides, box, true, eb) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = decode_split_kernel<D, GM, F8, CW, DR>;
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
    if ((size_t)(p.Hq / p.Hkv / p.vsub) * p.splits > (size_t)kCombineMaxW) return cudaErrorInvalidValue;
    LaunchCfg lc(dim3(p.B * p.Hkv * p.vsub), dim3(kCombineThreads), 0, stream, true);
    e = cudaLaunchKernelEx(&lc.cfg, decode_combine_kernel<DR>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int decode_head_subgroups(int G, int gm)
{
    // the fewest sub-groups of equal size that hold at most gm heads each
    for (int v = (G + gm - 1) / gm; v < G; ++v)
        if (G % v == 0) return v;
    return G;
}

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
    if (p.Hkv <= 0 || p.Hq % p.Hkv) return cudaErrorInvalidValue;
    const int G = p.Hq / p.Hkv;
    if (p.fp8) {
        // three groups of four consumer warps (the unpacking's latency; 185 -> 181 us against two groups on
        // the Qwen3-8B decode workload)
        if (p.d == 128) return run_decode<128, 8, true, 12>(p, err, stream);
        if (p.d == 64) return run_decode<128, 8, true, 12, 64>(p, err, stream);
        if (p.d == 80) return run_decode<128, 8, true, 12, 80>(p, err, stream);
        if (p.d == 96) return run_decode<128, 8, true, 12, 96>(p, err, stream);
        if (p.d == 256) return run_decode<256, 8, true, 4>(p, err, stream);  // one group: registers and partials
        return cudaErrorInvalidValue;
    }
    if (p.d == 128) return G <= 8 ? run_decode<128, 8, false>(p, err, stream) : run_decode<128, 16, false>(p, err, stream);
    if (p.d == 64) return G <= 8 ? run_decode<64, 8, false>(p, err, stream) : run_decode<64, 16, false>(p, err, stream);
    if (p.d == 80) return G <= 8 ? run_decode<80, 8, false>(p, err, stream) : run_decode<80, 16, false>(p, err, stream);
    if (p.d == 96) return G <= 8 ? run_decode<96, 8, false>(p, err, stream) : run_decode<96, 16, false>(p, err, stream);
    if (p.d == 256) return run_decode<256, 8, false>(p, err, stream);  // partials of 16 heads would not fit
    return cudaErrorInvalidValue;
}

}  // namespace gqa
