// gemm.cu -- persistent tcgen05 GEMM for the two projections of the layer.
//
//   QKV projection ([NeoX] "Fused QKV projection": hidden -> Hq*d + 2*Hkv*d)
//   with per-head RMSNorm of Q and K ([T07] §3 "QK-Norm") and RoPE on Q and K
//   ([T07] §4 step 3) fused into the epilogue, written head-major
//   ([T07] §4 step 4, (batch, heads, seq, head_dim)).
//
//   o_proj ([NeoX] "Output projection": Hq*d -> hidden) with the residual add
//   ([NeoX] "Qwen3-0.6B example", residual addition) fused into the epilogue.
//
// Structure (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: A/B k-slices into a STAGES-deep shared ring
//   warp 1      MMA issuer: tcgen05.mma 128 x BN x 16 into a TMEM accumulator;
//               two accumulators so tile i's epilogue overlaps tile i+1's loop
//   warps 2..5  epilogue: tcgen05.ld (one thread = one output row), fused
//               math, 32-byte global stores where the row address allows;
//               inputs it reads from memory (residual rows) are requested
//               into L2 before the accumulator is ready
//
// Problems with a single M block (the decode step's projections: 64 rows, a
// few dozen N tiles) would leave most SMs idle and stream the weights through
// few CTAs.  There the K dimension is split over a cluster of KS CTAs (one
// tile per cluster): each accumulates its K slice in its own TMEM, the others
// then write their partial sums into the first CTA's (now idle) operand ring
// through distributed shared memory, and the first CTA folds them into its
// accumulator and runs the epilogue unchanged.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int kThreads = 192;

enum { EPI_QKV = 0, EPI_RESIDUAL = 1, EPI_F32 = 2, EPI_HEAD16 = 3 };

// Operand storage: K-major (the contraction index contiguous: A [M, K], B
// [N, K]) or MN-major (the row / column index contiguous: A stored [K, M],
// B stored [K, N]).  MAJ bit 0: A is MN-major; bit 1: B is MN-major.  An
// MN-major tile sits in shared memory as 64-wide column chunks of BK rows
// (128-byte swizzle), the layout the tensor core reads with the operand's
// major bit set.
constexpr int kMnChunk = 64 * BK * 2;  // one 64-wide MN chunk of BK rows: 8 KB

struct GemmParams {
    int M, N, K;
    int num_m, num_n, num_k, num_tiles;
    int group_m;  // M-blocks per raster group
    unsigned *err;
    QkvEpilogue qkv;
    ResidualEpilogue res;
    float *f32_out;         // EPI_F32: C [M, N] fp32
    HeadEpilogue head;      // EPI_HEAD16
};

template <int BN, int STAGES>
struct Smem {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int RING = STAGES * (A_BYTES + B_BYTES);
    static constexpr int BARS = RING;                       // 2*STAGES + 5 mbarriers
    static constexpr int TMEM_SLOT = BARS + (2 * STAGES + 5) * 8;
    static constexpr int NORM = (TMEM_SLOT + 16 + 15) & ~15;  // q_norm_w, k_norm_w: 2 x 256 floats
    static constexpr int TOTAL = NORM + 2 * 256 * 4;
    static constexpr int ALLOC = TOTAL + 1024;               // slack for 1024-byte alignment
};

// Grouped rasterisation: walk GM M-blocks per N-block so that concurrently
// running CTAs share A rows and B rows in L2.  The A panels of a group stay in
// L2 while the group sweeps all N-blocks, and each B panel is read from DRAM
// once per group (GM = 32 for the QKV projection, 16 for o_proj, whose A
// panels are longer; both measured best at the Qwen3-32B shape).
DEVI void tile_coords(int tile, int num_m, int num_n, int GM, int &mb, int &nb)
{
    const int per_group = GM * num_n;
    const int grp = tile / per_group;
    const int first = grp * GM;
    const int gm = min(num_m - first, GM);
    const int local = tile - grp * per_group;
    mb = first + local % gm;
    nb = local / gm;
}

// W (2, 4, 8, 16 or 32) consecutive TMEM columns of this thread's lane, then wait.
template <int W>
DEVI void tmem_ldw(uint32_t taddr, uint32_t (&r)[W])
{
    if constexpr (W == 32) {
        tmem_ld32(taddr, r);
    } else if constexpr (W == 16) {
        tmem_ld16(taddr, r);
    } else if constexpr (W == 8) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
            : "r"(taddr)
            : "memory");
    } else if constexpr (W == 4) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
            : "r"(taddr)
            : "memory");
    } else {
        static_assert(W == 2, "TMEM load width");
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(r[0]), "=r"(r[1])
            : "r"(taddr)
            : "memory");
    }
}

// 32 bytes to global memory: one 256-bit store when p is 32-byte aligned
// (the epilogues write one row per thread, so every store is its own
// transaction and whole 32-byte sectors halve their count), else two
// 16-byte stores (the interface guarantees 16-byte alignment only).
DEVI void st_global32(void *p, const uint32_t (&w)[8])
{
    if (((uintptr_t)p & 31u) == 0) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else {
        uint4 *d4 = reinterpret_cast<uint4 *>(p);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

// W values of one row -> 16-bit storage (bf16, or binary16 clamped to its
// finite range; *clamped is set when a value had to be clamped).  dst is
// aligned to 2W bytes (16 at most).
template <int W>
DEVI void storew(uint16_t *dst, const float *v, bool f16, bool &clamped)
{
    uint32_t w[W / 2];
#pragma unroll
    for (int i = 0; i < W / 2; ++i) {
        float a = v[2 * i], b = v[2 * i + 1];
        if (f16) {
            const float ca = fminf(fmaxf(a, -kHalfMax), kHalfMax), cb = fminf(fmaxf(b, -kHalfMax), kHalfMax);
            clamped |= !(ca == a) || !(cb == b);
            w[i] = pack_f16(ca, cb);
        } else {
            w[i] = pack_bf16(a, b);
        }
    }
    if constexpr (W >= 16) {
#pragma unroll
        for (int i = 0; i < W / 16; ++i) {
            const uint32_t w8[8] = {w[8 * i], w[8 * i + 1], w[8 * i + 2], w[8 * i + 3],
                                    w[8 * i + 4], w[8 * i + 5], w[8 * i + 6], w[8 * i + 7]};
            st_global32(dst + 16 * i, w8);
        }
    } else if constexpr (W == 8) {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (W == 4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    } else {
        *reinterpret_cast<uint32_t *>(dst) = w[0];
    }
}

// Storage format of one projected head row: bf16, binary16 (clamped to its
// range and flagged), or E4M3 codes of value / scale (saturated and flagged).
struct OutFmt {
    int mode;     // 0 bf16, 1 binary16, 2 E4M3
    float scale;  // E4M3 only
};

// Columns [c, c + W) of a head row whose first element is at dst.
template <int W>
DEVI void putw(void *dst, int c, const float *v, OutFmt f, bool &clamped)
{
    if (f.mode != 2) {
        storew<W>(reinterpret_cast<uint16_t *>(dst) + c, v, f.mode == 1, clamped);
        return;
    }
    uint8_t *d8 = reinterpret_cast<uint8_t *>(dst) + c;
    if constexpr (W == 2) {
        const float q0 = __fdiv_rn(v[0], f.scale), q1 = __fdiv_rn(v[1], f.scale);
        clamped |= !(fabsf(q0) <= 448.0f) || !(fabsf(q1) <= 448.0f);
        *reinterpret_cast<uint16_t *>(d8) = (uint16_t)f32x2_to_e4m3x2(q0, q1);
        return;
    }
    constexpr int NW = W >= 4 ? W / 4 : 1;
    uint32_t w[NW];
#pragma unroll
    for (int i = 0; i < W / 4; ++i) {
        float q[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            q[k] = __fdiv_rn(v[4 * i + k], f.scale);
            clamped |= !(fabsf(q[k]) <= 448.0f);
        }
        w[i] = f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16);
    }
    if constexpr (W >= 16) {
#pragma unroll
        for (int i = 0; i < W / 16; ++i)
            reinterpret_cast<uint4 *>(d8)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    } else if constexpr (W == 8) {
        *reinterpret_cast<uint2 *>(d8) = make_uint2(w[0], w[1]);
    } else {
        *reinterpret_cast<uint32_t *>(d8) = w[0];
    }
}

// Widest TMEM chunk (<= 32 columns) that tiles n (even) columns.
__host__ __device__ constexpr int chunk_width(int n)
{
    return n % 32 == 0 ? 32 : n % 16 == 0 ? 16 : n % 8 == 0 ? 8 : n % 4 == 0 ? 4 : 2;
}

// Normalised (x * rinv * w) head row of a Q or K head, rotated on its first
// RD features (rotate-half pairs (i, i + RD/2), (cos, sin) of angle
// pos * theta^(-2i/RD) from cs[i * ld], the pair-major table at this row's
// position: the 32 rows of a warp are consecutive positions of one sequence in
// a prefill, so each of these loads is one coalesced read) and stored; features [RD, D) are only
// normalised.  The pairs are taken in chunks of W columns and the rest in
// chunks of CW, the widest that tile RD/2 and D - RD, so that every TMEM load
// starts at a multiple of its own width (head offsets are multiples of D).
template <int D, int RD>
DEVI void rope_store(uint32_t col, void *dst, float rinv, bool has_norm, const float *w, const float2 *cs,
                     int ld, bool row_ok, OutFmt fmt, bool &clamped)
{
    auto nrm = [&](float x, int c) { return has_norm ? x * rinv * w[c] : x * rinv; };
    if constexpr (RD > 0) {
        constexpr int H = RD / 2, W = chunk_width(H);
#pragma unroll 1
        for (int c = 0; c < H; c += W) {
            uint32_t r1[W], r2[W];
            tmem_ldw<W>(col + c, r1);
            tmem_ldw<W>(col + c + H, r2);
            float y1[W], y2[W];
            float2 t[W];
#pragma unroll
            for (int i = 0; i < W; ++i) t[i] = __ldg(cs + (size_t)(c + i) * ld);  // (cos, sin)
#pragma unroll
            for (int i = 0; i < W; ++i) {
                const float x1 = nrm(__uint_as_float(r1[i]), c + i);
                const float x2 = nrm(__uint_as_float(r2[i]), c + i + H);
                y1[i] = x1 * t[i].x - x2 * t[i].y;
                y2[i] = x2 * t[i].x + x1 * t[i].y;
            }
            if (row_ok) {
                putw<W>(dst, c, y1, fmt, clamped);
                putw<W>(dst, c + H, y2, fmt, clamped);
            }
        }
    }
    if constexpr (RD < D) {
        constexpr int CW = chunk_width(D - RD);
#pragma unroll 1
        for (int c = RD; c < D; c += CW) {  // features past the rotary width
            uint32_t r[CW];
            tmem_ldw<CW>(col + c, r);
            float y[CW];
#pragma unroll
            for (int i = 0; i < CW; ++i) y[i] = nrm(__uint_as_float(r[i]), c + i);
            if (row_ok) putw<CW>(dst, c, y, fmt, clamped);
        }
    }
}

// fp32 C rows (N a multiple of 8).
template <int BN>
DEVI void epilogue_f32(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok)
{
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int n = n0 + c;
        if (n >= P.N) break;  // uniform across the warp
        uint32_t r[32];
        tmem_ld32(tcol + c, r);
        if (!row_ok) continue;
        float4 *dst = reinterpret_cast<float4 *>(P.f32_out + (size_t)m * P.N + n);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            if (n + 4 * v >= P.N) break;
            dst[v] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                 __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
        }
    }
}

// binary16 head-major output: column n = j*d + c of row m = b*S + t goes to
// out[((b*H + j)*S + t)*d + c] (clamped to binary16's range and flagged).
// Stored 16 columns at a time: d is a multiple of 16 (64, 80, 96, 128), so a
// 16-column piece never crosses a head, while a 32-column one would at d = 80.
template <int BN>
DEVI void epilogue_head16(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok)
{
    const HeadEpilogue &e = P.head;
    const int b = m / e.S, t = m - (m / e.S) * e.S;
    bool clamped = false;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int n = n0 + c;
        if (n >= P.N) break;
        uint32_t r[32];
        tmem_ld32(tcol + c, r);
        if (!row_ok) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nh = n + 16 * h;
            if (nh >= P.N) break;
            const int j = nh / e.d, cc = nh - j * e.d;
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[16 * h + i]);
            storew<16>(e.out + ((size_t)(b * e.H + j) * e.S + t) * e.d + cc, v, true, clamped);
        }
    }
    if (clamped) atomicOr(P.err, kErrRange);
}

// Epilogue of one QKV tile row: BN columns = BN/D whole heads.
template <int BN, int D>
DEVI void epilogue_qkv(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok, const float *s_norm)
{
    static_assert(BN % D == 0, "a tile holds whole heads");
    constexpr int CWD = chunk_width(D);  // TMEM chunk that tiles a head row (32, or 16 for d = 80)
    const QkvEpilogue &e = P.qkv;
    const int HqD = e.Hq * D, HkvD = e.Hkv * D;
    int b = 0, pos = 0, q_slot = 0, kv_slot = 0;
    if (row_ok) {
        if (e.pos_dev) {  // new tokens after pos_dev[b] cached ones: position = slot = pos_dev[b] + t
            b = m / e.S;
            q_slot = m - b * e.S;
            pos = e.pos_dev[b] + q_slot;
            kv_slot = pos;
        } else {
            const int mg = e.m0 + m;  // row of the whole problem
            b = mg / e.S;
            pos = mg - b * e.S;
            q_slot = kv_slot = pos;
        }
        if (pos < 0 || pos >= e.rope_rows || kv_slot >= e.kv_seq) {
            atomicOr(P.err, kErrIndex);
            row_ok = false;
        }
    }
    const bool has_norm = e.q_norm_w != nullptr;
    bool clamped = false;
#pragma unroll 1
    for (int h = 0; h < BN / D; ++h) {
        const int n = n0 + h * D;
        if (n >= P.N) break;  // uniform across the warp
        const uint32_t col = tcol + h * D;
        int kind, head;
        if (n < HqD) {
            kind = 0;
            head = n / D;
        } else if (n < HqD + HkvD) {
            kind = 1;
            head = (n - HqD) / D;
        } else {
            kind = 2;
            head = (n - HqD - HkvD) / D;
        }
        // element offset of the head row; K/V rows hold 1-byte codes when kv_fp8
        void *dst;
        OutFmt fmt;
        if (kind == 0) {
            dst = e.q_out + ((size_t)(b * e.Hq + head) * e.q_seq + q_slot) * D;
            fmt = {e.q_f16 ? 1 : 0, 1.0f};
        } else {
            const size_t off = ((size_t)(b * e.Hkv + head) * e.kv_seq + kv_slot) * D;
            uint16_t *base = kind == 1 ? e.k_out : e.v_out;
            if (e.kv_fp8) {
                dst = reinterpret_cast<uint8_t *>(base) + off;
                fmt = {2, kind == 1 ? e.k_scale : e.v_scale};
            } else {
                dst = base + off;
                fmt = {e.kv_f16 ? 1 : 0, 1.0f};
            }
        }

        if (kind == 2) {  // V: no norm, no rotation
#pragma unroll 1
            for (int c = 0; c < D; c += CWD) {
                uint32_t r[CWD];
                tmem_ldw<CWD>(col + c, r);
                float v[CWD];
#pragma unroll
                for (int i = 0; i < CWD; ++i) v[i] = __uint_as_float(r[i]);
                if (row_ok) putw<CWD>(dst, c, v, fmt, clamped);
            }
            continue;
        }
        float rinv = 1.0f;
        if (has_norm) {
            float ss = 0.0f;
            // pre-norm Q/K rows for the backward's RMSNorm gradient: [M, (Hq+Hkv)*D] fp32
            float *pre = e.pre_out ? e.pre_out + (size_t)m * (e.Hq + e.Hkv) * D + (kind == 0 ? head : e.Hq + head) * D
                                   : nullptr;
#pragma unroll 1
            for (int c = 0; c < D; c += CWD) {
                uint32_t r[CWD];
                tmem_ldw<CWD>(col + c, r);
#pragma unroll
                for (int i = 0; i < CWD; ++i) {
                    const float f = __uint_as_float(r[i]);
                    ss = fmaf(f, f, ss);
                }
                if (pre && row_ok) {
                    float4 *d4 = reinterpret_cast<float4 *>(pre + c);
#pragma unroll
                    for (int i = 0; i < CWD / 4; ++i)
                        d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                }
            }
            rinv = 1.0f / sqrtf(ss * (1.0f / D) + e.eps);
        }
        const float *w = s_norm + (kind == 0 ? 0 : 256);
        const int p = row_ok ? pos : 0;
        const float2 *cs = e.rope ? e.rope + p : nullptr;  // pair 0 at this position
        if (e.rd == D)
            rope_store<D, D>(col, dst, rinv, has_norm, w, cs, e.rope_ld, row_ok, fmt, clamped);
        else if (e.rd == D / 2)
            rope_store<D, D / 2>(col, dst, rinv, has_norm, w, cs, e.rope_ld, row_ok, fmt, clamped);
        else if (e.rd == D / 4)
            rope_store<D, D / 4>(col, dst, rinv, has_norm, w, cs, e.rope_ld, row_ok, fmt, clamped);
        else
            rope_store<D, 0>(col, dst, rinv, has_norm, w, nullptr, 0, row_ok, fmt, clamped);
    }
    if (clamped) atomicOr(P.err, kErrRange);
}

template <int BN>
DEVI void epilogue_residual(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok)
{
    const ResidualEpilogue &e = P.res;
    // the residual of the next 32 columns is loaded while this chunk is added
    auto load = [&](int c, uint4 (&x)[4]) {
        const int n = n0 + c;
        const uint4 *src = reinterpret_cast<const uint4 *>(e.resid + (size_t)m * P.N + n);
#pragma unroll
        for (int v = 0; v < 4; ++v) x[v] = (row_ok && n + 8 * v < P.N) ? src[v] : make_uint4(0, 0, 0, 0);
    };
    uint4 cur[4], nxt[4];
    load(0, cur);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
        const int n = n0 + c;
        if (n >= P.N) break;  // uniform across the warp
        if (c + 32 < BN && n + 32 < P.N) load(c + 32, nxt);
        uint32_t r[32];
        tmem_ld32(tcol + c, r);
        if (row_ok) {
            uint16_t *dst = e.out + (size_t)m * P.N + n;
            uint32_t o[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const uint32_t xs[4] = {cur[v].x, cur[v].y, cur[v].z, cur[v].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o[4 * v + k] = pack_bf16(__uint_as_float(r[8 * v + 2 * k]) + bf16lo(xs[k]),
                                             __uint_as_float(r[8 * v + 2 * k + 1]) + bf16hi(xs[k]));
            }
            if (n + 32 <= P.N) {  // the whole chunk: two 32-byte stores
                const uint32_t a[8] = {o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]};
                const uint32_t b[8] = {o[8], o[9], o[10], o[11], o[12], o[13], o[14], o[15]};
                st_global32(dst, a);
                st_global32(dst + 16, b);
            } else {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    if (n + 8 * v < P.N) d4[v] = make_uint4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
            }
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) cur[v] = nxt[v];
    }
}

// Before a tile's accumulator is ready, the residual rows its epilogue adds are
// requested into L2 (one bulk prefetch per row segment), so the epilogue does
// not wait on DRAM once per chunk; short-K problems are otherwise bound by it.
// (The same for the RoPE table rows of the QKV epilogue measured slower.)
DEVI void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int BN, int EPI, int D>
DEVI void epilogue_prefetch(const GemmParams &P, int m, int n0, bool row_ok)
{
    if (!row_ok) return;
    if constexpr (EPI == EPI_RESIDUAL) {
        const int cols = min(BN, P.N - n0);  // a multiple of 8: whole 16-byte units
        if (cols > 0) prefetch_l2(P.res.resid + (size_t)m * P.N + n0, (uint32_t)cols * 2);
    }
}

// The tile's epilogue, one thread per accumulator row.
template <int BN, int EPI, int D>
DEVI void epilogue_tile(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok, const float *s_norm)
{
    if constexpr (EPI == EPI_QKV)
        epilogue_qkv<BN, D>(P, tcol, m, n0, row_ok, s_norm);
    else if constexpr (EPI == EPI_RESIDUAL)
        epilogue_residual<BN>(P, tcol, m, n0, row_ok);
    else if constexpr (EPI == EPI_F32)
        epilogue_f32<BN>(P, tcol, m, n0, row_ok);
    else
        epilogue_head16<BN>(P, tcol, m, n0, row_ok);
}

// KS: CTAs of a cluster that split K for one tile (1: no split, persistent
// over tiles).
template <int BN, int STAGES, int EPI, int D, int MAJ, int KS>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const GemmParams P)
{
    constexpr bool AMN = MAJ & 1, BMN = (MAJ >> 1) & 1;
    static_assert(KS >= 1 && KS <= 4, "K split");
    // split-K partial sums of one CTA: BM rows of BN fp32, rows padded by 16
    // bytes so a warp's 16-byte accesses to 32 rows spread over all banks
    constexpr int PART_LD = BN + 4;
    constexpr int PART = BM * PART_LD * 4;
    // TMEM columns per accumulator: BN rounded up to a power of two (the
    // allocation unit), so both accumulators start on aligned columns
    constexpr int ACC = BN <= 64 ? 64 : BN <= 128 ? 128 : 256;
    static_assert(BN <= ACC && BN % 16 == 0, "MMA N");
    using L = Smem<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * L::A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::BARS);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::TMEM_SLOT);
    float *s_norm = reinterpret_cast<float *>(smem + L::NORM);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;
    grid_dep_launch();  // the next kernel may start its prologue meanwhile
    // tiles this CTA walks, and its K blocks [kb0, kb1) of each
    const uint32_t crank = KS > 1 ? cluster_rank() : 0;
    const int tile0 = KS > 1 ? (int)(blockIdx.x / KS) : (int)blockIdx.x;
    const int tile_step = KS > 1 ? P.num_tiles : (int)gridDim.x;  // split K: one tile per cluster
    const int kb0 = (int)(crank * P.num_k / KS), kb1 = (int)((crank + 1) * P.num_k / KS);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 4);
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    bool acc_ready = false;  // split K: this warp's accumulator rows are complete
    if (warp == 1) tmem_alloc(tmem_slot, 2 * ACC);
    if (EPI == EPI_QKV && warp >= 2 && P.qkv.q_norm_w) {
        for (int i = threadIdx.x - 64; i < D; i += 128) {
            s_norm[i] = __uint_as_float((uint32_t)P.qkv.q_norm_w[i] << 16);
            s_norm[256 + i] = __uint_as_float((uint32_t)P.qkv.k_norm_w[i] << 16);
        }
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            auto load_a = [&](int s, int mb, int kb) {
                if constexpr (AMN) {
                    for (int c = 0; c < BM / 64; ++c)
                        tma_load_2d(sA + s * L::A_BYTES + c * kMnChunk, &tmA, mb * BM + c * 64, kb * BK, full + s);
                } else {
                    tma_load_2d(sA + s * L::A_BYTES, &tmA, kb * BK, mb * BM, full + s);
                }
            };
            auto load_b = [&](int s, int nb, int kb) {
                if constexpr (BMN) {
                    for (int c = 0; c < BN / 64; ++c)
                        tma_load_2d(sB + s * L::B_BYTES + c * kMnChunk, &tmB, nb * BN + c * 64, kb * BK, full + s);
                } else {
                    tma_load_2d(sB + s * L::B_BYTES, &tmB, kb * BK, nb * BN, full + s);
                }
            };
            // B (the weight matrix wherever this kernel follows another one as a
            // programmatic dependent) does not come from the previous kernel: the
            // first ring fill's B tiles go out before waiting for that kernel
            int pre = 0;
            if (tile0 < P.num_tiles) {
                int mb, nb;
                tile_coords(tile0, P.num_m, P.num_n, P.group_m, mb, nb);
                for (int kb = kb0; kb < kb1 && pre < STAGES; ++kb, ++pre) {
                    mbar_arrive_expect_tx(full + pre, L::A_BYTES + L::B_BYTES);
                    load_b(pre, nb, kb);
                }
            }
            grid_dep_wait();
            int it = 0;
            bool ok = true;
            for (int tile = tile0; ok && tile < P.num_tiles; tile += tile_step) {
                int mb, nb;
                tile_coords(tile, P.num_m, P.num_n, P.group_m, mb, nb);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (it >= pre) {
                        const uint32_t ph = (it / STAGES) & 1;
                        if (!mbar_wait(empty + s, ph ^ 1, err)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full + s, L::A_BYTES + L::B_BYTES);
                        load_b(s, nb, kb);
                    }
                    load_a(s, mb, kb);
                }
            }
            // every issued copy has landed before the CTA may exit
            for (int j = max(0, it - STAGES); j < it; ++j) mbar_wait(full + j % STAGES, (j / STAGES) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, AMN ? 1 : 0, BMN ? 1 : 0);
            int it = 0, use = 0;
            bool ok = true;
            for (int tile = tile0; ok && tile < P.num_tiles; tile += tile_step, ++use) {
                const int acc = use & 1;
                if (!mbar_wait(tempty + acc, ((use >> 1) & 1) ^ 1, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * ACC;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait(full + s, (it / STAGES) & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + s * L::A_BYTES);
                    const uint32_t b0 = smem_u32(sB + s * L::B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // K-major: the next 16 K values are 32 bytes along the row; MN-major:
                        // the next 16 K rows are 2 KB down each 64-wide chunk
                        const uint64_t ad = AMN ? sw128_desc(a0 + k * 16 * 128, kMnChunk, 1024)
                                                : sw128_desc(a0 + 32 * k, 16, 1024);
                        const uint64_t bd = BMN ? sw128_desc(b0 + k * 16 * 128, kMnChunk, 1024)
                                                : sw128_desc(b0 + 32 * k, 16, 1024);
                        umma_f16_ss(d_tmem, ad, bd, idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                    }
                    umma_commit(empty + s);  // frees the stage once these MMAs have read it
                }
                if (!ok) break;
                umma_commit(tfull + acc);  // accumulator ready for the epilogue
            }
            umma_commit(drain);
            mbar_wait(drain, 0, err);
        }
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;
        grid_dep_wait();  // the epilogue reads and writes what the previous kernel may touch
        int use = 0;
        for (int tile = tile0; tile < P.num_tiles; tile += tile_step, ++use) {
            int mb, nb;
            tile_coords(tile, P.num_m, P.num_n, P.group_m, mb, nb);
            const int acc = use & 1;
            epilogue_prefetch<BN, EPI, D>(P, mb * BM + row, nb * BN, mb * BM + row < P.M);
            const bool ready = mbar_wait(tfull + acc, (use >> 1) & 1, err);
            if constexpr (KS > 1) {  // the cluster sums the partials below
                acc_ready = __all_sync(0xffffffffu, ready);
                break;
            }
            if (!ready) break;
            tc_fence_after();
            const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16) + acc * ACC;
            const int m = mb * BM + row;
            epilogue_tile<BN, EPI, D>(P, tcol, m, nb * BN, m < P.M, s_norm);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_relaxed(tempty + acc);
        }
    }
    if constexpr (KS > 1) {
        // Every CTA of the cluster has its K slice in TMEM accumulator 0 (or
        // gave up on a bounded wait, recorded in *err) and the first CTA's
        // operand ring is idle: the others add their partials into it.
        static_assert((KS - 1) * PART <= L::RING, "split-K partials fit in the operand ring");
        __syncthreads();
        cluster_sync();
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16);
        int mb = 0, nb = 0;
        if (tile0 < P.num_tiles) tile_coords(tile0, P.num_m, P.num_n, P.group_m, mb, nb);
        const int m = mb * BM + row;
        const bool active = warp >= 2 && tile0 < P.num_tiles && acc_ready;  // warp-uniform
        if (active && crank != 0) {
            tc_fence_after();
            const uint32_t dst = cluster_map(smem_u32(smem), 0) + (uint32_t)(((crank - 1) * BM + row) * PART_LD * 4);
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t r[16];
                tmem_ld16(tcol + c, r);
                if (m < P.M)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_cluster_v4(dst + (c + 4 * i) * 4, r[4 * i], r[4 * i + 1], r[4 * i + 2], r[4 * i + 3]);
            }
        }
        cluster_sync();
        if (active && crank == 0) {
            tc_fence_after();
            // every lane loads and stores (the TMEM accesses are warp-collective);
            // only rows of the problem add partials
            const float *part = reinterpret_cast<const float *>(smem) + row * PART_LD;
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t r[16];
                tmem_ld16(tcol + c, r);
                if (m < P.M) {
#pragma unroll
                    for (int k = 1; k < KS; ++k) {
                        const float4 *p4 = reinterpret_cast<const float4 *>(part + (k - 1) * BM * PART_LD + c);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float4 q = p4[i];
                            r[4 * i] = __float_as_uint(__uint_as_float(r[4 * i]) + q.x);
                            r[4 * i + 1] = __float_as_uint(__uint_as_float(r[4 * i + 1]) + q.y);
                            r[4 * i + 2] = __float_as_uint(__uint_as_float(r[4 * i + 2]) + q.z);
                            r[4 * i + 3] = __float_as_uint(__uint_as_float(r[4 * i + 3]) + q.w);
                        }
                    }
                }
                tmem_st16_nowait(tcol + c, r);
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            tc_fence_after();
            epilogue_tile<BN, EPI, D>(P, tcol, m, nb * BN, m < P.M, s_norm);
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * ACC);
    }
}

// Two-SM form for problems with many 256 x 256 output tiles (the prefill
// projections).  A 2-CTA cluster computes one 256 x 256 tile with MMAs of
// M = 256 over the CTA pair: each CTA stages its own 128 rows of A and its
// own half (128 rows) of B, so per MMA each SM's tensor core reads 8 KB of
// shared memory instead of 12 KB and each SM's copies bring 32 KB per K step
// instead of 48 KB -- the single-SM 128 x 256 tile is bound by that traffic
// -- and the lighter stages allow a 6-deep ring.  Each CTA's TMEM holds its
// 128 accumulator rows, and its epilogue warps run the unchanged epilogue on
// them.
//   warp 0 (both CTAs)   TMA: A and B-half k-slices into the local ring; the
//                        copies' byte counts complete on the even CTA's
//                        `full` barrier, which only the even CTA arms
//   warp 1 (even CTA)    MMA issue; each commit arrives on the barrier of
//                        that offset in both CTAs (stage free, accumulator
//                        full)
//   warps 2..5 (both)    epilogue; the accumulator is released by arriving
//                        on the even CTA's `tempty` (8 arrivals: both CTAs)
template <int STAGES, int EPI, int D>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams P)
{
    constexpr int BN = 256, BNH = 128;  // N of the pair's MMA; B rows staged by each CTA
    constexpr int A_BYTES = BM * BK * 2, B_BYTES = BNH * BK * 2;
    constexpr int ACC = 256;            // TMEM columns per accumulator
    constexpr int RING = STAGES * (A_BYTES + B_BYTES);
    constexpr int BARS = RING;
    constexpr int TMEM_SLOT = BARS + (2 * STAGES + 5) * 8;
    constexpr int NORM = (TMEM_SLOT + 16 + 15) & ~15;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + BARS);
    uint64_t *empty = full + STAGES;
    uint64_t *tfull = empty + STAGES;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + TMEM_SLOT);
    float *s_norm = reinterpret_cast<float *>(smem + NORM);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    unsigned *err = P.err;
    grid_dep_launch();  // the next kernel may start its prologue meanwhile
    const uint32_t rank = cluster_rank();  // 0: the CTA that issues the MMAs
    const int tile0 = (int)(blockIdx.x / 2), tile_step = (int)(gridDim.x / 2);
    const int kb0 = 0, kb1 = P.num_k;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full + s, 1);   // armed by the even CTA's producer (both CTAs' bytes)
            mbar_init(empty + s, 1);  // one multicast commit per fill
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 8);  // the epilogue warps of both CTAs
        }
        mbar_init(drain, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, 2 * ACC);
    if (EPI == EPI_QKV && warp >= 2 && P.qkv.q_norm_w) {
        for (int i = threadIdx.x - 64; i < D; i += 128) {
            s_norm[i] = __uint_as_float((uint32_t)P.qkv.q_norm_w[i] << 16);
            s_norm[256 + i] = __uint_as_float((uint32_t)P.qkv.k_norm_w[i] << 16);
        }
    }
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised before any copy or arrival reaches them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t full_lead = cluster_map(smem_u32(full), 0);      // the even CTA's full[0]
    const uint32_t tempty_lead = cluster_map(smem_u32(tempty), 0);  // the even CTA's tempty[0]

    if (warp == 0) {
        if (lane == 0) {
            auto load_a = [&](int s, int mb, int kb) {
                tma_load_2d_pair(sA + s * A_BYTES, &tmA, kb * BK, mb * 2 * BM + (int)rank * BM, full_lead + 8 * s);
            };
            auto load_b = [&](int s, int nb, int kb) {
                tma_load_2d_pair(sB + s * B_BYTES, &tmB, kb * BK, nb * BN + (int)rank * BNH, full_lead + 8 * s);
            };
            auto arm = [&](int s) {
                if (rank == 0) mbar_arrive_expect_tx(full + s, 2 * (A_BYTES + B_BYTES));
            };
            // the weights (B) do not come from the previous kernel: the first ring
            // fill's B tiles go out before waiting for it
            int pre = 0;
            if (tile0 < P.num_tiles) {
                int mb, nb;
                tile_coords(tile0, P.num_m, P.num_n, P.group_m, mb, nb);
                for (int kb = kb0; kb < kb1 && pre < STAGES; ++kb, ++pre) {
                    arm(pre);
                    load_b(pre, nb, kb);
                }
            }
            grid_dep_wait();
            int it = 0;
            bool ok = true;
            for (int tile = tile0; ok && tile < P.num_tiles; tile += tile_step) {
                int mb, nb;
                tile_coords(tile, P.num_m, P.num_n, P.group_m, mb, nb);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (it >= pre) {
                        const uint32_t ph = (it / STAGES) & 1;
                        if (!mbar_wait(empty + s, ph ^ 1, err)) {
                            ok = false;
                            break;
                        }
                        arm(s);
                        load_b(s, nb, kb);
                    }
                    load_a(s, mb, kb);
                }
            }
            // every fill has been consumed (so every copy has landed) before the CTA may exit
            for (int j = max(0, it - STAGES); j < it; ++j) mbar_wait(empty + j % STAGES, (j / STAGES) & 1, err);
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(2 * BM, BN, 0, 0);
            int it = 0, use = 0;
            bool ok = true;
            for (int tile = tile0; ok && tile < P.num_tiles; tile += tile_step, ++use) {
                const int acc = use & 1;
                if (!mbar_wait<true>(tempty + acc, ((use >> 1) & 1) ^ 1, err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + acc * ACC;
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    if (!mbar_wait<true>(full + s, (it / STAGES) & 1, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + s * A_BYTES);
                    const uint32_t b0 = smem_u32(sB + s * B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        umma_f16_ss_pair(d_tmem, sw128_desc(a0 + 32 * k, 16, 1024), sw128_desc(b0 + 32 * k, 16, 1024),
                                         idesc, (kb != kb0 || k != 0) ? 1u : 0u);
                    umma_commit_pair(empty + s, 0x3);  // frees stage s in both CTAs
                }
                if (!ok) break;
                umma_commit_pair(tfull + acc, 0x3);  // both CTAs' accumulator rows ready
            }
            umma_commit_pair(drain, 0x1);
            mbar_wait(drain, 0, err);
        }
    } else {
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row = quarter * 32 + lane;
        grid_dep_wait();  // the epilogue reads and writes what the previous kernel may touch
        int use = 0;
        for (int tile = tile0; tile < P.num_tiles; tile += tile_step, ++use) {
            int mb, nb;
            tile_coords(tile, P.num_m, P.num_n, P.group_m, mb, nb);
            const int acc = use & 1;
            const int m = mb * 2 * BM + (int)rank * BM + row;
            epilogue_prefetch<BN, EPI, D>(P, m, nb * BN, m < P.M);
            if (!mbar_wait<true>(tfull + acc, (use >> 1) & 1, err)) break;
            tc_fence_after();
            const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16) + acc * ACC;
            epilogue_tile<BN, EPI, D>(P, tcol, m, nb * BN, m < P.M, s_norm);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_lead + 8 * acc);
        }
    }
    __syncthreads();
    cluster_sync();  // no CTA of the pair leaves while the other may still use its TMEM or barriers
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 2 * ACC);
    }
}

template <int BN, int STAGES, int EPI, int D, int MAJ = 0, int KS = 1>
cudaError_t run(const GemmProblem &p, const GemmParams &params, int num_sms, cudaStream_t stream)
{
    using L = Smem<BN, STAGES>;
    constexpr bool AMN = MAJ & 1, BMN = (MAJ >> 1) & 1;
    CUtensorMap ta, tb;
    // K-major A [M, K]: box {BK, BM}; MN-major A stored [K, M]: box {64, BK} per 64-wide chunk
    const uint64_t dA[2] = {AMN ? (uint64_t)p.M : (uint64_t)p.K, AMN ? (uint64_t)p.K : (uint64_t)p.M};
    const uint64_t sA[1] = {(AMN ? (uint64_t)p.M : (uint64_t)p.K) * 2};
    const uint64_t dB[2] = {BMN ? (uint64_t)p.N : (uint64_t)p.K, BMN ? (uint64_t)p.K : (uint64_t)p.N};
    const uint64_t sB[1] = {(BMN ? (uint64_t)p.N : (uint64_t)p.K) * 2};
    const uint32_t bA[2] = {AMN ? 64u : (uint32_t)BK, AMN ? (uint32_t)BK : (uint32_t)BM};
    const uint32_t bB[2] = {BMN ? 64u : (uint32_t)BK, BMN ? (uint32_t)BK : (uint32_t)BN};
    if (encode_tmap(&ta, p.A, 2, dA, sA, bA, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tb, p.B, 2, dB, sB, bB, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    auto kern = gemm_kernel<BN, STAGES, EPI, D, MAJ, KS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    // split K: one tile per cluster of KS CTAs; otherwise persistent, one CTA per SM at most
    const int grid = KS > 1 ? params.num_tiles * KS : (params.num_tiles < num_sms ? params.num_tiles : num_sms);
    LaunchCfg lc(dim3(grid), dim3(kThreads), L::ALLOC, stream, p.pdl != 0, KS);
    e = cudaLaunchKernelEx(&lc.cfg, kern, ta, tb, params);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// How many CTAs of this kernel's clusters of KS can be resident at once
// (0 if the query fails); cached per kernel.
template <int BN, int STAGES, int EPI, int D, int KS>
int cluster_capacity()
{
    static int cap = -1;
    if (cap >= 0) return cap;
    using L = Smem<BN, STAGES>;
    auto kern = gemm_kernel<BN, STAGES, EPI, D, 0, KS>;
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(KS);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = L::ALLOC;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = KS;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
    }
    (void)cudaGetLastError();
    cap = n * KS;
    return cap;
}

// A single-M-block problem with few tiles: split K over a cluster of 3 or 2
// CTAs when every cluster fits on the GPU at once and each CTA keeps at least
// four K blocks; otherwise no split.
template <int BN, int STAGES, int EPI, int D>
cudaError_t run_small_m(const GemmProblem &p, const GemmParams &g, int num_sms, cudaStream_t stream)
{
    if (g.num_m == 1) {
        if (g.num_tiles * 3 <= num_sms && g.num_k >= 12 && g.num_tiles * 3 <= cluster_capacity<BN, STAGES, EPI, D, 3>())
            return run<BN, STAGES, EPI, D, 0, 3>(p, g, num_sms, stream);
        if (g.num_tiles * 2 <= num_sms && g.num_k >= 8 && g.num_tiles * 2 <= cluster_capacity<BN, STAGES, EPI, D, 2>())
            return run<BN, STAGES, EPI, D, 0, 2>(p, g, num_sms, stream);
    }
    return run<BN, STAGES, EPI, D>(p, g, num_sms, stream);
}

GemmParams make_params(const GemmProblem &p, int BN, unsigned *err)
{
    GemmParams g{};
    g.M = p.M;
    g.N = p.N;
    g.K = p.K;
    g.num_m = (p.M + BM - 1) / BM;
    g.num_n = (p.N + BN - 1) / BN;
    g.num_k = (p.K + BK - 1) / BK;
    g.num_tiles = g.num_m * g.num_n;
    g.err = err;
    g.group_m = 32;
    return g;
}

// The pair kernel over 256 x 256 tiles (tile rows of 256 = two CTAs' 128), as
// many 2-CTA clusters as fit on the GPU at once; returns cudaErrorNotSupported
// when the cluster shape cannot be placed (the caller then runs the single-SM
// kernel).
template <int STAGES, int EPI, int D>
cudaError_t run_pair(const GemmProblem &p, GemmParams params, int group_m, cudaStream_t stream)
{
    constexpr int SMEM = STAGES * (BM * BK * 2 + 128 * BK * 2) + (2 * STAGES + 5) * 8 + 32 + 2 * 256 * 4 + 1024;
    CUtensorMap ta, tb;
    const uint64_t dA[2] = {(uint64_t)p.K, (uint64_t)p.M};
    const uint64_t sA[1] = {(uint64_t)p.K * 2};
    const uint64_t dB[2] = {(uint64_t)p.K, (uint64_t)p.N};
    const uint64_t sB[1] = {(uint64_t)p.K * 2};
    const uint32_t bA[2] = {(uint32_t)BK, (uint32_t)BM};
    const uint32_t bB[2] = {(uint32_t)BK, 128u};
    if (encode_tmap(&ta, p.A, 2, dA, sA, bA, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tb, p.B, 2, dB, sB, bB, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    params.num_m = (p.M + 2 * BM - 1) / (2 * BM);  // pair-tile rows
    params.num_n = (p.N + 255) / 256;
    params.num_tiles = params.num_m * params.num_n;
    params.group_m = group_m;
    if (!cta_pairs_enabled()) return cudaErrorNotSupported;
    auto kern = gemm_pair_kernel<STAGES, EPI, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    int clusters = 0;
    {
        LaunchCfg probe(dim3(2), dim3(kThreads), SMEM, stream, false, 2);
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &probe.cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            return cudaErrorNotSupported;
        }
    }
    const int n = params.num_tiles < clusters ? params.num_tiles : clusters;
    LaunchCfg lc(dim3(2 * n), dim3(kThreads), SMEM, stream, p.pdl != 0, 2);
    e = cudaLaunchKernelEx(&lc.cfg, kern, ta, tb, params);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_qkv(const GemmProblem &p, const QkvEpilogue &e, unsigned *err, int num_sms,
                            cudaStream_t stream)
{
    // Decode-sized problems (one M block) use narrower tiles so more SMs
    // stream the weight matrix.
    const bool small_m = p.M <= BM;
    if (e.d == 128) {
        if (small_m) {
            GemmParams g = make_params(p, 128, err);
            g.qkv = e;
            return run_small_m<128, 6, EPI_QKV, 128>(p, g, num_sms, stream);
        }
        GemmParams g = make_params(p, 256, err);
        g.qkv = e;
        const cudaError_t pe = run_pair<6, EPI_QKV, 128>(p, g, 16, stream);
        if (pe != cudaErrorNotSupported) return pe;
        return run<256, 4, EPI_QKV, 128>(p, g, num_sms, stream);
    }
    if (e.d == 256) {  // one 256-wide head per tile, also for decode-sized problems
        GemmParams g = make_params(p, 256, err);
        g.qkv = e;
        return run<256, 4, EPI_QKV, 256>(p, g, num_sms, stream);
    }
    if (e.d == 64) {
        if (small_m) {
            GemmParams g = make_params(p, 64, err);
            g.qkv = e;
            return run_small_m<64, 8, EPI_QKV, 64>(p, g, num_sms, stream);
        }
        GemmParams g = make_params(p, 256, err);
        g.qkv = e;
        const cudaError_t pe = run_pair<6, EPI_QKV, 64>(p, g, 16, stream);
        if (pe != cudaErrorNotSupported) return pe;
        return run<256, 4, EPI_QKV, 64>(p, g, num_sms, stream);
    }
    // widths that do not divide 256: a tile of whole heads (3 x 80, 2 x 96)
    if (e.d == 80) {
        GemmParams g = make_params(p, 240, err);
        g.qkv = e;
        return run<240, 4, EPI_QKV, 80>(p, g, num_sms, stream);
    }
    if (e.d == 96) {
        GemmParams g = make_params(p, 192, err);
        g.qkv = e;
        return run<192, 4, EPI_QKV, 96>(p, g, num_sms, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_residual(const GemmProblem &p, const ResidualEpilogue &e, unsigned *err, int num_sms,
                                 cudaStream_t stream)
{
    if (p.M <= BM) {
        GemmParams g = make_params(p, 64, err);
        g.res = e;
        return run_small_m<64, 8, EPI_RESIDUAL, 0>(p, g, num_sms, stream);
    }
    GemmParams g = make_params(p, 256, err);
    g.res = e;
    // o_proj's A panels are twice as long (K = Hq*d): half the QKV projection's group
    const cudaError_t pe = run_pair<6, EPI_RESIDUAL, 0>(p, g, 8, stream);
    if (pe != cudaErrorNotSupported) return pe;
    g.group_m = 16;
    return run<256, 4, EPI_RESIDUAL, 0>(p, g, num_sms, stream);
}

}  // namespace gqa

namespace gqa {

// Backward-pass products (see internal.h).
cudaError_t launch_gemm_general(const GemmProblem &p, int a_mn, int b_mn, int epi, const GemmOut &o, unsigned *err,
                                int num_sms, cudaStream_t stream)
{
    GemmParams g = make_params(p, 256, err);
    g.f32_out = o.f32;
    g.head = o.head;
    g.res = o.res;
    const int maj = (a_mn ? 1 : 0) | (b_mn ? 2 : 0);
#define GQA_RUN(E, M_) return run<256, 4, E, 0, M_>(p, g, num_sms, stream)
    if (epi == GEMM_OUT_F32) {
        if (maj == 3) GQA_RUN(EPI_F32, 3);
        if (maj == 0) GQA_RUN(EPI_F32, 0);
    } else if (epi == GEMM_OUT_HEAD16) {
        if (maj == 2) GQA_RUN(EPI_HEAD16, 2);
    } else if (epi == GEMM_OUT_RESIDUAL) {
        if (maj == 2) GQA_RUN(EPI_RESIDUAL, 2);
    }
#undef GQA_RUN
    return cudaErrorInvalidValue;
}

}  // namespace gqa
