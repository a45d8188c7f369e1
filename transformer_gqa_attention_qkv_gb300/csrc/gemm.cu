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
//   warps 2..5  epilogue: tcgen05.ld gives a thread one output row; fused
//               math on packed fp32 pairs, 32-byte global stores where the
//               row address allows; residual rows are requested into L2
//               before the accumulator is ready.  The QKV epilogue has a
//               second warpgroup (warps 6..9, on the same TMEM lanes), and
//               the two take alternate column chunks of each row
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
enum { EPI_QKV = 0, EPI_RESIDUAL = 1, EPI_F32 = 2, EPI_HEAD16 = 3 };

// Epilogue warpgroups per CTA: two for the QKV epilogue (RMSNorm, RoPE and
// head-major stores are its critical path on short-K problems), one for the
// others (their epilogues hide behind the main loop; a second warpgroup made
// the long-K o_proj 3-8% slower).  Warps 0 and 1 are the TMA and MMA warps.
template <int EPI>
__host__ __device__ constexpr int epi_groups() { return EPI == EPI_QKV ? 2 : 1; }
template <int EPI>
__host__ __device__ constexpr int kernel_threads() { return 64 + 128 * epi_groups<EPI>(); }

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

// Barrier `id` over the first n threads that reach it (n a multiple of 32).
DEVI void named_barrier_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// Two TMEM loads of W columns each (the two halves of a RoPE pair chunk) and
// one wait, in one statement (no use of a or b can be scheduled before the
// data has arrived); W = 16 or 8, other widths take two waits.
template <int W>
DEVI void tmem_ldw2(uint32_t t1, uint32_t (&a)[W], uint32_t t2, uint32_t (&b)[W])
{
    if constexpr (W == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
            "{%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
              "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
              "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
              "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
            : "r"(t1), "r"(t2)
            : "memory");
    } else if constexpr (W == 8) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
              "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7])
            : "r"(t1), "r"(t2)
            : "memory");
    } else {
        tmem_ldw<W>(t1, a);
        tmem_ldw<W>(t2, b);
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

// N consecutive 32-bit words to dst (aligned to 4N bytes, 16 at most).
template <int N>
DEVI void st_words(void *dst, const uint32_t (&w)[N])
{
    if constexpr (N >= 8) {
#pragma unroll
        for (int i = 0; i < N / 8; ++i) {
            const uint32_t w8[8] = {w[8 * i], w[8 * i + 1], w[8 * i + 2], w[8 * i + 3],
                                    w[8 * i + 4], w[8 * i + 5], w[8 * i + 6], w[8 * i + 7]};
            st_global32(reinterpret_cast<uint32_t *>(dst) + 8 * i, w8);
        }
    } else if constexpr (N == 4) {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    } else if constexpr (N == 2) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    } else {
        static_assert(N == 1, "store width");
        *reinterpret_cast<uint32_t *>(dst) = w[0];
    }
}

// Two floats -> packed binary16x2, rounded to nearest even and saturated at
// the finite range (+-65504; NaN stays NaN), lo in the low half.
DEVI uint32_t pack_f16_sat(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Storage format of one projected head row: bf16, binary16 (saturated at its
// range and flagged), or E4M3 codes of value / scale (saturated and flagged).
struct OutFmt {
    int mode;     // 0 bf16, 1 binary16, 2 E4M3
    float scale;  // E4M3 only
};

// Columns [c, c + N) (N even) of a head row whose first element is at dst,
// from N/2 packed pairs.  binary16: *amax takes the largest magnitude stored
// (the caller flags values past the finite range once per row); E4M3:
// *clamped is set when a code saturated.
template <int N>
DEVI void putv(void *dst, int c, const float2 (&v)[N / 2], OutFmt f, float &amax, bool &clamped)
{
    if (f.mode != 2) {
        uint32_t w[N / 2];
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            if (f.mode == 1) {
                w[i] = pack_f16_sat(v[i].x, v[i].y);
                amax = fmax3(amax, fabsf(v[i].x), fabsf(v[i].y));
            } else {
                w[i] = pack_bf16(v[i].x, v[i].y);
            }
        }
        st_words<N / 2>(reinterpret_cast<uint16_t *>(dst) + c, w);
        return;
    }
    uint8_t *d8 = reinterpret_cast<uint8_t *>(dst) + c;
    if constexpr (N == 2) {
        const float q0 = __fdiv_rn(v[0].x, f.scale), q1 = __fdiv_rn(v[0].y, f.scale);
        clamped |= !(fabsf(q0) <= 448.0f) || !(fabsf(q1) <= 448.0f);
        *reinterpret_cast<uint16_t *>(d8) = (uint16_t)f32x2_to_e4m3x2(q0, q1);
    } else {
        uint32_t w[N / 4];
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            float q[4] = {v[2 * i].x, v[2 * i].y, v[2 * i + 1].x, v[2 * i + 1].y};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                q[k] = __fdiv_rn(q[k], f.scale);
                clamped |= !(fabsf(q[k]) <= 448.0f);
            }
            w[i] = f32x2_to_e4m3x2(q[0], q[1]) | (f32x2_to_e4m3x2(q[2], q[3]) << 16);
        }
        st_words<N / 4>(d8, w);
    }
}

// Widest TMEM chunk (<= 32 columns) that tiles n (even) columns.
__host__ __device__ constexpr int chunk_width(int n)
{
    return n % 32 == 0 ? 32 : n % 16 == 0 ? 16 : n % 8 == 0 ? 8 : n % 4 == 0 ? 4 : 2;
}
// The same, at most 16: the unit of the epilogue's RoPE and store passes, whose
// chunks the two warpgroups take in turn.
__host__ __device__ constexpr int chunk16(int n) { return n % 16 == 0 ? 16 : chunk_width(n); }

DEVI float2 f2(uint32_t a, uint32_t b) { return make_float2(__uint_as_float(a), __uint_as_float(b)); }

// The RoPE table of one row: rotary width RD, pairs (i, i + RD/2) taken W at a
// time, a warpgroup's chunks every other one.  cs is the quad table at the
// row's position: entry k * ld holds (cos, cos, sin, sin) of pairs 2k and
// 2k + 1, so the 32 rows of a warp (consecutive positions of one sequence in a
// prefill) read one coalesced 512-byte run per two pairs.  (Holding a row's
// entries in registers across the tile's heads, which share them, needs 32
// more registers than the epilogue warps have at 10 warps per CTA: 168.)
template <int RD>
struct RopeTab {
    static constexpr int W = RD > 0 ? chunk16(RD / 2) : 2;
    const float4 *cs;
    int ld;
};

// Pairs [c, c + W) of a Q or K row: normalised (x * rinv * w), rotated
// (rotate-half pairs (i, i + H), angle pos * theta^(-2i/RD)) and stored, on
// packed fp32 pairs.
template <int RD, bool NORM>
DEVI void rope_chunk(uint32_t col, void *dst, int c, float2 rr, const float *w, const float4 (&t)[RopeTab<RD>::W / 2],
                     bool row_ok, OutFmt fmt, float &amax, bool &clamped)
{
    constexpr int H = RD / 2, W = RopeTab<RD>::W;
    uint32_t a[W], b[W];
    tmem_ldw2<W>(col + c, a, col + c + H, b);
    if constexpr (NORM) {  // a, b <- x * rinv * w (in place, as fp32 bits)
#pragma unroll
        for (int q = 0; q < W / 2; ++q) {
            const float2 w1 = *reinterpret_cast<const float2 *>(w + c + 2 * q);
            const float2 w2 = *reinterpret_cast<const float2 *>(w + c + H + 2 * q);
            const float2 x1 = __fmul2_rn(f2(a[2 * q], a[2 * q + 1]), __fmul2_rn(rr, w1));
            const float2 x2 = __fmul2_rn(f2(b[2 * q], b[2 * q + 1]), __fmul2_rn(rr, w2));
            a[2 * q] = __float_as_uint(x1.x);
            a[2 * q + 1] = __float_as_uint(x1.y);
            b[2 * q] = __float_as_uint(x2.x);
            b[2 * q + 1] = __float_as_uint(x2.y);
        }
    }
    float2 y[W / 2];
#pragma unroll
    for (int q = 0; q < W / 2; ++q)  // first halves: x1 cos - x2 sin
        y[q] = __ffma2_rn(f2(a[2 * q], a[2 * q + 1]), make_float2(t[q].x, t[q].y),
                          __fmul2_rn(f2(b[2 * q], b[2 * q + 1]), make_float2(-t[q].z, -t[q].w)));
    if (row_ok) putv<W>(dst, c, y, fmt, amax, clamped);
#pragma unroll
    for (int q = 0; q < W / 2; ++q)  // second halves: x2 cos + x1 sin
        y[q] = __ffma2_rn(f2(b[2 * q], b[2 * q + 1]), make_float2(t[q].x, t[q].y),
                          __fmul2_rn(f2(a[2 * q], a[2 * q + 1]), make_float2(t[q].z, t[q].w)));
    if (row_ok) putv<W>(dst, c + H, y, fmt, amax, clamped);
}

// Normalised (x * rinv * w) head row of a Q or K head, rotated on its first
// RD features and stored; features [RD, D) are only normalised.  Warpgroup wg
// takes every other chunk.
template <int D, int RD, bool NORM>
DEVI void rope_store(uint32_t col, void *dst, float rinv, const float *w, const RopeTab<RD> &tab, bool row_ok,
                     OutFmt fmt, int wg, float &amax, bool &clamped)
{
    const float2 rr = make_float2(rinv, rinv);
    if constexpr (RD > 0) {
        constexpr int H = RD / 2, W = RopeTab<RD>::W;
        static_assert(W % 2 == 0, "pairs are taken two at a time");
#pragma unroll 1
        for (int c = wg * W; c < H; c += 2 * W) {
            float4 t[W / 2];
#pragma unroll
            for (int q = 0; q < W / 2; ++q) t[q] = __ldg(tab.cs + (size_t)(c / 2 + q) * tab.ld);
            rope_chunk<RD, NORM>(col, dst, c, rr, w, t, row_ok, fmt, amax, clamped);
        }
    }
    if constexpr (RD < D) {
        constexpr int CW = chunk16(D - RD);
#pragma unroll 1
        for (int c = RD + wg * CW; c < D; c += 2 * CW) {  // features past the rotary width
            uint32_t r[CW];
            tmem_ldw<CW>(col + c, r);
            float2 y[CW / 2];
#pragma unroll
            for (int q = 0; q < CW / 2; ++q) {
                y[q] = f2(r[2 * q], r[2 * q + 1]);
                if constexpr (NORM)
                    y[q] = __fmul2_rn(y[q], __fmul2_rn(rr, *reinterpret_cast<const float2 *>(w + c + 2 * q)));
            }
            if (row_ok) putv<CW>(dst, c, y, fmt, amax, clamped);
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
// out[((b*H + j)*S + t)*d + c] (saturated at binary16's range and flagged).
// Stored 16 columns at a time: d is a multiple of 16 (64, 80, 96, 128), so a
// 16-column piece never crosses a head, while a 32-column one would at d = 80.
template <int BN>
DEVI void epilogue_head16(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok)
{
    const HeadEpilogue &e = P.head;
    const int b = m / e.S, t = m - (m / e.S) * e.S;
    float amax = 0.0f;
    bool unused = false;
    const OutFmt f16{1, 1.0f};
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
            float2 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = f2(r[16 * h + 2 * i], r[16 * h + 2 * i + 1]);
            putv<16>(e.out + ((size_t)(b * e.H + j) * e.S + t) * e.d, cc, v, f16, amax, unused);
        }
    }
    if (amax > kHalfMax) atomicOr(P.err, kErrRange);
}

// The heads of one QKV tile row (BN columns = BN/D whole heads) at rotary
// width RD.  Both warpgroups take the sum of squares of a Q or K row over all
// its D columns (each loads the whole row from TMEM, so they never wait for
// each other); each then rotates and stores its own chunks.
template <int BN, int D, int RD>
DEVI void qkv_heads(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok, const float *s_norm, int wg,
                    int b, int pos, int q_slot, int kv_slot, float &amax, bool &clamped)
{
    constexpr int CWN = chunk_width(D);  // norm pass: TMEM chunk that tiles a head row (32, or 16 for d = 80)
    constexpr int CWV = chunk16(D);      // V rows: store chunk
    const QkvEpilogue &e = P.qkv;
    const int HqD = e.Hq * D, HkvD = e.Hkv * D;
    const bool has_norm = e.q_norm_w != nullptr;
    const RopeTab<RD> tab{RD > 0 ? e.rope + (row_ok ? pos : 0) : nullptr, e.rope_ld};
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
            for (int c = wg * CWV; c < D; c += 2 * CWV) {
                uint32_t r[CWV];
                tmem_ldw<CWV>(col + c, r);
                float2 v[CWV / 2];
#pragma unroll
                for (int i = 0; i < CWV / 2; ++i) v[i] = f2(r[2 * i], r[2 * i + 1]);
                if (row_ok) putv<CWV>(dst, c, v, fmt, amax, clamped);
            }
            continue;
        }
        float rinv = 1.0f;
        if (has_norm) {
            float2 ss2 = make_float2(0.0f, 0.0f);
            // pre-norm Q/K rows for the backward's RMSNorm gradient: [M, (Hq+Hkv)*D] fp32
            float *pre = e.pre_out ? e.pre_out + (size_t)m * (e.Hq + e.Hkv) * D + (kind == 0 ? head : e.Hq + head) * D
                                   : nullptr;
#pragma unroll 1
            for (int c = 0; c < D; c += CWN) {
                uint32_t r[CWN];
                tmem_ldw<CWN>(col + c, r);
#pragma unroll
                for (int i = 0; i < CWN / 2; ++i) {
                    const float2 f = f2(r[2 * i], r[2 * i + 1]);
                    ss2 = __ffma2_rn(f, f, ss2);
                }
                if (pre && row_ok && ((c / CWN) & 1) == wg) {
                    float4 *d4 = reinterpret_cast<float4 *>(pre + c);
#pragma unroll
                    for (int i = 0; i < CWN / 4; ++i)
                        d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                            __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
                }
            }
            rinv = 1.0f / sqrtf((ss2.x + ss2.y) * (1.0f / D) + e.eps);
            rope_store<D, RD, true>(col, dst, rinv, s_norm + (kind == 0 ? 0 : 256), tab, row_ok, fmt, wg, amax,
                                    clamped);
        } else {
            rope_store<D, RD, false>(col, dst, rinv, s_norm, tab, row_ok, fmt, wg, amax, clamped);
        }
    }
}

// Epilogue of one QKV tile row: the row's position and output slots, then its
// heads at the rotary width in use.
template <int BN, int D>
DEVI void epilogue_qkv(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok, const float *s_norm, int wg)
{
    static_assert(BN % D == 0, "a tile holds whole heads");
    const QkvEpilogue &e = P.qkv;
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
            if (wg == 0) atomicOr(P.err, kErrIndex);
            row_ok = false;
        }
    }
    float amax = 0.0f;
    bool clamped = false;
    if (e.rd == D)
        qkv_heads<BN, D, D>(P, tcol, m, n0, row_ok, s_norm, wg, b, pos, q_slot, kv_slot, amax, clamped);
    else if (e.rd == D / 2)
        qkv_heads<BN, D, D / 2>(P, tcol, m, n0, row_ok, s_norm, wg, b, pos, q_slot, kv_slot, amax, clamped);
    else if (e.rd == D / 4)
        qkv_heads<BN, D, D / 4>(P, tcol, m, n0, row_ok, s_norm, wg, b, pos, q_slot, kv_slot, amax, clamped);
    else
        qkv_heads<BN, D, 0>(P, tcol, m, n0, row_ok, s_norm, wg, b, pos, q_slot, kv_slot, amax, clamped);
    if (amax > kHalfMax || clamped) atomicOr(P.err, kErrRange);
}

// out = acc + resid, bf16 rows; the residual of the next 32 columns is loaded
// while this chunk is added.
template <int BN>
DEVI void epilogue_residual(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok)
{
    const ResidualEpilogue &e = P.res;
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
                for (int q = 0; q < 4; ++q) {
                    const float2 sum = __fadd2_rn(f2(r[8 * v + 2 * q], r[8 * v + 2 * q + 1]),
                                                  make_float2(bf16lo(xs[q]), bf16hi(xs[q])));
                    o[4 * v + q] = pack_bf16(sum.x, sum.y);
                }
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
// (Loading them into registers at that point, and the same prefetch for the
// RoPE table rows of the QKV epilogue, measured slower.)
DEVI void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int BN, int EPI>
DEVI void epilogue_prefetch(const GemmParams &P, int m, int n0, bool row_ok)
{
    if constexpr (EPI == EPI_RESIDUAL) {
        const int cols = min(BN, P.N - n0);  // a multiple of 8: whole 16-byte units
        if (row_ok && cols > 0) prefetch_l2(P.res.resid + (size_t)m * P.N + n0, (uint32_t)cols * 2);
    }
}

// The tile's epilogue: one thread per accumulator row; wg is the thread's
// epilogue warpgroup (the QKV epilogue's two split the row's chunks).
template <int BN, int EPI, int D>
DEVI void epilogue_tile(const GemmParams &P, uint32_t tcol, int m, int n0, bool row_ok, const float *s_norm, int wg)
{
    if constexpr (EPI == EPI_QKV)
        epilogue_qkv<BN, D>(P, tcol, m, n0, row_ok, s_norm, wg);
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
__global__ void __launch_bounds__(kernel_threads<EPI>(), 1)
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
            mbar_init(tempty + a, 4 * epi_groups<EPI>());
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
        for (int i = threadIdx.x - 64; i < D; i += kernel_threads<EPI>() - 64) {
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
        const int quarter = warp & 3;    // TMEM lanes this warp may access
        const int wg = (warp - 2) >> 2;  // epilogue warpgroup: which column chunks
        const int row = quarter * 32 + lane;
        grid_dep_wait();  // the epilogue reads and writes what the previous kernel may touch
        int use = 0;
        for (int tile = tile0; tile < P.num_tiles; tile += tile_step, ++use) {
            int mb, nb;
            tile_coords(tile, P.num_m, P.num_n, P.group_m, mb, nb);
            const int acc = use & 1;
            const int m = mb * BM + row;
            if constexpr (KS > 1) {  // the cluster sums the partials below
                acc_ready = __all_sync(0xffffffffu, mbar_wait(tfull + acc, (use >> 1) & 1, err));
                break;
            }
            epilogue_prefetch<BN, EPI>(P, m, nb * BN, m < P.M);
            if (!mbar_wait(tfull + acc, (use >> 1) & 1, err)) break;
            tc_fence_after();
            const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16) + acc * ACC;
            epilogue_tile<BN, EPI, D>(P, tcol, m, nb * BN, m < P.M, s_norm, wg);
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
        // every epilogue warp of the CTA takes the same path below (they meet at a named barrier)
        const bool all_ready = __syncthreads_and(warp < 2 || acc_ready);
        cluster_sync();
        const int quarter = warp & 3;
        constexpr int NWG = epi_groups<EPI>();
        const int wg = (warp - 2) >> 2;  // epilogue warpgroup (warps >= 2): every NWG-th 16 columns
        const int row = quarter * 32 + lane;
        const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16);
        int mb = 0, nb = 0;
        if (tile0 < P.num_tiles) tile_coords(tile0, P.num_m, P.num_n, P.group_m, mb, nb);
        const int m = mb * BM + row;
        const bool active = warp >= 2 && tile0 < P.num_tiles && all_ready;  // uniform over the epilogue warps
        if (active && crank != 0) {
            tc_fence_after();
            const uint32_t dst = cluster_map(smem_u32(smem), 0) + (uint32_t)(((crank - 1) * BM + row) * PART_LD * 4);
#pragma unroll 1
            for (int c = 16 * wg; c < BN; c += 16 * NWG) {
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
            for (int c = 16 * wg; c < BN; c += 16 * NWG) {
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
            // every warpgroup's partial sums are in TMEM before another reads its columns
            tc_fence_before();
            if constexpr (NWG > 1)
                named_barrier_sync(1, NWG * 128);
            else
                __syncwarp();
            tc_fence_after();
            epilogue_tile<BN, EPI, D>(P, tcol, m, nb * BN, m < P.M, s_norm, wg);
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
//   warps 2.. (both)     epilogue; the accumulator is released by arriving
//                        on the even CTA's `tempty` (every epilogue warp of both CTAs)
// BN: N of the pair's MMA, a tile of whole heads (256; 240 = 3 x 80 and
// 192 = 2 x 96 for the head widths that do not divide 256), half of its B rows
// staged by each CTA.
template <int STAGES, int EPI, int D, int BN = 256>
__global__ void __launch_bounds__(kernel_threads<EPI>(), 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const GemmParams P)
{
    constexpr int BNH = BN / 2;  // B rows staged by each CTA
    static_assert(BN % 16 == 0 && BNH % 8 == 0 && BN <= 256, "pair MMA N; whole 8-row swizzle groups per CTA");
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
            mbar_init(tempty + a, 8 * epi_groups<EPI>());  // the epilogue warps of both CTAs
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
        for (int i = threadIdx.x - 64; i < D; i += kernel_threads<EPI>() - 64) {
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
        const int quarter = warp & 3;    // TMEM lanes this warp may access
        const int wg = (warp - 2) >> 2;  // epilogue warpgroup: which column chunks
        const int row = quarter * 32 + lane;
        grid_dep_wait();  // the epilogue reads and writes what the previous kernel may touch
        int use = 0;
        for (int tile = tile0; tile < P.num_tiles; tile += tile_step, ++use) {
            int mb, nb;
            tile_coords(tile, P.num_m, P.num_n, P.group_m, mb, nb);
            const int acc = use & 1;
            const int m = mb * 2 * BM + (int)rank * BM + row;
            epilogue_prefetch<BN, EPI>(P, m, nb * BN, m < P.M);
            if (!mbar_wait<true>(tfull + acc, (use >> 1) & 1, err)) break;
            tc_fence_after();
            const uint32_t tcol = tmem + ((uint32_t)(quarter * 32) << 16) + acc * ACC;
            epilogue_tile<BN, EPI, D>(P, tcol, m, nb * BN, m < P.M, s_norm, wg);
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
    LaunchCfg lc(dim3(grid), dim3(kernel_threads<EPI>()), L::ALLOC, stream, p.pdl != 0, KS);
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
        cfg.blockDim = dim3(kernel_threads<EPI>());
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

// The pair kernel over 256 x BN tiles (tile rows of 256 = two CTAs' 128), as
// many 2-CTA clusters as fit on the GPU at once; returns cudaErrorNotSupported
// when the cluster shape cannot be placed (the caller then runs the single-SM
// kernel).
template <int STAGES, int EPI, int D, int BN = 256>
cudaError_t run_pair(const GemmProblem &p, GemmParams params, int group_m, cudaStream_t stream)
{
    constexpr int SMEM = STAGES * (BM * BK * 2 + BN / 2 * BK * 2) + (2 * STAGES + 5) * 8 + 32 + 2 * 256 * 4 + 1024;
    CUtensorMap ta, tb;
    const uint64_t dA[2] = {(uint64_t)p.K, (uint64_t)p.M};
    const uint64_t sA[1] = {(uint64_t)p.K * 2};
    const uint64_t dB[2] = {(uint64_t)p.K, (uint64_t)p.N};
    const uint64_t sB[1] = {(uint64_t)p.K * 2};
    const uint32_t bA[2] = {(uint32_t)BK, (uint32_t)BM};
    const uint32_t bB[2] = {(uint32_t)BK, (uint32_t)(BN / 2)};
    if (encode_tmap(&ta, p.A, 2, dA, sA, bA, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (encode_tmap(&tb, p.B, 2, dB, sB, bB, true) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    params.num_m = (p.M + 2 * BM - 1) / (2 * BM);  // pair-tile rows
    params.num_n = (p.N + BN - 1) / BN;
    params.num_tiles = params.num_m * params.num_n;
    params.group_m = group_m;
    if (!cta_pairs_enabled()) return cudaErrorNotSupported;
    auto kern = gemm_pair_kernel<STAGES, EPI, D, BN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    int clusters = 0;
    {
        LaunchCfg probe(dim3(2), dim3(kernel_threads<EPI>()), SMEM, stream, false, 2);
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &probe.cfg) != cudaSuccess || clusters < 1) {
            cudaGetLastError();
            return cudaErrorNotSupported;
        }
    }
    const int n = params.num_tiles < clusters ? params.num_tiles : clusters;
    LaunchCfg lc(dim3(2 * n), dim3(kernel_threads<EPI>()), SMEM, stream, p.pdl != 0, 2);
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
    if (e.d == 256) {  // one 256-wide head per tile (its epilogue sets the pace: the pair form measured 9% slower)
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
        if (!small_m) {
            const cudaError_t pe = run_pair<6, EPI_QKV, 80, 240>(p, g, 16, stream);
            if (pe != cudaErrorNotSupported) return pe;
        }
        return run<240, 4, EPI_QKV, 80>(p, g, num_sms, stream);
    }
    if (e.d == 96) {
        GemmParams g = make_params(p, 192, err);
        g.qkv = e;
        if (!small_m) {
            const cudaError_t pe = run_pair<6, EPI_QKV, 96, 192>(p, g, 16, stream);
            if (pe != cudaErrorNotSupported) return pe;
        }
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
