// api.cu -- the C ABI declared in include/gqa_attn.h: argument validation,
// per-device state (error word, RoPE tables, default workspace), tensor-map
// encoding, and the launch sequences of the prefill forward and decode step.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "../../include/gqa_attn.h"
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace gqa {

// ------------------------------------------------------------ error state

static thread_local char g_msg[512] = "";
static thread_local int g_launches = 0;

static int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

void record_error_message(const char *msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

void set_launch_count(int n) { g_launches = n; }

static int cuda_fail(cudaError_t e, const char *what)
{
    return fail(GQA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// -------------------------------------------------------- tensor-map encoder

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encoder()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

CUresult encode_tmap(CUtensorMap *map, const void *base, int rank, const uint64_t *dims, const uint64_t *strides_bytes,
                     const uint32_t *box, bool swizzle128, int elem_bytes)
{
    EncodeTiledFn fn = get_encoder();
    if (!fn) return CUDA_ERROR_NOT_INITIALIZED;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    const CUtensorMapDataType type = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    return fn(map, type, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// --------------------------------------------------------- per-device state

struct RopeTable {
    double theta;
    int d;
    int rows;
    float2 *dev;    // [rows][d/2]: position-major (a warp reads one position's pairs)
    float4 *dev_t;  // [d/4][rows]: quads of pairs 2k, 2k + 1 (a warp reads one quad at 32 consecutive positions)
};

struct DeviceState {
    bool init = false;
    int num_sms = 0;
    unsigned *err = nullptr;             // device error word
    std::vector<RopeTable> ropes;        // kept until exit (kernels may still read old ones)
    void *ws = nullptr;                  // default workspace of gqa_attn_forward
    size_t ws_bytes = 0;
};

static std::mutex g_mu;
static DeviceState g_dev[64];

static int device_state(DeviceState **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(GQA_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);  // first calls from several threads initialise once
    DeviceState &st = g_dev[dev];
    if (!st.init) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(GQA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, major,
                        minor);
        e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaMalloc(&st.err, 256);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
        e = cudaMemset(st.err, 0, 256);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
        if (!get_encoder()) return fail(GQA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        st.init = true;
    }
    *out = &st;
    return GQA_OK;
}

// cos/sin(pos * theta^(-2i/d)) for pos < rows, i < d/2 (d: the rotary width), computed in double on
// the host and stored as fp32 (cos, sin) pairs.  Angles reach ~1.6e4 rad, where
// an fp32 angle would already be off by ~1e-3 rad.
// The (cos, sin) table of RoPE for (theta, width d) and at least `rows`
// positions, in two layouts: position-major (cos, sin) pairs, and the quad
// layout of the projection epilogue (entry [k][p] = (cos, cos, sin, sin) of
// pairs 2k and 2k + 1 at position p, so a warp's consecutive positions read
// one coalesced run and the epilogue rotates two pairs per packed fp32x2
// operation); *ld (if given) is the quad layout's row length.
static int rope_table(DeviceState &st, double theta, int d, int rows, const float2 **out,
                      const float4 **out_t = nullptr, int *ld = nullptr)
{
    for (const RopeTable &t : st.ropes)
        if (t.theta == theta && t.d == d && t.rows >= rows) {
            *out = t.dev;
            if (out_t) *out_t = t.dev_t;
            if (ld) *ld = t.rows;
            return GQA_OK;
        }
    int cap = 4096;
    while (cap < rows) cap *= 2;
    const int H = d / 2;  // even for every rotary width the kernels take
    std::vector<float2> host((size_t)cap * H);
    std::vector<float4> host_t((size_t)cap * (H / 2));
    for (int p = 0; p < cap; ++p)
        for (int i = 0; i < H; ++i) {
            const double f = (double)p * pow(theta, -2.0 * i / d);
            const float2 cs = make_float2((float)cos(f), (float)sin(f));
            host[(size_t)p * H + i] = cs;
            float4 &q = host_t[(size_t)(i / 2) * cap + p];
            if (i % 2 == 0) {
                q.x = cs.x;
                q.z = cs.y;
            } else {
                q.y = cs.x;
                q.w = cs.y;
            }
        }
    float2 *dev = nullptr;
    float4 *dev_t = nullptr;
    cudaError_t e = cudaMalloc(&dev, host.size() * sizeof(float2));
    if (e == cudaSuccess) e = cudaMalloc(&dev_t, host_t.size() * sizeof(float4));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(rope table)");
    e = cudaMemcpy(dev, host.data(), host.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemcpy(dev_t, host_t.data(), host_t.size() * sizeof(float4), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(rope table)");
    st.ropes.push_back({theta, d, cap, dev, dev_t});
    *out = dev;
    if (out_t) *out_t = dev_t;
    if (ld) *ld = cap;
    return GQA_OK;
}

// ------------------------------------------------------------- validation

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static bool overlap(const void *a, size_t na, const void *b, size_t nb)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + nb && y < x + na;
}

static int check_layer(int B, int S, int hidden, int Hq, int Hkv, int d, const void *qn, const void *kn)
{
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || d <= 0)
        return fail(GQA_ERR_ARG, "sizes must be positive (B=%d S=%d hidden=%d Hq=%d Hkv=%d head_dim=%d)", B, S, hidden,
                    Hq, Hkv, d);
    if (Hq % Hkv) return fail(GQA_ERR_ARG, "Hq=%d is not a multiple of Hkv=%d", Hq, Hkv);
    if (d & 1) return fail(GQA_ERR_ARG, "head_dim=%d is odd; RoPE pairs need an even head_dim", d);
    if ((qn == nullptr) != (kn == nullptr))
        return fail(GQA_ERR_ARG, "q_norm_w and k_norm_w must both be given or both be NULL");
    if (d != 64 && d != 80 && d != 96 && d != 128 && d != 256)
        return fail(GQA_ERR_UNSUPPORTED, "unsupported head_dim: %d (supported: 64, 80, 96, 128, 256)", d);
    if (hidden % 8) return fail(GQA_ERR_UNSUPPORTED, "unsupported hidden: %d (must be a multiple of 8)", hidden);
    if ((long long)B * S > (1LL << 30) || (long long)(Hq + 2 * Hkv) * d > (1 << 20) || hidden > (1 << 20))
        return fail(GQA_ERR_UNSUPPORTED, "problem too large");
    return GQA_OK;
}

// Forward attention: any group size up to the 128 rows of a query tile (the
// tile packs floor(128 / G) positions of each of the G heads).
static int check_group(int Hq, int Hkv)
{
    const int G = Hq / Hkv;
    if (G > 128) return fail(GQA_ERR_UNSUPPORTED, "unsupported group size Hq/Hkv=%d (at most 128)", G);
    return GQA_OK;
}

// rotary_dim: even, in [0, head_dim]; the kernels implement d, d/2, d/4 and 0.
static int check_rotary(int rd, int d)
{
    if (rd < 0 || rd > d || (rd & 1))
        return fail(GQA_ERR_ARG, "rotary_dim=%d must be even and in [0, head_dim=%d]", rd, d);
    if (rd != d && rd != d / 2 && rd != d / 4 && rd != 0)
        return fail(GQA_ERR_UNSUPPORTED, "unsupported rotary_dim=%d (supported: head_dim, head_dim/2, head_dim/4, 0)",
                    rd);
    return GQA_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct FwdLayout {
    size_t q, k, v, attn, total;
};

static FwdLayout fwd_layout(int B, int S, int Hq, int Hkv, int d)
{
    FwdLayout L;
    const size_t tok = (size_t)B * S;
    L.q = 0;
    L.k = L.q + align256(tok * Hq * d * 2);
    L.v = L.k + align256(tok * Hkv * d * 2);
    L.attn = L.v + align256(tok * Hkv * d * 2);
    L.total = L.attn + align256(tok * Hq * d * 2);
    return L;
}

// ------------------------------------------------------------ stage runners

static int run_qkv(DeviceState &st, const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *qn, const gqa_bf16 *kn,
                   float theta, float eps, int rd, int B, int S, int hidden, int Hq, int Hkv, int d, const int *pos_dev,
                   int q_seq, int kv_seq, int rope_rows, int q_f16, int kv_f16, uint16_t *q_out, uint16_t *k_out,
                   uint16_t *v_out, cudaStream_t stream, int kv_fp8 = 0, float k_scale = 1.0f, float v_scale = 1.0f,
                   float *pre_out = nullptr, int rows = -1, int m0 = 0)
{
    const float2 *rope = nullptr;
    const float4 *rope_t = nullptr;
    int rope_ld = 0;
    if (rd > 0) {
        int rc;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            rc = rope_table(st, (double)theta, rd, rope_rows, &rope, &rope_t, &rope_ld);
        }
        if (rc) return rc;
    }
    // rows >= 0: rows [m0, m0 + rows) of the B*S token rows, x pointing at row m0
    GemmProblem p{x, Wqkv, rows >= 0 ? rows : B * S, (Hq + 2 * Hkv) * d, hidden};
    QkvEpilogue e{};
    e.m0 = m0;
    e.Hq = Hq;
    e.Hkv = Hkv;
    e.d = d;
    e.S = S;
    e.pos_dev = pos_dev;
    e.q_seq = q_seq;
    e.kv_seq = kv_seq;
    e.q_norm_w = qn;
    e.k_norm_w = kn;
    e.eps = eps;
    e.rd = rd;
    e.rope = rope_t;
    e.rope_ld = rope_ld;
    e.rope_rows = rope_rows;
    e.q_f16 = q_f16;     // binary16 unless Q meets a bf16 cache in the same MMA
    e.kv_f16 = kv_f16;   // prefill: binary16 workspace; cached paths: the bf16 cache
    e.kv_fp8 = kv_fp8;   // decode into an E4M3 cache
    e.pre_out = pre_out; // backward: the pre-norm Q/K rows
    e.k_scale = k_scale;
    e.v_scale = v_scale;
    e.q_out = q_out;
    e.k_out = k_out;
    e.v_out = v_out;
    cudaError_t ce = launch_gemm_qkv(p, e, st.err, st.num_sms, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "QKV projection launch");
    ++g_launches;
    return GQA_OK;
}

// pdl (here and below): the kernel follows one of this library's kernels in the
// same entry point and is launched as its programmatic dependent.
static int run_attention(DeviceState &st, const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int S,
                         int Hq, int Hkv, int d, int causal, gqa_bf16 *out, cudaStream_t stream, int kv_seq = 0,
                         const int *kv_start = nullptr, int cached = 0, float *lse = nullptr, int lse_ld = 0,
                         int pdl = 0, int kv_splits = 1, uint16_t *part_o = nullptr, float *part_lse = nullptr)
{
    AttentionProblem p{q,         k,        v,        out, B,   S,      Hq, Hkv, d, causal ? 1 : 0,
                       kv_seq > 0 ? kv_seq : S, kv_start, cached, lse, lse_ld, pdl, kv_splits, part_o, part_lse};
    cudaError_t ce = launch_attention(p, st.err, st.num_sms, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "attention launch");
    g_launches += kv_splits > 1 && part_o && part_lse && cached && d != 256 ? 2 : 1;
    return GQA_OK;
}

static int run_oproj(DeviceState &st, const gqa_bf16 *attn, const gqa_bf16 *Wo, const gqa_bf16 *x, int M, int hidden,
                     int qw, gqa_bf16 *out, cudaStream_t stream, int pdl = 0)
{
    GemmProblem p{attn, Wo, M, hidden, qw, pdl};
    ResidualEpilogue e{x, out};
    cudaError_t ce = launch_gemm_residual(p, e, st.err, st.num_sms, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "o_proj launch");
    ++g_launches;
    return GQA_OK;
}

static int run_decode_attn(DeviceState &st, const gqa_bf16 *q, const void *kc, const void *vc,
                           const int *len, int bias, int B, int Hq, int Hkv, int d, int Lmax, gqa_bf16 *out,
                           float *partials, int splits, cudaStream_t stream, int fp8 = 0, float k_scale = 1.0f,
                           float v_scale = 1.0f, int pdl = 0)
{
    DecodeAttentionProblem p{};
    p.pdl = pdl;
    p.q = q;
    p.k_cache = kc;
    p.v_cache = vc;
    p.fp8 = fp8;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.len = len;
    p.len_bias = bias;
    p.out = out;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.Lmax = Lmax;
    p.partials = partials;
    p.splits = splits;
    cudaError_t ce = launch_decode_attention(p, st.err, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "decode attention launch");
    g_launches += 2;
    return GQA_OK;
}

}  // namespace gqa

using namespace gqa;

namespace gqa {
static std::atomic<int> g_cta_pairs{1};
bool cta_pairs_enabled() { return g_cta_pairs.load(std::memory_order_relaxed) != 0; }
int set_cta_pairs(int enable) { return g_cta_pairs.exchange(enable ? 1 : 0); }
}  // namespace gqa

// =================================================================== C ABI

extern "C" {

const char *gqa_last_error(void) { return g_msg; }

int gqa_last_launch_count(void) { return g_launches; }

int gqa_set_cta_pairs(int enable) { return set_cta_pairs(enable); }

size_t gqa_attn_workspace_size(int B, int S, int hidden, int Hq, int Hkv, int head_dim)
{
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0) return 0;
    return fwd_layout(B, S, Hq, Hkv, head_dim).total;
}

int gqa_qkv_proj_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                 float rope_theta, float eps, int rotary_dim, int B, int S, int hidden, int Hq, int Hkv, int head_dim,
                 gqa_f16 *q_out, gqa_f16 *k_out, gqa_f16 *v_out, void *stream)
{
    g_launches = 0;
    int rc = check_layer(B, S, hidden, Hq, Hkv, head_dim, q_norm_w, k_norm_w);
    if (rc) return rc;
    if (!x || !Wqkv || !q_out || !k_out || !v_out) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(q_out) || !aligned16(k_out) || !aligned16(v_out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    if ((rc = check_rotary(rotary_dim, head_dim))) return rc;
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    return run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim,
                   nullptr, S, S, S, 1, 1, q_out, k_out, v_out, (cudaStream_t)stream);
}

int gqa_attention(const gqa_f16 *q, const gqa_f16 *k, const gqa_f16 *v, int B, int S, int Hq, int Hkv,
                  int head_dim, int causal, gqa_bf16 *attn_out, void *stream)
{
    g_launches = 0;
    int rc = check_layer(B, S, 8, Hq, Hkv, head_dim, nullptr, nullptr);
    if (rc) return rc;
    if ((rc = check_group(Hq, Hkv))) return rc;
    if (!q || !k || !v || !attn_out) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(attn_out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    return run_attention(*st, q, k, v, B, S, Hq, Hkv, head_dim, causal, attn_out, (cudaStream_t)stream);
}

int gqa_oproj_residual(const gqa_bf16 *attn, const gqa_bf16 *Wo, const gqa_bf16 *x, int M, int hidden, int q_width,
                       gqa_bf16 *out, void *stream)
{
    g_launches = 0;
    if (M <= 0 || hidden <= 0 || q_width <= 0) return fail(GQA_ERR_ARG, "sizes must be positive");
    if (hidden % 8 || q_width % 8) return fail(GQA_ERR_UNSUPPORTED, "hidden and q_width must be multiples of 8");
    if (!attn || !Wo || !x || !out) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (!aligned16(attn) || !aligned16(Wo) || !aligned16(x) || !aligned16(out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (overlap(out, (size_t)M * hidden * 2, x, (size_t)M * hidden * 2))
        return fail(GQA_ERR_ARG, "out must not overlap x");
    DeviceState *st;
    int rc;
    if ((rc = device_state(&st))) return rc;
    return run_oproj(*st, attn, Wo, x, M, hidden, q_width, out, (cudaStream_t)stream);
}

int gqa_attn_forward_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                        const gqa_bf16 *k_norm_w, float rope_theta, float eps, int rotary_dim, int B, int S,
                        int hidden, int Hq, int Hkv, int head_dim, int causal, gqa_bf16 *out, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_layer(B, S, hidden, Hq, Hkv, head_dim, q_norm_w, k_norm_w);
    if (rc) return rc;
    if ((rc = check_group(Hq, Hkv))) return rc;
    if (!x || !Wqkv || !Wo || !out) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    if ((rc = check_rotary(rotary_dim, head_dim))) return rc;
    const size_t nx = (size_t)B * S * hidden * 2;
    const size_t nw = (size_t)(Hq + 2 * Hkv) * head_dim * hidden * 2, no = (size_t)hidden * Hq * head_dim * 2;
    if (overlap(out, nx, x, nx) || overlap(out, nx, Wqkv, nw) || overlap(out, nx, Wo, no))
        return fail(GQA_ERR_ARG, "out must not overlap x or the weights");
    const FwdLayout L = fwd_layout(B, S, Hq, Hkv, head_dim);
    if (!workspace || workspace_bytes < L.total)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", L.total,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    if (overlap(workspace, L.total, out, nx) || overlap(workspace, L.total, x, nx))
        return fail(GQA_ERR_ARG, "workspace must not overlap the arguments");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    uint8_t *ws = (uint8_t *)workspace;
    gqa_bf16 *q = (gqa_bf16 *)(ws + L.q), *k = (gqa_bf16 *)(ws + L.k), *v = (gqa_bf16 *)(ws + L.v);
    gqa_bf16 *attn = (gqa_bf16 *)(ws + L.attn);
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim,
                      nullptr, S, S, S, 1, 1, q, k, v, s)))
        return rc;
    if ((rc = run_attention(*st, q, k, v, B, S, Hq, Hkv, head_dim, causal, attn, s, 0, nullptr, 0, nullptr, 0, 1)))
        return rc;
    return run_oproj(*st, attn, Wo, x, B * S, hidden, Hq * head_dim, out, s, 1);
}

// ----------------------------------------------- forward from host buffers

size_t gqa_attn_forward_host_workspace_size(int B, int S, int hidden, int Hq, int Hkv, int head_dim)
{
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0) return 0;
    const size_t nx = align256((size_t)B * S * hidden * 2);
    return fwd_layout(B, S, Hq, Hkv, head_dim).total + 2 * nx;  // + device copies of x and out
}

// Token chunks of the host pipeline: at most kHostChunks, each a multiple of
// the 128-row GEMM tile (so every output element is computed exactly as by
// the one-shot forward), and none below 2048 rows.
static constexpr int kHostChunks = 4;
static int host_chunk_rows(int M)
{
    int n = M / 2048;
    n = n < 1 ? 1 : (n > kHostChunks ? kHostChunks : n);
    int r = (M + n - 1) / n;
    return (r + 127) / 128 * 128;
}

// A copy stream and its events, per device, created on first use.
struct HostPipe {
    std::mutex mu;  // one call at a time enqueues through these events
    bool init = false;
    cudaStream_t copy = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, in[kHostChunks] = {}, out[kHostChunks] = {};
};
static HostPipe g_pipe[64];

static int host_pipe(HostPipe **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(GQA_ERR_CUDA, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    HostPipe &p = g_pipe[dev];
    if (!p.init) {
        if ((e = cudaStreamCreateWithFlags(&p.copy, cudaStreamNonBlocking)) != cudaSuccess)
            return cuda_fail(e, "copy stream");
        cudaEvent_t *evs[2 + 2 * kHostChunks] = {&p.fork, &p.join};
        for (int i = 0; i < kHostChunks; ++i) {
            evs[2 + i] = &p.in[i];
            evs[2 + kHostChunks + i] = &p.out[i];
        }
        for (cudaEvent_t *ev : evs)
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "pipeline event");
        p.init = true;
    }
    *out = &p;
    return GQA_OK;
}

int gqa_attn_forward_host(const gqa_bf16 *x_host, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                          const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B,
                          int S, int hidden, int Hq, int Hkv, int head_dim, int causal, gqa_bf16 *out_host,
                          void *workspace, size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_layer(B, S, hidden, Hq, Hkv, head_dim, q_norm_w, k_norm_w);
    if (rc) return rc;
    if ((rc = check_group(Hq, Hkv))) return rc;
    if (!x_host || !Wqkv || !Wo || !out_host) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (!aligned16(Wqkv) || !aligned16(Wo)) return fail(GQA_ERR_ARG, "weight pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    const size_t nx = (size_t)B * S * hidden * 2;
    if (overlap(out_host, nx, x_host, nx)) return fail(GQA_ERR_ARG, "out_host must not overlap x_host");
    for (const void *h : {(const void *)x_host, (const void *)out_host}) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, h) == cudaSuccess && a.type == cudaMemoryTypeDevice)
            return fail(GQA_ERR_ARG, "x_host and out_host must be host memory");
        (void)cudaGetLastError();
    }
    const FwdLayout L = fwd_layout(B, S, Hq, Hkv, head_dim);
    const size_t nx_al = align256(nx);
    const size_t need = L.total + 2 * nx_al;
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    HostPipe *pp;
    if ((rc = host_pipe(&pp))) return rc;
    std::lock_guard<std::mutex> lk(pp->mu);
    uint8_t *ws = (uint8_t *)workspace;
    gqa_bf16 *q = (gqa_bf16 *)(ws + L.q), *k = (gqa_bf16 *)(ws + L.k), *v = (gqa_bf16 *)(ws + L.v);
    gqa_bf16 *attn = (gqa_bf16 *)(ws + L.attn);
    gqa_bf16 *x = (gqa_bf16 *)(ws + L.total), *out = (gqa_bf16 *)(ws + L.total + nx_al);
    cudaStream_t s = (cudaStream_t)stream, c = pp->copy;
    const int M = B * S, R = host_chunk_rows(M), n = (M + R - 1) / R;
    const int qw = Hq * head_dim;
    cudaError_t e;
    // on any failure past this point the caller's stream still waits for the
    // copies already queued, so no later work of the caller races them
    auto bail = [&](int code) {
        if (cudaEventRecord(pp->join, c) == cudaSuccess) cudaStreamWaitEvent(s, pp->join, 0);
        return code;
    };
    // copies of x in, chunk by chunk, on the copy stream (after the caller's prior work)
    if ((e = cudaEventRecord(pp->fork, s)) != cudaSuccess || (e = cudaStreamWaitEvent(c, pp->fork, 0)) != cudaSuccess)
        return cuda_fail(e, "pipeline fork");
    for (int i = 0; i < n; ++i) {
        const size_t r0 = (size_t)i * R, rows = (size_t)(i + 1 < n ? R : M - i * R);
        if ((e = cudaMemcpyAsync(x + r0 * hidden, x_host + r0 * hidden, rows * hidden * 2, cudaMemcpyHostToDevice,
                                 c)) != cudaSuccess ||
            (e = cudaEventRecord(pp->in[i], c)) != cudaSuccess)
            return bail(cuda_fail(e, "host-to-device copy"));
    }
    // each chunk's projection as soon as its rows have landed
    for (int i = 0; i < n; ++i) {
        const int r0 = i * R, rows = i + 1 < n ? R : M - i * R;
        if ((e = cudaStreamWaitEvent(s, pp->in[i], 0)) != cudaSuccess) return bail(cuda_fail(e, "pipeline wait"));
        if ((rc = run_qkv(*st, x + (size_t)r0 * hidden, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, S,
                          hidden, Hq, Hkv, head_dim, nullptr, S, S, S, 1, 1, q, k, v, s, 0, 1.0f, 1.0f, nullptr,
                          rows, r0)))
            return bail(rc);
    }
    if ((rc = run_attention(*st, q, k, v, B, S, Hq, Hkv, head_dim, causal, attn, s, 0, nullptr, 0, nullptr, 0, 1)))
        return bail(rc);
    // o_proj chunk by chunk, each copied out while the next one is computed
    for (int i = 0; i < n; ++i) {
        const int r0 = i * R, rows = i + 1 < n ? R : M - i * R;
        if ((rc = run_oproj(*st, attn + (size_t)r0 * qw, Wo, x + (size_t)r0 * hidden, rows, hidden, qw,
                            out + (size_t)r0 * hidden, s, i == 0 ? 1 : 0)))
            return bail(rc);
        if ((e = cudaEventRecord(pp->out[i], s)) != cudaSuccess || (e = cudaStreamWaitEvent(c, pp->out[i], 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(out_host + (size_t)r0 * hidden, out + (size_t)r0 * hidden, (size_t)rows * hidden * 2,
                                 cudaMemcpyDeviceToHost, c)) != cudaSuccess)
            return bail(cuda_fail(e, "device-to-host copy"));
    }
    // the caller's stream resumes after the last copy
    if ((e = cudaEventRecord(pp->join, c)) != cudaSuccess || (e = cudaStreamWaitEvent(s, pp->join, 0)) != cudaSuccess)
        return cuda_fail(e, "pipeline join");
    return GQA_OK;
}

int gqa_attn_forward(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                     const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int S, int hidden, int Hq, int Hkv,
                     int head_dim, int causal, gqa_bf16 *out)
{
    g_launches = 0;
    int rc = check_layer(B, S, hidden, Hq, Hkv, head_dim, q_norm_w, k_norm_w);
    if (rc) return rc;
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    const size_t need = fwd_layout(B, S, Hq, Hkv, head_dim).total;
    void *ws;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (st->ws_bytes < need) {
            if (st->ws) {
                cudaError_t e = cudaDeviceSynchronize();
                if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
                cudaFree(st->ws);
                st->ws = nullptr;
                st->ws_bytes = 0;
            }
            cudaError_t e = cudaMalloc(&st->ws, need);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
            st->ws_bytes = need;
        }
        ws = st->ws;
    }
    return gqa_attn_forward_ex(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, B, S, hidden, Hq, Hkv, head_dim,
                               causal, out, ws, need, nullptr);
}

// ---------------------------------------------------------------- backward

// Attention backward workspace: o (bf16 [B*S, Hq*d]), lse and D (fp32 [B*Hq, ld]).
struct AttnBwdLayout {
    size_t o, lse, dsum, total;
    int ld;
};

static AttnBwdLayout attn_bwd_layout(int B, int S, int Hq, int d)
{
    AttnBwdLayout L;
    L.ld = (S + 3) & ~3;
    L.o = 0;
    L.lse = align256((size_t)B * S * Hq * d * 2);
    L.dsum = L.lse + align256((size_t)B * Hq * L.ld * 4);
    L.total = L.dsum + align256((size_t)B * Hq * L.ld * 4);
    return L;
}

static int check_backward(int B, int S, int hidden, int Hq, int Hkv, int d, const void *qn, const void *kn)
{
    int rc = check_layer(B, S, hidden, Hq, Hkv, d, qn, kn);
    if (rc) return rc;
    if (d != 64 && d != 80 && d != 96 && d != 128)
        return fail(GQA_ERR_UNSUPPORTED, "the backward supports head_dim 64, 80, 96 and 128 (got %d)", d);
    if (Hq / Hkv > 32)
        return fail(GQA_ERR_UNSUPPORTED, "the backward supports groups of up to 32 query heads (got %d)", Hq / Hkv);
    return GQA_OK;
}

// The attention backward from q, k, v: the forward attention (o and lse) is
// recomputed into ws, or, with saved, already there (gqa_attn_forward_train).
static int run_attention_bwd(DeviceState &st, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             const uint16_t *dO, int B, int S, int Hq, int Hkv, int d, int causal, float *dq,
                             float *dk, float *dv, uint8_t *ws, cudaStream_t s, bool saved = false)
{
    const AttnBwdLayout L = attn_bwd_layout(B, S, Hq, d);
    gqa_bf16 *o = (gqa_bf16 *)(ws + L.o);
    float *lse = (float *)(ws + L.lse), *dsum = (float *)(ws + L.dsum);
    int rc = saved ? GQA_OK : run_attention(st, q, k, v, B, S, Hq, Hkv, d, causal, o, s, 0, nullptr, 0, lse, L.ld);
    if (rc) return rc;
    AttnBwdProblem p{q, k, v, o, dO, lse, dsum, L.ld, dq, dk, dv, B, S, Hq, Hkv, d, causal ? 1 : 0};
    cudaError_t ce = launch_attention_backward(p, st.err, s);
    if (ce != cudaSuccess) return cuda_fail(ce, "attention backward launch");
    g_launches += 3;  // D, dK/dV, dQ
    return GQA_OK;
}

size_t gqa_attention_backward_workspace_size(int B, int S, int Hq, int head_dim)
{
    if (B <= 0 || S <= 0 || Hq <= 0 || head_dim <= 0) return 0;
    return attn_bwd_layout(B, S, Hq, head_dim).total;
}

int gqa_attention_backward(const gqa_f16 *q, const gqa_f16 *k, const gqa_f16 *v, const gqa_f16 *dO, int B, int S,
                           int Hq, int Hkv, int head_dim, int causal, float *dq, float *dk, float *dv,
                           void *workspace, size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_backward(B, S, 8, Hq, Hkv, head_dim, nullptr, nullptr);
    if (rc) return rc;
    if (!q || !k || !v || !dO || !dq || !dk || !dv) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    const size_t need = attn_bwd_layout(B, S, Hq, head_dim).total;
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    return run_attention_bwd(*st, q, k, v, dO, B, S, Hq, Hkv, head_dim, causal, dq, dk, dv, (uint8_t *)workspace,
                             (cudaStream_t)stream);
}

// Layer backward workspace: the forward's q, k, v (binary16, head-major) and
// pre-norm Q/K rows (fp32), dO (binary16, head-major), the attention-input
// gradients (fp32), dqkv (bf16), then the attention backward's own part.
struct LayerBwdLayout {
    size_t q, k, v, pre, dO, dq, dk, dv, dqkv, norm, attn, total;
};

static LayerBwdLayout layer_bwd_layout(int B, int S, int Hq, int Hkv, int d)
{
    LayerBwdLayout L;
    const size_t M = (size_t)B * S;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    L.q = take(M * Hq * d * 2);
    L.k = take(M * Hkv * d * 2);
    L.v = take(M * Hkv * d * 2);
    L.pre = take(M * (Hq + Hkv) * d * 4);
    L.dO = take(M * Hq * d * 2);
    L.dq = take(M * Hq * d * 4);
    L.dk = take(M * Hkv * d * 4);
    L.dv = take(M * Hkv * d * 4);
    L.dqkv = take(M * (Hq + 2 * Hkv) * d * 2);
    L.norm = take(2 * d * 4);
    L.attn = take(attn_bwd_layout(B, S, Hq, d).total);
    L.total = off;
    return L;
}

size_t gqa_attn_backward_workspace_size(int B, int S, int hidden, int Hq, int Hkv, int head_dim)
{
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0) return 0;
    return layer_bwd_layout(B, S, Hq, Hkv, head_dim).total;
}

// The layer backward; saved: the forward's Q, K, V, pre-norm rows, O and lse
// are already in the workspace (gqa_attn_forward_train), so nothing is recomputed.
static int layer_backward(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                          const gqa_bf16 *k_norm_w, float rope_theta, float eps, int rd, int B, int S, int hidden,
                          int Hq, int Hkv, int head_dim, int causal, const gqa_bf16 *dout, gqa_bf16 *dx,
                          float *dWqkv, float *dWo, float *dq_norm_w, float *dk_norm_w, void *workspace,
                          size_t workspace_bytes, void *stream, bool saved)
{
    g_launches = 0;
    int rc = check_backward(B, S, hidden, Hq, Hkv, head_dim, q_norm_w, k_norm_w);
    if (rc) return rc;
    if ((rc = check_rotary(rd, head_dim))) return rc;
    if (!x || !Wqkv || !Wo || !dout || !dx || !dWqkv || !dWo) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (q_norm_w && (!dq_norm_w || !dk_norm_w))
        return fail(GQA_ERR_ARG, "dq_norm_w and dk_norm_w are required with QK-norm");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(dout) || !aligned16(dx) ||
        !aligned16(dWqkv) || !aligned16(dWo))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    const size_t nx = (size_t)B * S * hidden * 2;
    if (overlap(dx, nx, dout, nx) || overlap(dx, nx, x, nx)) return fail(GQA_ERR_ARG, "dx must not overlap x or dout");
    const LayerBwdLayout L = layer_bwd_layout(B, S, Hq, Hkv, head_dim);
    if (!workspace || workspace_bytes < L.total)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", L.total,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    uint8_t *ws = (uint8_t *)workspace;
    const int d = head_dim, M = B * S, NQ = Hq * d, N = (Hq + 2 * Hkv) * d;
    uint16_t *q = (uint16_t *)(ws + L.q), *k = (uint16_t *)(ws + L.k), *v = (uint16_t *)(ws + L.v);
    uint16_t *dO = (uint16_t *)(ws + L.dO), *dqkv = (uint16_t *)(ws + L.dqkv);
    float *pre = q_norm_w ? (float *)(ws + L.pre) : nullptr;
    float *dq = (float *)(ws + L.dq), *dk = (float *)(ws + L.dk), *dv = (float *)(ws + L.dv);
    float *dqn = dq_norm_w ? dq_norm_w : (float *)(ws + L.norm);
    float *dkn = dk_norm_w ? dk_norm_w : (float *)(ws + L.norm) + d;
    uint8_t *aws = ws + L.attn;
    const gqa_bf16 *o = (const gqa_bf16 *)(aws + attn_bwd_layout(B, S, Hq, d).o);
    cudaStream_t s = (cudaStream_t)stream;
    // 1. the forward's Q, K, V (binary16) and pre-norm rows
    if (!saved && (rc = run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rd, B, S, hidden, Hq, Hkv, d,
                                nullptr, S, S, S, 1, 1, q, k, v, s, 0, 1.0f, 1.0f, pre)))
        return rc;
    // 2. dO = dout Wo, head-major binary16
    {
        GemmProblem p{dout, Wo, M, NQ, hidden};
        GemmOut go{};
        go.head = HeadEpilogue{dO, S, Hq, d};
        cudaError_t ce = launch_gemm_general(p, 0, 1, GEMM_OUT_HEAD16, go, st->err, st->num_sms, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "dO = dout Wo launch");
        ++g_launches;
    }
    // 3. attention backward (forward recomputed for o and lse unless saved)
    if ((rc = run_attention_bwd(*st, q, k, v, dO, B, S, Hq, Hkv, d, causal, dq, dk, dv, aws, s, saved))) return rc;
    // 4. inverse RoPE and the QK-norm gradient -> dqkv
    {
        const float2 *rope = nullptr;
        if (rd > 0) {
            std::lock_guard<std::mutex> lk(g_mu);
            rc = rope_table(*st, (double)rope_theta, rd, S, &rope);
        }
        if (rc) return rc;
        cudaError_t ce = cudaMemsetAsync(dqn, 0, d * sizeof(float), s);
        if (ce == cudaSuccess) ce = cudaMemsetAsync(dkn, 0, d * sizeof(float), s);
        if (ce != cudaSuccess) return cuda_fail(ce, "cudaMemsetAsync(norm-weight gradients)");
        RopeNormBwd rp{dq, dk, dv, pre, rope, q_norm_w, k_norm_w, eps, dqkv, dqn, dkn, M, S, N, Hq, Hkv, d, rd};
        ce = launch_rope_norm_bwd(rp, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "RoPE / QK-norm backward launch");
        ++g_launches;
    }
    // 5. dx = dout + dqkv Wqkv
    {
        GemmProblem p{dqkv, Wqkv, M, hidden, N};
        GemmOut go{};
        go.res = ResidualEpilogue{dout, dx};
        cudaError_t ce = launch_gemm_general(p, 0, 1, GEMM_OUT_RESIDUAL, go, st->err, st->num_sms, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "dx launch");
        ++g_launches;
    }
    // 6. dWqkv = dqkv^T x;  7. dWo = dout^T attn
    {
        GemmProblem p{dqkv, x, N, hidden, M};
        GemmOut go{};
        go.f32 = dWqkv;
        cudaError_t ce = launch_gemm_general(p, 1, 1, GEMM_OUT_F32, go, st->err, st->num_sms, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "dWqkv launch");
        ++g_launches;
    }
    {
        GemmProblem p{dout, o, hidden, NQ, M};
        GemmOut go{};
        go.f32 = dWo;
        cudaError_t ce = launch_gemm_general(p, 1, 1, GEMM_OUT_F32, go, st->err, st->num_sms, s);
        if (ce != cudaSuccess) return cuda_fail(ce, "dWo launch");
        ++g_launches;
    }
    return GQA_OK;
}

int gqa_attn_backward_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                         const gqa_bf16 *k_norm_w, float rope_theta, float eps, int rotary_dim, int B, int S,
                         int hidden, int Hq, int Hkv, int head_dim, int causal, const gqa_bf16 *dout, gqa_bf16 *dx,
                         float *dWqkv, float *dWo, float *dq_norm_w, float *dk_norm_w, void *workspace,
                         size_t workspace_bytes, void *stream)
{
    return layer_backward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv,
                          head_dim, causal, dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, workspace_bytes,
                          stream, false);
}

int gqa_attn_backward(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                      const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int S, int hidden, int Hq,
                      int Hkv, int head_dim, int causal, const gqa_bf16 *dout, gqa_bf16 *dx, float *dWqkv,
                      float *dWo, float *dq_norm_w, float *dk_norm_w, void *workspace, size_t workspace_bytes,
                      void *stream)
{
    return layer_backward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, S, hidden, Hq, Hkv, head_dim,
                          causal, dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, workspace_bytes, stream,
                          false);
}

int gqa_attn_backward_saved_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                               const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w, float rope_theta, float eps,
                               int rotary_dim, int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                               const gqa_bf16 *dout, gqa_bf16 *dx, float *dWqkv, float *dWo, float *dq_norm_w,
                               float *dk_norm_w, void *workspace, size_t workspace_bytes, void *stream)
{
    return layer_backward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv,
                          head_dim, causal, dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, workspace_bytes,
                          stream, true);
}

int gqa_attn_backward_saved(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                            const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int S, int hidden, int Hq,
                            int Hkv, int head_dim, int causal, const gqa_bf16 *dout, gqa_bf16 *dx, float *dWqkv,
                            float *dWo, float *dq_norm_w, float *dk_norm_w, void *workspace, size_t workspace_bytes,
                            void *stream)
{
    return layer_backward(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, S, hidden, Hq, Hkv, head_dim,
                          causal, dout, dx, dWqkv, dWo, dq_norm_w, dk_norm_w, workspace, workspace_bytes, stream,
                          true);
}

int gqa_attn_forward_train(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                           const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int S, int hidden, int Hq,
                           int Hkv, int head_dim, int causal, gqa_bf16 *out, void *workspace, size_t workspace_bytes,
                           void *stream)
{
    return gqa_attn_forward_train_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, S, hidden, Hq, Hkv,
                                     head_dim, causal, out, workspace, workspace_bytes, stream);
}

int gqa_attn_forward_train_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                              const gqa_bf16 *k_norm_w, float rope_theta, float eps, int rotary_dim, int B, int S,
                              int hidden, int Hq, int Hkv, int head_dim, int causal, gqa_bf16 *out, void *workspace,
                              size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_backward(B, S, hidden, Hq, Hkv, head_dim, q_norm_w, k_norm_w);
    if (rc) return rc;
    if ((rc = check_rotary(rotary_dim, head_dim))) return rc;
    if (!x || !Wqkv || !Wo || !out) return fail(GQA_ERR_ARG, "null tensor pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    const size_t nx = (size_t)B * S * hidden * 2;
    const size_t nw = (size_t)(Hq + 2 * Hkv) * head_dim * hidden * 2, no = (size_t)hidden * Hq * head_dim * 2;
    if (overlap(out, nx, x, nx) || overlap(out, nx, Wqkv, nw) || overlap(out, nx, Wo, no))
        return fail(GQA_ERR_ARG, "out must not overlap x or the weights");
    const LayerBwdLayout L = layer_bwd_layout(B, S, Hq, Hkv, head_dim);
    if (!workspace || workspace_bytes < L.total)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", L.total,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    if (overlap(workspace, L.total, out, nx) || overlap(workspace, L.total, x, nx))
        return fail(GQA_ERR_ARG, "workspace must not overlap the arguments");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    uint8_t *ws = (uint8_t *)workspace;
    const int d = head_dim;
    uint16_t *q = (uint16_t *)(ws + L.q), *k = (uint16_t *)(ws + L.k), *v = (uint16_t *)(ws + L.v);
    float *pre = q_norm_w ? (float *)(ws + L.pre) : nullptr;
    const AttnBwdLayout A = attn_bwd_layout(B, S, Hq, d);
    gqa_bf16 *o = (gqa_bf16 *)(ws + L.attn + A.o);
    float *lse = (float *)(ws + L.attn + A.lse);
    cudaStream_t s = (cudaStream_t)stream;
    // the backward's inputs, written where gqa_attn_backward_saved reads them
    if ((rc = run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, d, nullptr,
                      S, S, S, 1, 1, q, k, v, s, 0, 1.0f, 1.0f, pre)))
        return rc;
    if ((rc = run_attention(*st, q, k, v, B, S, Hq, Hkv, d, causal, o, s, 0, nullptr, 0, lse, A.ld, 1))) return rc;
    return run_oproj(*st, o, Wo, x, B * S, hidden, Hq * d, out, s, 1);
}

// ------------------------------------------------------------------ decode

static size_t decode_layout(int B, int Hq, int Hkv, int d, int Lmax, int num_sms, size_t *off_attn,
                            size_t *off_part, int *splits)
{
    const int sp = decode_choose_splits(B, Hkv, Lmax, num_sms);
    const size_t q = align256((size_t)B * Hq * d * 2);
    const size_t a = align256((size_t)B * Hq * d * 2);
    const size_t p = align256(decode_partials_floats(B, Hq, sp, d) * 4);
    if (off_attn) *off_attn = q;
    if (off_part) *off_part = q + a;
    if (splits) *splits = sp;
    return q + a + p;
}

static int num_sms_current()
{
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

size_t gqa_decode_attention_workspace_size(int B, int Hq, int Hkv, int head_dim, int Lmax)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0 || Lmax <= 0) return 0;
    const int sp = decode_choose_splits(B, Hkv, Lmax, num_sms_current());
    return align256(decode_partials_floats(B, Hq, sp, head_dim) * 4);
}

size_t gqa_attn_decode_workspace_size(int B, int hidden, int Hq, int Hkv, int head_dim, int Lmax)
{
    if (B <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0 || Lmax <= 0) return 0;
    return decode_layout(B, Hq, Hkv, head_dim, Lmax, num_sms_current(), nullptr, nullptr, nullptr);
}

static int check_decode(int B, int hidden, int Hq, int Hkv, int d, int Lmax, const void *qn, const void *kn)
{
    int rc = check_layer(B, 1, hidden, Hq, Hkv, d, qn, kn);
    if (rc) return rc;
    if (Lmax <= 0) return fail(GQA_ERR_ARG, "Lmax must be positive");
    if (d != 64 && d != 80 && d != 96 && d != 128 && d != 256)
        return fail(GQA_ERR_UNSUPPORTED, "decode supports head_dim 64, 80, 96, 128 and 256 (got %d)", d);
    const int G = Hq / Hkv;
    if (G > 128) return fail(GQA_ERR_UNSUPPORTED, "unsupported decode group size Hq/Hkv=%d (at most 128)", G);
    if ((long long)B * Hkv * Lmax * d > (1LL << 40)) return fail(GQA_ERR_UNSUPPORTED, "cache too large");
    return GQA_OK;
}

int gqa_decode_qkv_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                   float rope_theta, float eps, int rotary_dim, int B, int hidden, int Hq, int Hkv, int head_dim,
                   gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax, gqa_f16 *q_out, void *stream)
{
    g_launches = 0;
    int rc = check_decode(B, hidden, Hq, Hkv, head_dim, Lmax, q_norm_w, k_norm_w);
    if (rc) return rc;
    if (!x || !Wqkv || !k_cache || !v_cache || !cache_len || !q_out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q_out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    if ((rc = check_rotary(rotary_dim, head_dim))) return rc;
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    return run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, 1, hidden, Hq, Hkv, head_dim,
                   cache_len, 1, Lmax, Lmax, 1, 0, q_out, k_cache, v_cache, (cudaStream_t)stream);
}

int gqa_decode_attention(const gqa_f16 *q, const gqa_bf16 *k_cache, const gqa_bf16 *v_cache, const int *kv_len,
                         int B, int Hq, int Hkv, int head_dim, int Lmax, gqa_bf16 *attn_out, void *workspace,
                         size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_decode(B, 8, Hq, Hkv, head_dim, Lmax, nullptr, nullptr);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !kv_len || !attn_out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(attn_out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    const int sp = decode_choose_splits(B, Hkv, Lmax, st->num_sms);
    const size_t need = align256(decode_partials_floats(B, Hq, sp, head_dim) * 4);
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (!aligned16(workspace)) return fail(GQA_ERR_ARG, "workspace must be 16-byte aligned");
    return run_decode_attn(*st, q, k_cache, v_cache, kv_len, 0, B, Hq, Hkv, head_dim, Lmax, attn_out,
                           (float *)workspace, sp, (cudaStream_t)stream);
}

int gqa_attn_decode_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                    const gqa_bf16 *k_norm_w, float rope_theta, float eps, int rotary_dim, int B, int hidden, int Hq,
                    int Hkv, int head_dim, gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                    gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_decode(B, hidden, Hq, Hkv, head_dim, Lmax, q_norm_w, k_norm_w);
    if (rc) return rc;
    if (!x || !Wqkv || !Wo || !k_cache || !v_cache || !cache_len || !out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    if ((rc = check_rotary(rotary_dim, head_dim))) return rc;
    if (overlap(out, (size_t)B * hidden * 2, x, (size_t)B * hidden * 2))
        return fail(GQA_ERR_ARG, "out must not overlap x");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    size_t off_attn, off_part;
    int sp;
    const size_t need = decode_layout(B, Hq, Hkv, head_dim, Lmax, st->num_sms, &off_attn, &off_part, &sp);
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    uint8_t *ws = (uint8_t *)workspace;
    gqa_f16 *q = (gqa_f16 *)ws;  // binary16 q of the new tokens
    gqa_bf16 *attn = (gqa_bf16 *)(ws + off_attn);
    float *part = (float *)(ws + off_part);
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, 1, hidden, Hq, Hkv, head_dim,
                      cache_len, 1, Lmax, Lmax, 1, 0, q, k_cache, v_cache, s)))
        return rc;
    if ((rc = run_decode_attn(*st, q, k_cache, v_cache, cache_len, 1, B, Hq, Hkv, head_dim, Lmax, attn, part, sp, s, 0,
                              1.0f, 1.0f, 1)))
        return rc;
    return run_oproj(*st, attn, Wo, x, B, hidden, Hq * head_dim, out, s, 1);
}

// ------------------------------------------------------ prefill into a cache

// Workspace of the cached prefill: Q (bf16), attn (bf16), and for the
// attention's key splits (kCachedSplits at most) their binary16 partial
// outputs and fp32 log2-sum-exp rows; then the binary16 copies of the two
// caches that the attention reads ([B, Hkv, Lmax, d] each).
static constexpr int kCachedSplits = 2;
struct CachedLayout {
    size_t q, attn, part_o, part_lse, k16, v16, total;
};
static size_t widened_bytes(int B, int Hkv, int d, int Lmax) { return align256((size_t)B * Hkv * Lmax * d * 2); }
static CachedLayout cached_layout(int B, int S, int Hq, int Hkv, int d, int Lmax)
{
    CachedLayout L;
    const size_t n = align256((size_t)B * S * Hq * d * 2);
    L.q = 0;
    L.attn = n;
    L.part_o = 2 * n;
    L.part_lse = L.part_o + kCachedSplits * n;
    L.k16 = L.part_lse + align256((size_t)kCachedSplits * B * Hq * S * 4);
    L.v16 = L.k16 + widened_bytes(B, Hkv, d, Lmax);
    L.total = L.v16 + widened_bytes(B, Hkv, d, Lmax);
    return L;
}

size_t gqa_attn_prefill_cached_workspace_size(int B, int S, int Hq, int Hkv, int head_dim, int Lmax)
{
    if (B <= 0 || S <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0 || Lmax <= 0) return 0;
    return cached_layout(B, S, Hq, Hkv, head_dim, Lmax).total;
}

size_t gqa_attention_cached_workspace_size(int B, int Hkv, int head_dim, int Lmax)
{
    if (B <= 0 || Hkv <= 0 || head_dim <= 0 || Lmax <= 0) return 0;
    return 2 * widened_bytes(B, Hkv, head_dim, Lmax);
}

// Key splits for the cached prefill's attention.  Its work items (sequence,
// KV head, block of 256/G query positions: B*Hq*S/256 of them) all see the
// whole cache, so they are about equally long, and below eight waves of the
// GPU the last, partly filled wave leaves many SMs idle; splitting every
// item's keys in two halves that idle share.
static int cached_splits(int B, int S, int Hq, int num_sms)
{
    const long long items = ((long long)B * Hq * S + 255) / 256;
    return items < 8LL * num_sms ? kCachedSplits : 1;
}

static int check_cached(int B, int S, int hidden, int Hq, int Hkv, int d, int Lmax, const void *qn, const void *kn)
{
    int rc = check_layer(B, S, hidden, Hq, Hkv, d, qn, kn);
    if (rc) return rc;
    if ((rc = check_group(Hq, Hkv))) return rc;
    if (Lmax < S) return fail(GQA_ERR_ARG, "Lmax=%d is smaller than the %d new tokens", Lmax, S);
    if ((long long)B * Hkv * Lmax * d > (1LL << 40)) return fail(GQA_ERR_UNSUPPORTED, "cache too large");
    return GQA_OK;
}

// Binary16 copies of cache rows [0, cache_len[b] + S) into k16 / v16, the keys
// and values the cached attention reads.
static int run_widen(DeviceState &st, const gqa_bf16 *k_cache, const gqa_bf16 *v_cache, uint16_t *k16,
                     uint16_t *v16, const int *cache_len, int B, int S, int Hkv, int d, int Lmax, cudaStream_t stream,
                     int pdl)
{
    CacheWiden w{k_cache, v_cache, k16, v16, cache_len, B, S, Hkv, Lmax, d, 128, pdl};  // key tiles of 128
    cudaError_t ce = launch_cache_widen(w, st.err, stream);
    if (ce != cudaSuccess) return cuda_fail(ce, "cache widening launch");
    ++g_launches;
    return GQA_OK;
}

int gqa_attention_cached(const gqa_f16 *q, const gqa_bf16 *k_cache, const gqa_bf16 *v_cache, const int *cache_len,
                         int B, int S, int Hq, int Hkv, int head_dim, int Lmax, int causal, gqa_bf16 *attn_out,
                         void *workspace, size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_cached(B, S, 8, Hq, Hkv, head_dim, Lmax, nullptr, nullptr);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !cache_len || !attn_out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(attn_out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    const size_t need = gqa_attention_cached_workspace_size(B, Hkv, head_dim, Lmax);
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    uint16_t *k16 = (uint16_t *)workspace, *v16 = k16 + widened_bytes(B, Hkv, head_dim, Lmax) / 2;
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = run_widen(*st, k_cache, v_cache, k16, v16, cache_len, B, S, Hkv, head_dim, Lmax, s, 0))) return rc;
    return run_attention(*st, q, k16, v16, B, S, Hq, Hkv, head_dim, causal, attn_out, s, Lmax, cache_len, 1, nullptr,
                         0, 1);
}

int gqa_attn_prefill_cached_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                            const gqa_bf16 *k_norm_w, float rope_theta, float eps, int rotary_dim, int B, int S,
                            int hidden, int Hq, int Hkv, int head_dim, int causal, gqa_bf16 *k_cache, gqa_bf16 *v_cache,
                            const int *cache_len, int Lmax, gqa_bf16 *out, void *workspace, size_t workspace_bytes,
                            void *stream)
{
    g_launches = 0;
    int rc = check_cached(B, S, hidden, Hq, Hkv, head_dim, Lmax, q_norm_w, k_norm_w);
    if (rc) return rc;
    if (!x || !Wqkv || !Wo || !k_cache || !v_cache || !cache_len || !out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    if ((rc = check_rotary(rotary_dim, head_dim))) return rc;
    const size_t nx = (size_t)B * S * hidden * 2;
    if (overlap(out, nx, x, nx)) return fail(GQA_ERR_ARG, "out must not overlap x");
    const size_t need = gqa_attn_prefill_cached_workspace_size(B, S, Hq, Hkv, head_dim, Lmax);
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    uint8_t *ws = (uint8_t *)workspace;
    const CachedLayout CL = cached_layout(B, S, Hq, Hkv, head_dim, Lmax);
    gqa_f16 *q = (gqa_f16 *)(ws + CL.q);  // binary16; the attention widens the bf16 cache tiles to match
    gqa_bf16 *attn = (gqa_bf16 *)(ws + CL.attn);
    const int splits = cached_splits(B, S, Hq, st->num_sms);
    cudaStream_t s = (cudaStream_t)stream;
    // K/V of the new tokens go straight into the cache at slots cache_len[b] + t
    if ((rc = run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, rotary_dim, B, S, hidden, Hq, Hkv, head_dim,
                      cache_len, S, Lmax, Lmax, 1, 0, q, k_cache, v_cache, s)))
        return rc;
    uint16_t *k16 = (uint16_t *)(ws + CL.k16), *v16 = (uint16_t *)(ws + CL.v16);
    if ((rc = run_widen(*st, k_cache, v_cache, k16, v16, cache_len, B, S, Hkv, head_dim, Lmax, s, 1))) return rc;
    if ((rc = run_attention(*st, q, k16, v16, B, S, Hq, Hkv, head_dim, causal, attn, s, Lmax, cache_len, 1, nullptr,
                            0, 1, splits, (uint16_t *)(ws + CL.part_o), (float *)(ws + CL.part_lse))))
        return rc;
    return run_oproj(*st, attn, Wo, x, B * S, hidden, Hq * head_dim, out, s, 1);
}

// ------------------------------------------------------ FP8 (E4M3) KV cache

static int check_fp8(int d, float k_scale, float v_scale)
{
    if (!(k_scale > 0.0f) || !(v_scale > 0.0f) || !isfinite(k_scale) || !isfinite(v_scale))
        return fail(GQA_ERR_ARG, "k_scale and v_scale must be finite and > 0");
    if (d != 64 && d != 80 && d != 96 && d != 128 && d != 256)
        return fail(GQA_ERR_UNSUPPORTED, "unsupported head_dim for E4M3 caches: %d (supported: 64, 80, 96, 128, 256)",
                    d);
    return GQA_OK;
}

int gqa_decode_attention_fp8(const gqa_f16 *q, const gqa_e4m3 *k_cache, const gqa_e4m3 *v_cache, float k_scale,
                             float v_scale, const int *kv_len, int B, int Hq, int Hkv, int head_dim, int Lmax,
                             gqa_bf16 *attn_out, void *workspace, size_t workspace_bytes, void *stream)
{
    g_launches = 0;
    int rc = check_decode(B, 8, Hq, Hkv, head_dim, Lmax, nullptr, nullptr);
    if (rc) return rc;
    if ((rc = check_fp8(head_dim, k_scale, v_scale))) return rc;
    if (!q || !k_cache || !v_cache || !kv_len || !attn_out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(attn_out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    const int sp = decode_choose_splits(B, Hkv, Lmax, st->num_sms);
    const size_t need = align256(decode_partials_floats(B, Hq, sp, head_dim) * 4);
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (!aligned16(workspace)) return fail(GQA_ERR_ARG, "workspace must be 16-byte aligned");
    return run_decode_attn(*st, q, k_cache, v_cache, kv_len, 0, B, Hq, Hkv, head_dim, Lmax, attn_out,
                           (float *)workspace, sp, (cudaStream_t)stream, 1, k_scale, v_scale);
}

int gqa_decode_qkv_fp8(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                       float rope_theta, float eps, int B, int hidden, int Hq, int Hkv, int head_dim,
                       gqa_e4m3 *k_cache, gqa_e4m3 *v_cache, float k_scale, float v_scale, const int *cache_len,
                       int Lmax, gqa_f16 *q_out, void *stream)
{
    g_launches = 0;
    int rc = check_decode(B, hidden, Hq, Hkv, head_dim, Lmax, q_norm_w, k_norm_w);
    if (rc) return rc;
    if ((rc = check_fp8(head_dim, k_scale, v_scale))) return rc;
    if (!x || !Wqkv || !k_cache || !v_cache || !cache_len || !q_out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q_out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    return run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, 1, hidden, Hq, Hkv, head_dim,
                   cache_len, 1, Lmax, Lmax, 1, 0, q_out, (uint16_t *)k_cache, (uint16_t *)v_cache,
                   (cudaStream_t)stream, 1, k_scale, v_scale);
}

int gqa_attn_decode_fp8(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                        const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int hidden, int Hq, int Hkv,
                        int head_dim, gqa_e4m3 *k_cache, gqa_e4m3 *v_cache, float k_scale, float v_scale,
                        const int *cache_len, int Lmax, gqa_bf16 *out, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    g_launches = 0;
    int rc = check_decode(B, hidden, Hq, Hkv, head_dim, Lmax, q_norm_w, k_norm_w);
    if (rc) return rc;
    if ((rc = check_fp8(head_dim, k_scale, v_scale))) return rc;
    if (!x || !Wqkv || !Wo || !k_cache || !v_cache || !cache_len || !out) return fail(GQA_ERR_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(Wo) || !aligned16(k_cache) || !aligned16(v_cache) ||
        !aligned16(out))
        return fail(GQA_ERR_ARG, "tensor pointers must be 16-byte aligned");
    if (!(rope_theta > 0.0f) || !(eps >= 0.0f)) return fail(GQA_ERR_ARG, "rope_theta must be > 0 and eps >= 0");
    if (overlap(out, (size_t)B * hidden * 2, x, (size_t)B * hidden * 2))
        return fail(GQA_ERR_ARG, "out must not overlap x");
    DeviceState *st;
    if ((rc = device_state(&st))) return rc;
    size_t off_attn, off_part;
    int sp;
    const size_t need = decode_layout(B, Hq, Hkv, head_dim, Lmax, st->num_sms, &off_attn, &off_part, &sp);
    if (!workspace || workspace_bytes < need)
        return fail(GQA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                    workspace ? workspace_bytes : (size_t)0);
    if (((uintptr_t)workspace & 255u) != 0) return fail(GQA_ERR_ARG, "workspace must be 256-byte aligned");
    uint8_t *ws = (uint8_t *)workspace;
    gqa_f16 *q = (gqa_f16 *)ws;
    gqa_bf16 *attn = (gqa_bf16 *)(ws + off_attn);
    float *part = (float *)(ws + off_part);
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = run_qkv(*st, x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, 1, hidden, Hq, Hkv, head_dim,
                      cache_len, 1, Lmax, Lmax, 1, 0, q, (uint16_t *)k_cache, (uint16_t *)v_cache, s, 1, k_scale,
                      v_scale)))
        return rc;
    if ((rc = run_decode_attn(*st, q, k_cache, v_cache, cache_len, 1, B, Hq, Hkv, head_dim, Lmax, attn, part, sp, s,
                              1, k_scale, v_scale, 1)))
        return rc;
    return run_oproj(*st, attn, Wo, x, B, hidden, Hq * head_dim, out, s, 1);
}

// ------------------------------------------- full rotary (rotary_dim = head_dim)

int gqa_qkv_proj(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                 float rope_theta, float eps, int B, int S, int hidden, int Hq, int Hkv, int head_dim, gqa_f16 *q_out,
                 gqa_f16 *k_out, gqa_f16 *v_out, void *stream)
{
    return gqa_qkv_proj_rd(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, S, hidden, Hq, Hkv, head_dim,
                           q_out, k_out, v_out, stream);
}

int gqa_attn_forward_ex(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                        const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int S, int hidden, int Hq,
                        int Hkv, int head_dim, int causal, gqa_bf16 *out, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    return gqa_attn_forward_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, S, hidden, Hq, Hkv,
                               head_dim, causal, out, workspace, workspace_bytes, stream);
}

int gqa_decode_qkv(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                   float rope_theta, float eps, int B, int hidden, int Hq, int Hkv, int head_dim, gqa_bf16 *k_cache,
                   gqa_bf16 *v_cache, const int *cache_len, int Lmax, gqa_f16 *q_out, void *stream)
{
    return gqa_decode_qkv_rd(x, Wqkv, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, hidden, Hq, Hkv, head_dim,
                             k_cache, v_cache, cache_len, Lmax, q_out, stream);
}

int gqa_attn_decode(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                    const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int hidden, int Hq, int Hkv,
                    int head_dim, gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                    gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream)
{
    return gqa_attn_decode_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, hidden, Hq, Hkv, head_dim,
                              k_cache, v_cache, cache_len, Lmax, out, workspace, workspace_bytes, stream);
}

int gqa_attn_prefill_cached(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo, const gqa_bf16 *q_norm_w,
                            const gqa_bf16 *k_norm_w, float rope_theta, float eps, int B, int S, int hidden, int Hq,
                            int Hkv, int head_dim, int causal, gqa_bf16 *k_cache, gqa_bf16 *v_cache,
                            const int *cache_len, int Lmax, gqa_bf16 *out, void *workspace, size_t workspace_bytes,
                            void *stream)
{
    return gqa_attn_prefill_cached_rd(x, Wqkv, Wo, q_norm_w, k_norm_w, rope_theta, eps, head_dim, B, S, hidden, Hq, Hkv,
                                      head_dim, causal, k_cache, v_cache, cache_len, Lmax, out, workspace,
                                      workspace_bytes, stream);
}

// ---------------------------------------------------------------- accounting

int gqa_attn_cost(int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal, long long *weights,
                  long long *proj_macs_per_token, long long *attn_macs, long long *flops)
{
    if (B <= 0 || S <= 0 || hidden <= 0 || Hq <= 0 || Hkv <= 0 || head_dim <= 0)
        return fail(GQA_ERR_ARG, "sizes must be positive");
    const long long h = hidden, d = head_dim;
    const long long w = h * (Hq + 2LL * Hkv) * d + (long long)Hq * d * h;
    const long long pairs = causal ? (long long)S * (S + 1) / 2 : (long long)S * S;
    const long long am = 2LL * d * Hq * pairs * B;
    if (weights) *weights = w;
    if (proj_macs_per_token) *proj_macs_per_token = w;
    if (attn_macs) *attn_macs = am;
    if (flops) *flops = 2LL * ((long long)B * S * w + am);
    return GQA_OK;
}

// --------------------------------------------------------------- diagnostics

// The status an error word reports (the worst of its bits first).
static int error_word_status(unsigned word)
{
    if (word & kErrTimeout) return fail(GQA_ERR_TIMEOUT, "a bounded device wait gave up (error word 0x%x)", word);
    if (word & kErrIndex) return fail(GQA_ERR_ARG, "a device-side index check failed (error word 0x%x)", word);
    if (word & kErrRange)
        return fail(GQA_ERR_RANGE, "a Q/K/V value beyond the binary16 range was clamped (error word 0x%x)", word);
    return GQA_OK;
}

int gqa_check_device_error(void)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(GQA_ERR_CUDA, "device index %d out of range", dev);
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    bool have_state;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        have_state = g_dev[dev].init;
    }
    // Without per-device state no kernel of the workspace-taking entry points
    // has run on this device, so its word is not read (nor set up: a caller of
    // gqa_decode_attention_noalloc alone gets this check without an allocation).
    unsigned word = 0;
    if (have_state) {
        DeviceState &st = g_dev[dev];
        e = cudaMemcpy(&word, st.err, sizeof word, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(error word)");
        if (word) {
            e = cudaMemset(st.err, 0, sizeof word);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
        }
    }
    word |= noalloc_take_error_word(dev);
    return error_word_status(word);
}

int gqa_check_stream_error(void *stream)
{
    const cudaStream_t s = (cudaStream_t)stream;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(GQA_ERR_CUDA, "device index %d out of range", dev);
    bool have_state;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        have_state = g_dev[dev].init;
    }
    unsigned word = 0;
    if (have_state) {
        DeviceState &st = g_dev[dev];
        // after the stream's queued work; the stream alone is waited for
        if ((e = cudaMemcpyAsync(&word, st.err, sizeof word, cudaMemcpyDeviceToHost, s)) != cudaSuccess ||
            (e = cudaStreamSynchronize(s)) != cudaSuccess)
            return cuda_fail(e, "reading the error word on the stream");
        if (word && (e = cudaMemsetAsync(st.err, 0, sizeof word, s)) != cudaSuccess)
            return cuda_fail(e, "clearing the error word on the stream");
    }
    word |= noalloc_take_error_word(dev, s, true);
    return error_word_status(word);
}

int gqa_selftest_bounded_wait(int limit_ms)
{
    if (limit_ms < 1 || limit_ms > 5000) return fail(GQA_ERR_ARG, "limit_ms must be in [1, 5000]");
    DeviceState *st;
    int rc = device_state(&st);
    if (rc) return rc;
    if ((rc = gqa_check_device_error())) return rc;  // start from a clean word
    cudaError_t e = launch_selftest_wait(st->err, (unsigned long long)limit_ms * 1000000ull, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return gqa_check_device_error();
}

}  // extern "C"

namespace gqa {

int check_decode_attention_args(int B, int Hq, int Hkv, int d, int Lmax)
{
    return check_decode(B, 8, Hq, Hkv, d, Lmax, nullptr, nullptr);
}

}  // namespace gqa
