// internal.h -- host-side declarations shared by the library's translation
// units (launchers and their argument blocks).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gqa {

// ---------------------------------------------------------------- GEMM core
// C[M, N] = A[M, K] @ B[N, K]^T on tcgen05, A and B bf16 row-major (K
// contiguous), fp32 accumulation in TMEM, with one of two fused epilogues.

// Epilogue "qkv": the N columns are Hq query heads, then Hkv key heads, then
// Hkv value heads, each d wide.  Q and K heads are RMS-normed (optional) and
// rotated (RoPE) at the row's position; results are written head-major.
struct QkvEpilogue {
    int Hq, Hkv, d;
    int S;                 // tokens per sequence (row m0 + m = b*S + t)
    int m0;                // rows of the whole problem before this GEMM's row 0 (token chunks; pos_dev NULL only)
    const int *pos_dev;    // cached: position = K/V slot = pos_dev[b] + t; NULL: position t
    int q_seq;             // sequence extent of q_out (S, or 1 for decode)
    int kv_seq;            // sequence extent of k_out / v_out (S, or Lmax for decode)
    const uint16_t *q_norm_w, *k_norm_w;  // [d] bf16, or both NULL
    float eps;
    int rd;                // rotary width: d, d/2, d/4 or 0 (RoPE on features [0, rd))
    const float4 *rope;    // [rd/4][rope_ld] quads: (cos, cos, sin, sin) of pos * theta^(-2i/rd) for pairs
                           // i = 2k, 2k + 1 at entry [k][pos]; NULL when rd = 0
    int rope_ld;           // positions per quad row of rope (>= rope_rows)
    int rope_rows;         // positions the table covers
    int q_f16;             // 1: Q stored as binary16 (clamped, flagged); 0: bf16
    int kv_f16;            // 1: K and V stored as binary16 (clamped, flagged); 0: bf16
    int kv_fp8;            // 1: K and V stored as E4M3 codes of value / k_scale, value / v_scale
    float k_scale, v_scale;
    float *pre_out;        // non-NULL (with QK-norm): pre-norm Q and K rows, [M, (Hq+Hkv)*d] fp32
    uint16_t *q_out, *k_out, *v_out;
};

// Epilogue "residual": out[m, n] = acc[m, n] + resid[m, n] (bf16, [M, N]).
struct ResidualEpilogue {
    const uint16_t *resid;
    uint16_t *out;
};

// Epilogue "head16": C written head-major in binary16 (the attention
// gradient dO of the backward): column j*d + c of row b*S + t goes to
// out[((b*H + j)*S + t)*d + c].
struct HeadEpilogue {
    uint16_t *out;
    int S, H, d;
};

struct GemmProblem {
    const void *A;  // [M, K] bf16 (stored [K, M] when MN-major)
    const void *B;  // [N, K] bf16 (stored [K, N] when MN-major)
    int M, N, K;
    int pdl = 0;    // launch as the programmatic dependent of the previous kernel (see LaunchCfg)
};

// Output of launch_gemm_general.
enum { GEMM_OUT_F32 = 0, GEMM_OUT_HEAD16 = 1, GEMM_OUT_RESIDUAL = 2 };
struct GemmOut {
    float *f32;             // GEMM_OUT_F32: [M, N]
    HeadEpilogue head;      // GEMM_OUT_HEAD16
    ResidualEpilogue res;   // GEMM_OUT_RESIDUAL: bf16 out = C + resid
};

// Launchers return a cudaError_t (cudaSuccess when enqueued).
cudaError_t launch_gemm_qkv(const GemmProblem &p, const QkvEpilogue &e, unsigned *err, int num_sms,
                            cudaStream_t stream);
cudaError_t launch_gemm_residual(const GemmProblem &p, const ResidualEpilogue &e, unsigned *err, int num_sms,
                                 cudaStream_t stream);
// The backward's products: A and/or B MN-major (a_mn, b_mn), 256-wide tiles.
// Implemented: F32 with both K-major or both MN-major; HEAD16 and RESIDUAL with B
// MN-major.  Other combinations return cudaErrorInvalidValue.
cudaError_t launch_gemm_general(const GemmProblem &p, int a_mn, int b_mn, int epi, const GemmOut &o, unsigned *err,
                                int num_sms, cudaStream_t stream);

// ------------------------------------------------------ KV-cache widening
// Binary16 copies k16 / v16 [B, Hkv, Lmax, d] of the bf16 caches' rows
// [0, cache_len[b] + S), zero-filled up to the next multiple of `tile` keys
// (the attention's key tile); values beyond +-65504 saturate and set
// kErrRange.  Sequences with cache_len[b] + S > Lmax are skipped.
struct CacheWiden {
    const uint16_t *k_cache, *v_cache;
    uint16_t *k16, *v16;
    const int *cache_len;
    int B, S, Hkv, Lmax, d, tile;
    int pdl = 0;
};
cudaError_t launch_cache_widen(const CacheWiden &p, unsigned *err, cudaStream_t stream);

// ------------------------------------------------------- prefill attention
struct AttentionProblem {
    const uint16_t *q;  // [B, Hq, S, d]
    const uint16_t *k;  // [B, Hkv, kv_seq, d]
    const uint16_t *v;  // [B, Hkv, kv_seq, d]
    uint16_t *out;      // [B, S, Hq*d]
    int B, S, Hq, Hkv, d, causal;
    int kv_seq;            // sequence extent of k/v (S, or Lmax for a cache)
    const int *kv_start;   // device [B]: keys already cached before the S queries (NULL: 0)
    int cached;            // 1: queries after kv_start[b] cached keys (k/v: kv_seq rows per head); all binary16
    float *lse;            // non-NULL (plain prefill only): per (b, head, t) log2-sum-exp of the
                           // scaled scores, at lse[(b*Hq + head)*lse_ld + t]: P = 2^(s*log2(e)/sqrt(d) - lse)
    int lse_ld;
    int pdl = 0;           // launch as the programmatic dependent of the previous kernel
    // cached variant (kv_start): split each query block's keys into kv_splits
    // ranges, partials in part_o [kv_splits][B, S, Hq*d] binary16 and part_lse
    // [kv_splits][B*Hq, S] fp32, merged by a second kernel (1 or NULL buffers: no split)
    int kv_splits = 1;
    uint16_t *part_o = nullptr;
    float *part_lse = nullptr;
};
// Whether launchers may use their 2-CTA-cluster kernels (process-wide, default
// on); off, every problem runs on the one-CTA kernels.
bool cta_pairs_enabled();
int set_cta_pairs(int enable);  // returns the previous setting
cudaError_t launch_attention(const AttentionProblem &p, unsigned *err, int num_sms, cudaStream_t stream);
// Backward of the attention (head_dim 64, 80, 96 or 128, Hq/Hkv <= 32).  q, k, v, dO
// binary16 head-major ([B, H, S, d]); o the forward's bf16 output [B, S,
// Hq*d]; lse the forward's log2-sum-exp and dsum a workspace, both fp32
// [B*Hq, ld] with ld >= S, ld % 4 == 0; dq [B, Hq, S, d], dk/dv [B, Hkv, S, d]
// fp32 (written, not accumulated).
struct AttnBwdProblem {
    const uint16_t *q, *k, *v, *o, *dO;
    const float *lse;
    float *dsum;
    int ld;
    float *dq, *dk, *dv;
    int B, S, Hq, Hkv, d, causal;
};
cudaError_t launch_attention_backward(const AttnBwdProblem &p, unsigned *err, cudaStream_t stream);

// Inverse RoPE and the QK-norm gradient (backward.cu): dq [B, Hq, S, d], dk /
// dv [B, Hkv, S, d] fp32 -> dqkv [M, N] bf16 (N = (Hq + 2 Hkv) d, the fused
// projection's output gradient), with the norm-weight gradients added to
// dq_norm_w / dk_norm_w (fp32 [d], zeroed by the caller).  pre: the forward's
// pre-norm Q and K rows [M, (Hq + Hkv) d] fp32, or NULL without QK-norm.
struct RopeNormBwd {
    const float *dq, *dk, *dv, *pre;
    const float2 *rope;  // [S rows][rd/2] (cos, sin) of the rotary width's angles; NULL when rd = 0
    const uint16_t *q_norm_w, *k_norm_w;
    float eps;
    uint16_t *dqkv;
    float *dq_norm_w, *dk_norm_w;
    int M, S, N, Hq, Hkv, d;
    int rd;              // rotary width (RoPE on features [0, rd))
};
cudaError_t launch_rope_norm_bwd(const RopeNormBwd &p, cudaStream_t stream);
// head_dim 256 (called by launch_attention)
cudaError_t launch_attention256(const AttentionProblem &p, unsigned *err, cudaStream_t stream);

// -------------------------------------------------------- decode attention
struct DecodeAttentionProblem {
    const uint16_t *q;        // [B, Hq, d] binary16
    const void *k_cache;      // [B, Hkv, Lmax, d] bf16, or E4M3 codes when fp8
    const void *v_cache;
    int fp8;                  // caches hold E4M3 codes worth code * k_scale / v_scale
    float k_scale, v_scale;
    const int *len;           // device [B]; keys attended = len[b] + len_bias
    int len_bias;
    uint16_t *out;            // [B, Hq*d]
    int B, Hq, Hkv, d, Lmax;
    float *partials;          // split partials (see decode_partials_floats)
    int splits;               // number of key splits per (b, kv head)
    int pdl;                  // launch the split kernel as the programmatic dependent of the previous kernel
    int vsub;                 // set by the launcher: sub-groups of Hq/Hkv/vsub query heads per KV head
};
// Sub-groups a group of G query heads is taken as when a work item holds at
// most gm of them (the fewest that divide G).
int decode_head_subgroups(int G, int gm);
int decode_choose_splits(int B, int Hkv, int Lmax, int num_sms);
size_t decode_partials_floats(int B, int Hq, int splits, int d);
cudaError_t launch_decode_attention(const DecodeAttentionProblem &p, unsigned *err, cudaStream_t stream);

// --------------------------------------------------------------- self test
cudaError_t launch_selftest_wait(unsigned *err, unsigned long long limit_ns, cudaStream_t stream);

// Sets the message gqa_last_error() returns on the calling thread.
void record_error_message(const char *msg);
// Sets the count gqa_last_launch_count() returns on the calling thread.
void set_launch_count(int n);
// The argument checks of gqa_decode_attention (sizes, group size, head_dim,
// cache size): GQA_OK or the status (with the message recorded) it returns.
int check_decode_attention_args(int B, int Hq, int Hkv, int d, int Lmax);
// Reads and clears the error word of gqa_decode_attention_noalloc on device
// `dev` (0 if that entry point never ran there).  Host-synchronous (call with
// the device idle), or, on_stream, ordered on `stream` and waiting for it
// alone.  Allocates nothing.
unsigned noalloc_take_error_word(int dev, cudaStream_t stream = nullptr, bool on_stream = false);

// Launch configuration for cudaLaunchKernelEx: optional thread-block cluster
// (cluster > 1 CTAs along x) and optional programmatic dependent launch (pdl:
// the kernel may start while the previous kernel in the stream finishes; it
// must call grid_dep_wait before touching that kernel's outputs).  Used in
// place: cfg.attrs points into the object.
struct LaunchCfg {
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl, int cluster = 1)
    {
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        int n = 0;
        if (cluster > 1) {
            attr[n].id = cudaLaunchAttributeClusterDimension;
            attr[n].val.clusterDim.x = (unsigned)cluster;
            attr[n].val.clusterDim.y = 1;
            attr[n].val.clusterDim.z = 1;
            ++n;
        }
        if (pdl) {
            attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        cfg.attrs = attr;
        cfg.numAttrs = (unsigned)n;
    }
    LaunchCfg(const LaunchCfg &) = delete;
    LaunchCfg &operator=(const LaunchCfg &) = delete;
};

// Tensor-map encoder (driver entry point, resolved once); elements of 2 bytes
// (16-bit floats, copied bit for bit), 1 byte (FP8 codes) or 4 bytes (fp32).
CUresult encode_tmap(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box, bool swizzle128, int elem_bytes = 2);

}  // namespace gqa
