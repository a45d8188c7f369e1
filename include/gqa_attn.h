/*
 * gqa_attn.h -- C ABI of the GB300 (sm_103a) grouped-query attention layer.
 *
 * The layer: a fused QKV projection hidden -> (Hq + 2*Hkv)*head_dim,
 * per-head RMSNorm of Q and K (QK-norm), RoPE on Q and K, causal
 * grouped-query attention softmax(Q K^T / sqrt(head_dim)) V where every KV
 * head serves Hq/Hkv query heads, and an output projection Hq*head_dim ->
 * hidden followed by the residual add.  head_dim is an explicit argument,
 * independent of hidden / Hq.
 *
 * Sources (page title, section):
 *   [NeoX] "Support explicit attention head_dim independent of hidden_size /
 *          num_attention_heads": "Background" (projection shapes), "Fused QKV
 *          projection", "Attention output flattening", "Output projection",
 *          "Scaling and RoPE", "Checkpoint conversion" (weight shapes),
 *          "Qwen3-0.6B example" (residual addition, 2 query heads per KV head).
 *   [T07]  "Tutorial 07: Multi-Head and Grouped-Query Attention (Full Layer)":
 *          §3 QK-Norm, §4 the complete layer (steps 1-7), §6 reshape flow.
 *   [Knob] "num_heads Is Not a Capacity Knob": "Why the cost does not move"
 *          (weight and multiply-accumulate counts), "Where the invariance
 *          breaks" (head_dim is a kernel tile dimension).
 *
 * Conventions for every entry point
 *   - Tensors are bf16, passed as pointers to their 16-bit patterns
 *     (gqa_bf16), dense row-major with the shapes given per argument.  Unless
 *     a comment says "host", a pointer is a DEVICE pointer of the current CUDA
 *     device.  The caller owns all memory; the library never frees or keeps
 *     a caller pointer past the call.
 *   - Weights are stored [out_features, in_features] and applied as x @ W^T
 *     ([NeoX] "Checkpoint conversion").  Wqkv stacks, by rows, W_q
 *     [Hq*d, hidden], then W_k [Hkv*d, hidden], then W_v [Hkv*d, hidden].
 *   - Query head j attends with KV head j / (Hq/Hkv).
 *   - RMSNorm(v) = v * w / sqrt(mean(v^2) + eps) over head_dim.  RoPE pairs
 *     element i with i + head_dim/2 at angle pos * theta^(-2i/head_dim)
 *     (the *_rd entry points rotate only the first rotary_dim features).
 *   - `stream` is a cudaStream_t passed as void* (NULL: the legacy default
 *     stream).  Work is enqueued asynchronously; the function returns after
 *     validation and launch.  Outputs are valid once the stream reaches them.
 *   - Status: GQA_OK (0) or a negative GQA_ERR_* code.  Arguments are
 *     validated before anything is launched; a rejected call launches nothing
 *     and writes nothing.  gqa_last_error() returns a message for the last
 *     failing call on the calling thread.
 *   - Supported shapes: hidden a multiple of 8; Hq a multiple of Hkv;
 *     head_dim 64, 80, 96, 128 or 256 for the prefill paths (projection,
 *     attention, layer forward, prefill into a cache) and for decode over
 *     bf16 or E4M3 caches, 64, 80, 96 or 128 for the backward.  Other
 *     head_dim values return GQA_ERR_UNSUPPORTED,
 *     naming the dimension ([Knob] "Where the invariance breaks": head_dim is
 *     a tile dimension of the fused kernels; 80 and 96 run in 128-wide tiles
 *     whose extra columns are zero).
 *   - Device-side waits are bounded.  A wait that runs out records
 *     GQA_ERR_TIMEOUT in a per-device error word that gqa_check_device_error()
 *     reports; the kernel then returns without hanging the GPU.
 */
#ifndef GQA_ATTN_H
#define GQA_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t gqa_bf16; /* bit pattern of one bf16 value */

#define GQA_OK 0
#define GQA_ERR_ARG (-1)         /* null/aliasing pointer, bad size, bad combination */
#define GQA_ERR_UNSUPPORTED (-2) /* valid layer, shape outside what the kernels tile */
#define GQA_ERR_CUDA (-3)        /* a CUDA runtime call failed (message has details) */
#define GQA_ERR_TIMEOUT (-4)     /* a bounded device wait gave up */
#define GQA_ERR_WORKSPACE (-5)   /* workspace missing or smaller than required */
#define GQA_ERR_RANGE (-6)       /* reported by gqa_check_device_error: a prefill Q/K/V value
                                    beyond +-65504 was clamped to the binary16 range */

typedef uint16_t gqa_f16; /* bit pattern of one IEEE binary16 value */

/* ------------------------------------------------------------------ prefill */

/* Bytes of device workspace gqa_attn_forward_ex needs: Q [B,Hq,S,d],
 * K and V [B,Hkv,S,d] (binary16) and attn [B,S,Hq*d] (bf16), each 256-byte
 * aligned.  Returns 0 for invalid sizes.
 *
 * Why binary16 for Q, K and V: the attention step computes in fp32 from them
 * ([T07] §4 step 6 casts the 16-bit projections to float32).  binary16 keeps 3
 * more mantissa bits than bf16, so storing them costs the scores and outputs
 * an 8x smaller rounding error at the same bandwidth and tensor-core rate.
 * QK-norm bounds every Q and K row by sqrt(head_dim) * max|w|; a value beyond
 * the binary16 range (possible only for V, or without QK-norm, at magnitudes
 * above 65504) is clamped and reported as GQA_ERR_RANGE. */
size_t gqa_attn_workspace_size(int B, int S, int hidden, int Hq, int Hkv, int head_dim);

/* The whole layer forward ([T07] §4 steps 1-7; [NeoX] "Qwen3-0.6B example"):
 *   x        [B, S, hidden]
 *   Wqkv     [(Hq + 2*Hkv)*head_dim, hidden]   rows W_q; W_k; W_v
 *   Wo       [hidden, Hq*head_dim]
 *   q_norm_w [head_dim] or NULL; k_norm_w [head_dim] or NULL -- both NULL
 *            (no QK-norm) or both non-NULL, else GQA_ERR_ARG
 *   rope_theta > 0, eps >= 0; positions are 0..S-1 in every sequence
 *   causal   1: query t sees keys u <= t; 0: every key of its sequence
 *   out      [B, S, hidden] = x + o_proj(attn); must not overlap x or the
 *            weights (GQA_ERR_ARG)
 *   workspace: device memory of at least gqa_attn_workspace_size(...) bytes,
 *            256-byte aligned, not overlapping any argument; contents on exit
 *            are the intermediate Q, K, V and attn.
 * Stages run in order on `stream`: QKV projection (+ QK-norm + RoPE),
 * attention, o_proj (+ residual). */
int gqa_attn_forward_ex(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                        const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                        float rope_theta, float eps,
                        int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                        gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);

/* Same as gqa_attn_forward_ex on the legacy default stream with a workspace
 * the library allocates on first use and grows on demand (kept until exit).
 * Calls that overlap on the device share that workspace: serialise them. */
int gqa_attn_forward(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                     const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                     float rope_theta, float eps,
                     int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                     gqa_bf16 *out);

/* Bytes of device workspace gqa_attn_forward_host needs: that of
 * gqa_attn_workspace_size plus device copies of x and out (each 256-byte
 * aligned).  Returns 0 for invalid sizes. */
size_t gqa_attn_forward_host_workspace_size(int B, int S, int hidden, int Hq, int Hkv, int head_dim);

/* The layer forward of gqa_attn_forward_ex with x and out in HOST memory
 * (x_host [B, S, hidden] read, out_host [B, S, hidden] written; page-locked
 * memory lets the copies run asynchronously, pageable memory works but the
 * copies then serialise with the host).  Weights, norm weights and workspace
 * are device memory as for gqa_attn_forward_ex; workspace: at least
 * gqa_attn_forward_host_workspace_size(...) bytes, 256-byte aligned.
 * The copies overlap the compute: x is copied in by token chunks (at most four,
 * each a multiple of 128 rows, none below 2048 rows) on a copy stream the
 * library keeps per device, and each chunk's QKV projection starts on `stream`
 * when its rows have landed; after the attention, o_proj runs chunk by chunk
 * and each finished chunk of out is copied back while the next is computed.
 * The result is bit-identical to gqa_attn_forward_ex on the same inputs.  All
 * of it is ordered after the work already on `stream`, and `stream` resumes
 * after the last copy, so out_host is complete once `stream` is.  Calls that
 * share a workspace must not overlap on the device; the host-side enqueue is
 * serialised per device.  GQA_ERR_ARG also when x_host or out_host is device
 * memory or they overlap. */
int gqa_attn_forward_host(const gqa_bf16 *x_host, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                          const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                          float rope_theta, float eps,
                          int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                          gqa_bf16 *out_host, void *workspace, size_t workspace_bytes, void *stream);

/* Stage 1 alone: qkv = x @ Wqkv^T, then QK-norm and RoPE at positions
 * 0..S-1, written head-major ([T07] §4 steps 1-4), as binary16:
 *   q_out [B, Hq, S, head_dim], k_out and v_out [B, Hkv, S, head_dim]. */
int gqa_qkv_proj(const gqa_bf16 *x, const gqa_bf16 *Wqkv,
                 const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                 float rope_theta, float eps,
                 int B, int S, int hidden, int Hq, int Hkv, int head_dim,
                 gqa_f16 *q_out, gqa_f16 *k_out, gqa_f16 *v_out, void *stream);

/* Stage 2 alone: grouped-query attention with scale head_dim^-0.5, fp32
 * softmax and accumulation ([T07] §4 step 6; [NeoX] "Scaling and RoPE"):
 *   q [B, Hq, S, head_dim], k and v [B, Hkv, S, head_dim], binary16
 *   attn_out [B, S, Hq*head_dim], bf16 ([NeoX] "Attention output flattening").
 * Supported group sizes Hq/Hkv: up to 128 (a query tile packs floor(128/G)
 * positions of each of the G heads). */
int gqa_attention(const gqa_f16 *q, const gqa_f16 *k, const gqa_f16 *v,
                  int B, int S, int Hq, int Hkv, int head_dim, int causal,
                  gqa_bf16 *attn_out, void *stream);

/* Stage 3 alone: out = x + attn @ Wo^T ([NeoX] "Output projection"):
 *   attn [M, q_width], Wo [hidden, q_width], x and out [M, hidden];
 *   q_width and hidden multiples of 8; out must not overlap x. */
int gqa_oproj_residual(const gqa_bf16 *attn, const gqa_bf16 *Wo, const gqa_bf16 *x,
                       int M, int hidden, int q_width, gqa_bf16 *out, void *stream);

/* ---------------------------------------------------- prefill into a cache */

/* Bytes of workspace gqa_attn_prefill_cached needs, each part 256-byte
 * aligned: Q [B,Hq,S,d] binary16 and attn [B,S,Hq*d] bf16; room for the
 * attention's two key splits (their binary16 outputs [2][B,S,Hq*d] and fp32
 * log2-sum-exp rows [2][B*Hq,S]); and binary16 copies of both caches
 * [B,Hkv,Lmax,d], of which the call fills the rows it attends.  The keys are
 * split when the attention would otherwise run fewer than eight waves of work
 * items on the GPU (B*Hq*S/256 items against the SM count); a binary16 partial
 * beyond +-65504 is clamped and reported as GQA_ERR_RANGE.  Returns 0 for
 * invalid sizes. */
size_t gqa_attn_prefill_cached_workspace_size(int B, int S, int Hq, int Hkv, int head_dim, int Lmax);

/* Chunked prefill: S new tokens per sequence appended to a KV cache
 * ([T07] §4: RoPE at the position offsets, step 5 the cache returns the
 * whole history; [Part]: masks and positions use global token positions).
 *   x          [B, S, hidden], the new tokens of each sequence
 *   k_cache, v_cache [B, Hkv, Lmax, head_dim] bf16: entries [0, cache_len[b])
 *              hold earlier tokens (normed, rotated K; V); this call writes
 *              the new tokens' K and V at slots cache_len[b] .. cache_len[b]+S-1
 *   cache_len  device int32 [B]: tokens already cached = the first new
 *              token's position; needs cache_len[b] + S <= Lmax (checked on the
 *              device: violating sequences get zero attention rows and
 *              gqa_check_device_error reports GQA_ERR_ARG).  Not modified.
 *   causal     1: new token t sees keys u <= cache_len[b] + t; 0: all
 *              cache_len[b] + S keys
 *   out        [B, S, hidden] = x + o_proj(attn)
 * With cache_len = 0 this is the plain prefill that also fills the cache.
 * Q and P are binary16 as in the plain prefill: after the projection a
 * streaming kernel copies cache rows [0, cache_len[b] + S) of both caches,
 * widened to binary16, into the workspace (exact for every bf16 value below
 * 2^16; a cached value beyond +-65504 is saturated and reported as
 * GQA_ERR_RANGE by gqa_check_device_error), and the attention reads those
 * copies.  Cache slots past cache_len[b] + S are never read as keys or
 * values, whatever they hold. */
int gqa_attn_prefill_cached(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                            const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                            float rope_theta, float eps,
                            int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                            gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                            gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace gqa_attention_cached needs: binary16 copies of both
 * caches [B,Hkv,Lmax,d], each 256-byte aligned.  0 for invalid sizes. */
size_t gqa_attention_cached_workspace_size(int B, int Hkv, int head_dim, int Lmax);

/* Its attention stage alone (the widening copy, then the attention):
 * q [B, Hq, S, head_dim] binary16 (positions cache_len[b] + t) over keys
 * [0, cache_len[b] + S) of the bf16 caches (the new tokens' keys already
 * appended); attn_out [B, S, Hq*head_dim] bf16; workspace at least
 * gqa_attention_cached_workspace_size(...) bytes, 256-byte aligned. */
int gqa_attention_cached(const gqa_f16 *q, const gqa_bf16 *k_cache, const gqa_bf16 *v_cache,
                         const int *cache_len, int B, int S, int Hq, int Hkv, int head_dim, int Lmax,
                         int causal, gqa_bf16 *attn_out, void *workspace, size_t workspace_bytes,
                         void *stream);

/* ------------------------------------------------------------------- decode */

/* Bytes of device workspace gqa_attn_decode needs (Q of the new tokens,
 * attn, and the split-KV partial results).  Returns 0 for invalid sizes. */
size_t gqa_attn_decode_workspace_size(int B, int hidden, int Hq, int Hkv, int head_dim, int Lmax);

/* One decode step: one new token per sequence over a KV cache ([T07] §4
 * with L = 1; step 5 "update and fetch" of the cache).
 *   x          [B, hidden], the new tokens
 *   k_cache, v_cache [B, Hkv, Lmax, head_dim]: entries [0, cache_len[b]) hold
 *              the normed and rotated keys / the values of earlier tokens;
 *              this call writes the new token's K and V at slot cache_len[b]
 *   cache_len  device int32 [B]: tokens already cached; the new token's
 *              position and slot.  Must satisfy 0 <= cache_len[b] < Lmax
 *              (device-side values are not checked on the host; out-of-range
 *              rows are skipped and reported as GQA_ERR_ARG through
 *              gqa_check_device_error).  Not modified: the caller advances it.
 *   out        [B, hidden] = x + o_proj(attn over keys 0..cache_len[b])
 *   workspace  at least gqa_attn_decode_workspace_size(...) bytes. */
int gqa_attn_decode(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                    const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                    float rope_theta, float eps,
                    int B, int hidden, int Hq, int Hkv, int head_dim,
                    gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                    gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);

/* Decode stage 1 alone: projection + QK-norm + RoPE at position
 * cache_len[b]; q_out [B, Hq, head_dim] as binary16 (see
 * gqa_attn_workspace_size for why); K and V written as bf16 into the caches at
 * slot cache_len[b]. */
int gqa_decode_qkv(const gqa_bf16 *x, const gqa_bf16 *Wqkv,
                   const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                   float rope_theta, float eps,
                   int B, int hidden, int Hq, int Hkv, int head_dim,
                   gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                   gqa_f16 *q_out, void *stream);

/* Bytes of workspace gqa_decode_attention needs for its split partials. */
size_t gqa_decode_attention_workspace_size(int B, int Hq, int Hkv, int head_dim, int Lmax);

/* Decode stage 2 alone: split-KV attention of one query per sequence,
 * q [B, Hq, head_dim] binary16, over keys [0, kv_len[b]) of the bf16 caches
 * [B, Hkv, Lmax, head_dim]; kv_len device int32 [B], 1 <= kv_len[b] <= Lmax.
 * attn_out [B, Hq*head_dim] bf16. */
int gqa_decode_attention(const gqa_f16 *q, const gqa_bf16 *k_cache, const gqa_bf16 *v_cache,
                         const int *kv_len, int B, int Hq, int Hkv, int head_dim, int Lmax,
                         gqa_bf16 *attn_out, void *workspace, size_t workspace_bytes,
                         void *stream);

/* The same decode attention as gqa_decode_attention, for callers that cannot
 * allocate device memory: no workspace argument, and the call itself performs
 * no allocation.  It is meant for hosts that give a kernel only its input and
 * output buffers (plugin or custom-op interfaces without a workspace hook) and
 * for serving loops whose device memory is owned entirely by another
 * allocator.  The pages have no counterpart for this entry point; it exists
 * only for those callers.
 *   Scratch: a fixed 16 MiB array of fp32 split partials compiled into the
 *   library (kept on every GPU that loads the library until the process
 *   exits).  Sizes whose partials for a single split exceed it
 *   (B*Hq*(head_dim+2) > 4194304 floats) return GQA_ERR_UNSUPPORTED; larger
 *   problems may use fewer splits than gqa_decode_attention does, so results
 *   agree to rounding, not bit for bit.
 *   Sharing: every call uses the same array and leaves its last partials in
 *   it; calls that overlap on the GPU race and give wrong results, so order
 *   them (one stream, or events).
 *   Set-up: the first call on a device looks up the array's device address
 *   with that device current; make that first call before any stream capture.
 *   Errors found on the device: a bounded wait that gave up (GQA_ERR_TIMEOUT)
 *   or a kv_len outside [1, Lmax] (GQA_ERR_ARG; that sequence gets zero rows)
 *   is recorded in an error word that lives beside the array.  Each call
 *   clears that word on its stream before its kernels run, so one call's
 *   timeout never affects a later call; gqa_check_device_error() reads and
 *   clears it, so check after a call and before the next one is enqueued to
 *   see that call's errors.  Neither the clearing nor the check allocates.
 * Arguments, size limits and the statuses of invalid arguments are those of
 * gqa_decode_attention; gqa_last_launch_count() is 2 after a call that
 * launched. */
int gqa_decode_attention_noalloc(const gqa_f16 *q, const gqa_bf16 *k_cache, const gqa_bf16 *v_cache,
                                 const int *kv_len, int B, int Hq, int Hkv, int head_dim, int Lmax,
                                 gqa_bf16 *attn_out, void *stream);

/* ------------------------------------------------ FP8 (E4M3) KV cache */

/* The decode step with its caches in FP8 ("Head Dimension" article, §5.2:
 * FP8 precision for the K, V cache).  A cache element is one OCP FP8 E4M3
 * code (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest finite
 * value 448) and stands for code * k_scale (keys) or code * v_scale (values),
 * one scale per tensor.  A new key or value is stored as the code nearest to
 * value / scale (value / scale computed in fp32, ties to even), saturated to
 * +-448; a saturated or NaN value sets the range flag that
 * gqa_check_device_error() reports as GQA_ERR_RANGE.  Caches are
 * [B, Hkv, Lmax, head_dim] codes, half the bytes of bf16 caches; everything
 * else (arguments, workspace and its size, positions, statuses) is as for
 * the bf16 functions of the same name without _fp8.  head_dim must be 64,
 * 80, 96, 128 or 256 (else GQA_ERR_UNSUPPORTED); k_scale and v_scale must be
 * finite and > 0 (else GQA_ERR_ARG). */
typedef uint8_t gqa_e4m3; /* one OCP FP8 E4M3 code */

int gqa_attn_decode_fp8(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                        const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                        float rope_theta, float eps,
                        int B, int hidden, int Hq, int Hkv, int head_dim,
                        gqa_e4m3 *k_cache, gqa_e4m3 *v_cache, float k_scale, float v_scale,
                        const int *cache_len, int Lmax,
                        gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);

/* Stage alone: projection, QK-norm and RoPE of the new token, its key and
 * value appended to the E4M3 caches at slot cache_len[b]; q_out [B, Hq,
 * head_dim] binary16. */
int gqa_decode_qkv_fp8(const gqa_bf16 *x, const gqa_bf16 *Wqkv,
                       const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                       float rope_theta, float eps,
                       int B, int hidden, int Hq, int Hkv, int head_dim,
                       gqa_e4m3 *k_cache, gqa_e4m3 *v_cache, float k_scale, float v_scale,
                       const int *cache_len, int Lmax, gqa_f16 *q_out, void *stream);

/* Stage alone: split-KV attention of q [B, Hq, head_dim] (binary16) over
 * keys [0, kv_len[b]) of the E4M3 caches; attn_out [B, Hq*head_dim] bf16;
 * workspace of gqa_decode_attention_workspace_size(...) bytes. */
int gqa_decode_attention_fp8(const gqa_f16 *q, const gqa_e4m3 *k_cache, const gqa_e4m3 *v_cache,
                             float k_scale, float v_scale, const int *kv_len,
                             int B, int Hq, int Hkv, int head_dim, int Lmax,
                             gqa_bf16 *attn_out, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------- partial rotary */

/* The same five layer entry points with the rotary width as an argument:
 * RoPE rotates only the first rotary_dim features of every Q and K head,
 * pairing element i with i + rotary_dim/2 at angle
 * pos * theta^(-2i/rotary_dim); features [rotary_dim, head_dim) are
 * normalised but not rotated ([NeoX] "Scaling and RoPE": RoPE is built from
 * the effective head_dim subject to the rotary_pct setting, i.e. rotary_dim =
 * head_dim * rotary_pct, and an even width).  rotary_dim = head_dim is the
 * plain entry point; rotary_dim = 0 applies no rotation.  rotary_dim odd,
 * negative or above head_dim: GQA_ERR_ARG; a value other than head_dim,
 * head_dim/2, head_dim/4 or 0: GQA_ERR_UNSUPPORTED.  Every other argument,
 * layout, ownership rule and status is that of the function without _rd. */
int gqa_attn_forward_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                        const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                        float rope_theta, float eps, int rotary_dim,
                        int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                        gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);
int gqa_qkv_proj_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv,
                    const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                    float rope_theta, float eps, int rotary_dim,
                    int B, int S, int hidden, int Hq, int Hkv, int head_dim,
                    gqa_f16 *q_out, gqa_f16 *k_out, gqa_f16 *v_out, void *stream);
int gqa_attn_prefill_cached_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                               const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                               float rope_theta, float eps, int rotary_dim,
                               int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                               gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                               gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);
int gqa_attn_decode_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                       const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                       float rope_theta, float eps, int rotary_dim,
                       int B, int hidden, int Hq, int Hkv, int head_dim,
                       gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                       gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);
int gqa_decode_qkv_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv,
                      const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                      float rope_theta, float eps, int rotary_dim,
                      int B, int hidden, int Hq, int Hkv, int head_dim,
                      gqa_bf16 *k_cache, gqa_bf16 *v_cache, const int *cache_len, int Lmax,
                      gqa_f16 *q_out, void *stream);

/* ---------------------------------------------------------------- backward */

/* Gradients of the whole layer (the derivatives of [T07] §4 steps 1-7 in
 * reverse order; the K and V projections receive the gradients of every
 * query head of their group, [NeoX] "Qwen3-0.6B example", [Part]).  Given the
 * forward's inputs and dout = dL/dout [B, S, hidden] (bf16), writes
 *   dx        [B, S, hidden]               bf16  (dout plus the path through the projection)
 *   dWqkv     [(Hq+2Hkv)*head_dim, hidden] fp32
 *   dWo       [hidden, Hq*head_dim]        fp32
 *   dq_norm_w, dk_norm_w [head_dim]        fp32  (required with QK-norm, else may be NULL)
 * The forward is recomputed (Q, K, V, the attention's per-row log-sum-exp);
 * the attention backward recomputes its probabilities from them.  Full
 * rotary (the *_rd forms below take a rotary width); head_dim 64, 80, 96 or
 * 128; Hq/Hkv up to 32, else GQA_ERR_UNSUPPORTED (head_dim
 * 256: the dK and dV accumulators of a 128-key block would fill all 512 TMEM
 * columns).  dx must not overlap x or dout.  workspace: at least
 * gqa_attn_backward_workspace_size(...) bytes, 256-byte aligned.  Enqueued on
 * `stream`. */
size_t gqa_attn_backward_workspace_size(int B, int S, int hidden, int Hq, int Hkv, int head_dim);
int gqa_attn_backward(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                      const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                      float rope_theta, float eps,
                      int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                      const gqa_bf16 *dout, gqa_bf16 *dx, float *dWqkv, float *dWo,
                      float *dq_norm_w, float *dk_norm_w,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Training pair.  gqa_attn_forward_train is the layer forward of
 * gqa_attn_forward_ex (same arguments, same out bit for bit) that also keeps,
 * in `workspace` (gqa_attn_backward_workspace_size bytes, 256-byte aligned),
 * what the backward needs: Q, K, V (binary16, head-major), the pre-norm Q and
 * K rows (fp32, with QK-norm), the attention output and its log2-sum-exp.
 * gqa_attn_backward_saved then computes the gradients of gqa_attn_backward
 * (same arguments, same results bit for bit) from that workspace instead of
 * recomputing the QKV projection and the forward attention.  Between the two
 * calls the workspace must not be changed, and x, the weights, the norm
 * weights, rope_theta, eps, sizes and causal must be the same; nothing checks
 * this.  Shape limits as for gqa_attn_backward. */
int gqa_attn_forward_train(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                           const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                           float rope_theta, float eps,
                           int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                           gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);
int gqa_attn_backward_saved(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                            const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                            float rope_theta, float eps,
                            int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                            const gqa_bf16 *dout, gqa_bf16 *dx, float *dWqkv, float *dWo,
                            float *dq_norm_w, float *dk_norm_w,
                            void *workspace, size_t workspace_bytes, void *stream);

/* The three above with RoPE on the first rotary_dim features only ([NeoX]
 * "Scaling and RoPE", rotary_pct; as the other *_rd entry points: rotary_dim
 * head_dim, head_dim/2, head_dim/4 or 0, else GQA_ERR_UNSUPPORTED; odd or out
 * of [0, head_dim]: GQA_ERR_ARG).  The inverse rotation of the backward
 * acts on the same features; the training pair's two calls must take the same
 * rotary_dim. */
int gqa_attn_backward_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                         const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                         float rope_theta, float eps, int rotary_dim,
                         int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                         const gqa_bf16 *dout, gqa_bf16 *dx, float *dWqkv, float *dWo,
                         float *dq_norm_w, float *dk_norm_w,
                         void *workspace, size_t workspace_bytes, void *stream);
int gqa_attn_forward_train_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                              const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                              float rope_theta, float eps, int rotary_dim,
                              int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                              gqa_bf16 *out, void *workspace, size_t workspace_bytes, void *stream);
int gqa_attn_backward_saved_rd(const gqa_bf16 *x, const gqa_bf16 *Wqkv, const gqa_bf16 *Wo,
                               const gqa_bf16 *q_norm_w, const gqa_bf16 *k_norm_w,
                               float rope_theta, float eps, int rotary_dim,
                               int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                               const gqa_bf16 *dout, gqa_bf16 *dx, float *dWqkv, float *dWo,
                               float *dq_norm_w, float *dk_norm_w,
                               void *workspace, size_t workspace_bytes, void *stream);

/* Stage alone: the attention backward.  q [B, Hq, S, head_dim], k and v
 * [B, Hkv, S, head_dim], dO [B, Hq, S, head_dim] (all binary16, head-major);
 * writes dq [B, Hq, S, head_dim] and dk, dv [B, Hkv, S, head_dim] in fp32
 * (dk and dv summed over each group's query heads).  The forward attention
 * is recomputed into the workspace (gqa_attention_backward_workspace_size
 * bytes, 256-byte aligned).  Same shape limits as gqa_attn_backward. */
size_t gqa_attention_backward_workspace_size(int B, int S, int Hq, int head_dim);
int gqa_attention_backward(const gqa_f16 *q, const gqa_f16 *k, const gqa_f16 *v, const gqa_f16 *dO,
                           int B, int S, int Hq, int Hkv, int head_dim, int causal,
                           float *dq, float *dk, float *dv,
                           void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------ accounting */

/* Algorithmic cost of one prefill forward, all pointers host, any may be NULL
 * ([Knob] "Why the cost does not move"):
 *   weights          q/k/v/o projection weights = hidden*(Hq+2Hkv)*d + Hq*d*hidden
 *   proj_macs_per_token = weights (each weight used once per token)
 *   attn_macs        score + value multiply-accumulates over the whole batch:
 *                    2*d per (query head, query, visible key); causal counts
 *                    the S(S+1)/2 visible pairs per sequence
 *   flops            2*(B*S*proj_macs_per_token + attn_macs)
 * Returns GQA_ERR_ARG for non-positive sizes. */
int gqa_attn_cost(int B, int S, int hidden, int Hq, int Hkv, int head_dim, int causal,
                  long long *weights, long long *proj_macs_per_token,
                  long long *attn_macs, long long *flops);

/* ------------------------------------------------------------- diagnostics */

/* Message for the last nonzero status returned on the calling thread. */
const char *gqa_last_error(void);

/* Synchronises the current device, then reads and clears its device error
 * words: the per-device word of the workspace-taking entry points and the one
 * of gqa_decode_attention_noalloc.  Returns GQA_OK, GQA_ERR_TIMEOUT (a bounded
 * wait gave up), GQA_ERR_ARG (a device-side index check failed),
 * GQA_ERR_RANGE (a value was clamped) or GQA_ERR_CUDA.  Allocates nothing on
 * a device where only gqa_decode_attention_noalloc has run. */
int gqa_check_device_error(void);

/* The same check without synchronising the whole device: waits only for the
 * work queued on `stream` (a cudaStream_t; NULL: the legacy default stream,
 * which waits for every blocking stream), then reads and clears the current
 * device's error words with copies ordered on that stream.  The words are per
 * device, so an error recorded by another stream's kernel that has already
 * run is reported here too (and cleared).  Returns as gqa_check_device_error. */
int gqa_check_stream_error(void *stream);

/* Watchdog self-test: launches one kernel whose mbarrier wait can never
 * complete, with a wait limit of limit_ms milliseconds (1..5000), waits for
 * it, and returns what the kernel reported: GQA_ERR_TIMEOUT when the bounded
 * wait works.  The device stays usable afterwards. */
int gqa_selftest_bounded_wait(int limit_ms);

/* Number of kernels the last successful host call enqueued (for launch
 * accounting in benchmarks). */
int gqa_last_launch_count(void);

/* Process-wide choice of kernel forms.  By default the prefill projections
 * (head_dim 64 / 128 QKV and o_proj with more than 128 rows) and the
 * head_dim 256 attention run on 2-CTA clusters (tcgen05 cta_group::2) whenever
 * that cluster shape can be placed on the device; enable = 0 makes every
 * later launch use the one-CTA kernels instead (same results up to rounding
 * order), enable != 0 restores the default.  Returns the previous setting
 * (1 or 0).  A diagnostic and tuning switch: it is read at each launch, so it
 * should not be changed while another thread enqueues work. */
int gqa_set_cta_pairs(int enable);

#ifdef __cplusplus
}
#endif
#endif /* GQA_ATTN_H */
