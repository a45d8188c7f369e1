// noalloc.cu -- decode attention for callers that cannot allocate device
// memory.
//
// gqa_decode_attention needs a scratch buffer for its split-KV partial
// results, and the caller passes it in.  Some callers have no way to provide
// one: a plugin or custom-op host that hands out only input and output
// buffers, or a serving loop whose device memory is entirely owned by another
// allocator with nothing left to hand out.  For them this file keeps the
// scratch in a fixed array inside the library image, so the call itself
// allocates nothing.
//
// Limits and sharing:
//   - the array holds kScratchFloats floats (16 MiB); every GPU that loads the
//     library keeps it until the process exits;
//   - all calls share it and it keeps the last call's partials.  Each call
//     overwrites every partial record it reads, so nothing has to start at
//     zero; but two calls that overlap on the GPU (different streams, no
//     ordering between them) race on it and give wrong results;
//   - the first call on a device looks up the array's device address (once
//     per device, with that device current), so make that first call before
//     any stream capture begins;
//   - the kernels' error word (a bounded wait that gave up) sits beside the
//     array: each call clears it on its own stream before its kernels run, so
//     a timeout in one call cannot cut short the waits of later calls, and
//     gqa_check_device_error() reads and clears it (it reports GQA_ERR_TIMEOUT
//     for a call whose waits gave up, if made before the next call's clearing
//     runs).  Neither needs an allocation.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "../../include/gqa_attn.h"
#include "internal.h"

namespace gqa {
namespace {

constexpr size_t kScratchFloats = (size_t)4 << 20;  // 16 MiB of fp32 partials

__device__ __align__(256) float g_noalloc_scratch[kScratchFloats];
__device__ __align__(256) unsigned g_noalloc_err[64];  // word 0 is used

struct NoAllocDevice {
    bool ready = false;
    float *scratch = nullptr;  // device address of g_noalloc_scratch
    unsigned *err = nullptr;   // device address of g_noalloc_err
    int num_sms = 0;
};

std::mutex g_noalloc_mu;
NoAllocDevice g_noalloc_dev[64];

// the message is what gqa_last_error() returns on this thread
int noalloc_fail(int code, const char *msg)
{
    record_error_message(msg);
    return code;
}

// Host code may not use g_noalloc_scratch directly: in host code that name is a
// host-side stand-in, not a device address.  Look the address up per device.
int noalloc_setup(NoAllocDevice **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return noalloc_fail(GQA_ERR_CUDA, "gqa_decode_attention_noalloc: no current CUDA device");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return noalloc_fail(GQA_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed");
        d.scratch = static_cast<float *>(p);
        e = cudaGetSymbolAddress(&p, g_noalloc_err);
        if (e != cudaSuccess) return noalloc_fail(GQA_ERR_CUDA, "cudaGetSymbolAddress(error word) failed");
        d.err = static_cast<unsigned *>(p);
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return noalloc_fail(GQA_ERR_CUDA, "cudaDeviceGetAttribute failed");
        d.ready = true;
    }
    *out = &d;
    return GQA_OK;
}

}  // namespace

unsigned noalloc_take_error_word(int dev, cudaStream_t stream, bool on_stream)
{
    if (dev < 0 || dev >= 64) return 0;
    unsigned *err;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_dev[dev].ready) return 0;
        err = g_noalloc_dev[dev].err;
    }
    unsigned word = 0;
    if (on_stream) {  // ordered on the stream, which alone is waited for
        if (cudaMemcpyAsync(&word, err, sizeof word, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return 0;
        if (word) cudaMemsetAsync(err, 0, sizeof word, stream);
        return word;
    }
    if (cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return 0;
    if (word) cudaMemset(err, 0, sizeof word);
    return word;
}

}  // namespace gqa

using namespace gqa;

extern "C" int gqa_decode_attention_noalloc(const gqa_f16 *q, const gqa_bf16 *k_cache, const gqa_bf16 *v_cache,
                                            const int *kv_len, int B, int Hq, int Hkv, int head_dim, int Lmax,
                                            gqa_bf16 *attn_out, void *stream)
{
    set_launch_count(0);
    // the same sizes, group sizes and head widths as gqa_decode_attention, with the same statuses
    int rc = check_decode_attention_args(B, Hq, Hkv, head_dim, Lmax);
    if (rc) return rc;
    if (!q || !k_cache || !v_cache || !kv_len || !attn_out)
        return noalloc_fail(GQA_ERR_ARG, "gqa_decode_attention_noalloc: null pointer");
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)attn_out) & 15u)
        return noalloc_fail(GQA_ERR_ARG, "gqa_decode_attention_noalloc: tensor pointers must be 16-byte aligned");
    // the partials of one split must fit in the fixed array
    const size_t per_split = decode_partials_floats(B, Hq, 1, head_dim);
    if (per_split > kScratchFloats) {
        char m[256];
        snprintf(m, sizeof m,
                 "gqa_decode_attention_noalloc: B*Hq*(head_dim+2) = %zu floats of scratch exceed the fixed "
                 "%zu-float array; use gqa_decode_attention with a caller workspace",
                 per_split, kScratchFloats);
        return noalloc_fail(GQA_ERR_UNSUPPORTED, m);
    }
    NoAllocDevice *d;
    rc = noalloc_setup(&d);
    if (rc) return rc;
    int splits = decode_choose_splits(B, Hkv, Lmax, d->num_sms);
    const int fit = (int)(kScratchFloats / per_split);
    if (splits > fit) splits = fit;
    DecodeAttentionProblem p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.len = kv_len;
    p.len_bias = 0;
    p.out = attn_out;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = head_dim;
    p.Lmax = Lmax;
    p.partials = d->scratch;
    p.splits = splits;
    // a timeout recorded by an earlier call must not make this call's waits give up
    cudaError_t e = cudaMemsetAsync(d->err, 0, sizeof(unsigned), (cudaStream_t)stream);
    if (e != cudaSuccess)
        return noalloc_fail(GQA_ERR_CUDA, "gqa_decode_attention_noalloc: clearing the error word failed");
    e = launch_decode_attention(p, d->err, (cudaStream_t)stream);
    if (e != cudaSuccess) return noalloc_fail(GQA_ERR_CUDA, "gqa_decode_attention_noalloc: launch failed");
    set_launch_count(2);
    return GQA_OK;
}
