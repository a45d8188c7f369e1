// cache.cu -- the binary16 copy of the bf16 KV-cache rows that prefill into a
// cache attends ([T07] §4 steps 5-6: the cache returns the whole history and
// the attention of the new tokens reads all of it).
//
// The attention kernels compute in binary16 (Q, K, V and P): binary16 keeps 3
// more mantissa bits than bf16, and Q or P rounded to bf16 to meet a bf16 key
// or value in one tensor-core product (both operands of a product share their
// type) would add that rounding to every score and output.  So before the
// attention of a chunk, this kernel widens rows [0, cache_len[b] + S) of every
// KV head of both caches to binary16 -- once per call, where widening inside
// the attention would repeat it for every block of queries that reads the
// row.  It is a pure streaming kernel: each row is read once (bf16) and
// written once (binary16), 16 bytes per thread access.
//
// Every bf16 value below 2^16 in magnitude is exactly a binary16 value (8
// significant bits fit in 11; bf16 values under binary16's normal range lose
// only bits far below the rows' scale); larger ones saturate to +-65504 and
// set the range flag.  Rows from cache_len[b] + S up to the end of the last
// key tile the attention reads are zero-filled: those cache slots were never
// written and may hold anything, and a NaN value times a zero probability
// would still reach the output.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kThreadsW = 256;
constexpr int kUnroll = 4;  // 16-byte units per thread

// grid: (b * Hkv + g) * per_head + block, per_head blocks over the Lmax * d / 8
// units of one head.
__global__ void __launch_bounds__(kThreadsW) cache_widen_kernel(const uint4 *k_cache, const uint4 *v_cache,
                                                                uint4 *k16, uint4 *v16, const int *cache_len, int S,
                                                                int Hkv, int Lmax, int d, int tile, int per_head,
                                                                unsigned *err)
{
    grid_dep_launch();  // the attention may start its prologue meanwhile
    grid_dep_wait();    // the new tokens' keys and values come from the projection kernel
    const int bg = blockIdx.x / per_head;
    const int blk = blockIdx.x - bg * per_head;
    const int b = bg / Hkv;
    const int p0 = cache_len[b];
    if (p0 < 0 || p0 + S > Lmax) return;  // the attention reports and skips this sequence
    const int valid = p0 + S;
    const int rows = min(Lmax, (valid + tile - 1) / tile * tile);
    const int upr = d / 8;  // 16-byte units per row
    const long long n = (long long)rows * upr;
    const size_t head = (size_t)bg * Lmax * upr;
    uint32_t over = 0;
    const long long base = (long long)blk * kThreadsW * kUnroll + threadIdx.x;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const uint4 *src = (c ? v_cache : k_cache) + head;
        uint4 *dst = (c ? v16 : k16) + head;
        uint4 w[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const long long i = base + (long long)k * kThreadsW;
            w[k] = (i < n && i / upr < valid) ? src[i] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const long long i = base + (long long)k * kThreadsW;
            if (i < n) {
                uint4 o;
                o.x = bf16x2_to_f16x2(w[k].x, over);
                o.y = bf16x2_to_f16x2(w[k].y, over);
                o.z = bf16x2_to_f16x2(w[k].z, over);
                o.w = bf16x2_to_f16x2(w[k].w, over);
                dst[i] = o;
            }
        }
    }
    if (over & 0x80008000u) atomicOr(err, kErrRange);
}

}  // namespace

cudaError_t launch_cache_widen(const CacheWiden &p, unsigned *err, cudaStream_t stream)
{
    if (p.d % 8 || p.tile <= 0 || p.B <= 0 || p.Hkv <= 0 || p.Lmax <= 0) return cudaErrorInvalidValue;
    const long long units = (long long)p.Lmax * (p.d / 8);
    const long long per_block = (long long)kThreadsW * kUnroll;
    const long long per_head = (units + per_block - 1) / per_block;
    const long long blocks = per_head * p.B * p.Hkv;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    LaunchCfg lc(dim3((unsigned)blocks), dim3(kThreadsW), 0, stream, p.pdl != 0);
    cudaError_t e = cudaLaunchKernelEx(&lc.cfg, cache_widen_kernel, reinterpret_cast<const uint4 *>(p.k_cache),
                                       reinterpret_cast<const uint4 *>(p.v_cache), reinterpret_cast<uint4 *>(p.k16),
                                       reinterpret_cast<uint4 *>(p.v16), p.cache_len, p.S, p.Hkv, p.Lmax, p.d, p.tile,
                                       (int)per_head, err);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace gqa
