// backward.cu -- the elementwise part of the layer's backward: inverse RoPE
// and the RMSNorm (QK-norm) gradient, from the attention-input gradients to
// the gradient of the fused projection's output.
//
// For one Q or K head row at position t (the derivatives of [T07] §3 and §4
// steps 2-3; rotation pairs (i, i + rd/2) of the first rd features at angle
// t * theta^(-2i/rd), rd the rotary width):
//   dn = RoPE^T(dy)                       (rotation by -angle; features >= rd unchanged)
//   u = x r, r = (mean(x^2) + eps)^(-1/2)  (x: the pre-norm row of the forward)
//   dx_i = r (w_i dn_i - u_i / d * sum_k u_k w_k dn_k),   dw_i += u_i dn_i
// Without QK-norm dx = dn.  V rows pass unchanged.  One warp per (token,
// head) row at a time, each warp walking rows with a grid stride (a few
// blocks per SM); lane l holds elements l, l + 32, ... of the row, and the
// rotation partner of an element comes through the warp's row in shared
// memory (partners are rd/2 apart, which at head widths 80 and 96 or a
// partial rotary width is not a multiple of 32).  The norm-weight gradients
// are summed in each lane's registers over its rows, then per block in shared
// memory, and added to the global [d] vectors once per block (a block per row
// would send every row's terms through the same d global addresses).
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

constexpr int kWarpsPerBlock = 8;

template <int D>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    rope_norm_bwd_kernel(const RopeNormBwd P)
{
    constexpr int E = (D + 31) / 32;  // elements per lane (the last may be partly past d)
    __shared__ float s_dw[2][D];      // q_norm_w, k_norm_w gradients of this block
    __shared__ float s_row[kWarpsPerBlock][D];  // each warp's row, for the rotation partners
    for (int i = threadIdx.x; i < 2 * D; i += blockDim.x) (&s_dw[0][0])[i] = 0.0f;
    __syncthreads();
    const int lane = threadIdx.x % 32;
    float *buf = s_row[threadIdx.x / 32];
    const int NH = P.Hq + P.Hkv;
    const int rd = P.rd, hr = rd / 2;
    float accq[E], acck[E];  // this lane's norm-weight gradient terms (q_norm_w, k_norm_w) over its rows
#pragma unroll
    for (int e = 0; e < E; ++e) accq[e] = acck[e] = 0.0f;
    const long rows = (long)P.M * NH;
    for (long row = (long)blockIdx.x * kWarpsPerBlock + threadIdx.x / 32; row < rows;
         row += (long)gridDim.x * kWarpsPerBlock) {  // row = m * NH + h
        const long m = row / NH;
        const int h = (int)(row - m * NH);
        const int b = (int)(m / P.S), t = (int)(m - (long)b * P.S);
        const bool isq = h < P.Hq;
        const int head = isq ? h : h - P.Hq;
        const float *dy = isq ? P.dq + ((size_t)(b * P.Hq + head) * P.S + t) * D
                              : P.dk + ((size_t)(b * P.Hkv + head) * P.S + t) * D;
        float y[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = lane + 32 * e;
            y[e] = i < D ? dy[i] : 0.0f;
        }
        if (rd > 0) {  // inverse rotation of pairs (i, i + rd/2), i < rd/2
#pragma unroll
            for (int e = 0; e < E; ++e)
                if (lane + 32 * e < D) buf[lane + 32 * e] = y[e];
            __syncwarp();
            const float2 *cs = P.rope + (size_t)t * hr;  // (cos, sin) of the rotary width's angles
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int i = lane + 32 * e;
                if (i < hr) {
                    const float2 c = cs[i];
                    y[e] = buf[i] * c.x + buf[i + hr] * c.y;
                } else if (i < rd) {
                    const float2 c = cs[i - hr];
                    y[e] = buf[i] * c.x - buf[i - hr] * c.y;
                }
            }
            __syncwarp();  // the row buffer is rewritten for the next row
        }
        const int col = isq ? head * D : P.Hq * D + head * D;
        uint16_t *dst = P.dqkv + (size_t)m * P.N + col;
        if (P.pre) {
            const uint16_t *w = isq ? P.q_norm_w : P.k_norm_w;
            const float *x = P.pre + (size_t)m * NH * D + (size_t)h * D;
            float xv[E], wv[E], ss = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int i = lane + 32 * e;
                xv[e] = i < D ? x[i] : 0.0f;
                wv[e] = i < D ? bf16lo(w[i]) : 0.0f;
                ss = fmaf(xv[e], xv[e], ss);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            const float r = 1.0f / sqrtf(ss * (1.0f / D) + P.eps);
            float dot = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) dot = fmaf(xv[e] * r * wv[e], y[e], dot);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float u = xv[e] * r;
                const float term = u * y[e];
                accq[e] += isq ? term : 0.0f;
                acck[e] += isq ? 0.0f : term;
                y[e] = r * (wv[e] * y[e] - u * dot * (1.0f / D));
            }
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = lane + 32 * e;
            if (i < D) {
                const __nv_bfloat16 v = __float2bfloat16_rn(y[e]);
                dst[i] = *reinterpret_cast<const uint16_t *>(&v);
            }
        }
        if (!isq) {  // the V row of the same KV head passes unchanged
            const float *dv = P.dv + ((size_t)(b * P.Hkv + head) * P.S + t) * D;
            uint16_t *vdst = P.dqkv + (size_t)m * P.N + (P.Hq + P.Hkv) * D + head * D;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int i = lane + 32 * e;
                if (i < D) {
                    const __nv_bfloat16 v = __float2bfloat16_rn(dv[i]);
                    vdst[i] = *reinterpret_cast<const uint16_t *>(&v);
                }
            }
        }
    }
    if (P.pre) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int i = lane + 32 * e;
            if (i < D) {
                atomicAdd(&s_dw[0][i], accq[e]);
                atomicAdd(&s_dw[1][i], acck[e]);
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < D; i += blockDim.x) {
            atomicAdd(P.dq_norm_w + i, s_dw[0][i]);
            atomicAdd(P.dk_norm_w + i, s_dw[1][i]);
        }
    }
}

}  // namespace

cudaError_t launch_rope_norm_bwd(const RopeNormBwd &p, cudaStream_t stream)
{
    const long rows = (long)p.M * (p.Hq + p.Hkv);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    const unsigned grid = (unsigned)(blocks < 4L * sms ? blocks : 4L * sms);  // grid-stride over the rest
    if (p.rd < 0 || p.rd > p.d || (p.rd & 1) || (p.rd > 0 && !p.rope)) return cudaErrorInvalidValue;
    if (p.d == 128)
        rope_norm_bwd_kernel<128><<<grid, 32 * kWarpsPerBlock, 0, stream>>>(p);
    else if (p.d == 64)
        rope_norm_bwd_kernel<64><<<grid, 32 * kWarpsPerBlock, 0, stream>>>(p);
    else if (p.d == 80)
        rope_norm_bwd_kernel<80><<<grid, 32 * kWarpsPerBlock, 0, stream>>>(p);
    else if (p.d == 96)
        rope_norm_bwd_kernel<96><<<grid, 32 * kWarpsPerBlock, 0, stream>>>(p);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace gqa
