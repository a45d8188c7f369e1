// selftest.cu -- watchdog self-test: a kernel that waits on an mbarrier no
// thread will ever arrive at.  The bounded wait must give up after limit_ns,
// record kErrTimeout in the device error word and let the kernel return, so
// the device stays usable.
#include "internal.h"
#include "ptx.cuh"

namespace gqa {

namespace {

__global__ void selftest_wait_kernel(unsigned *err, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, err, limit_ns);  // never completes: returns false
    __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(unsigned *err, unsigned long long limit_ns, cudaStream_t stream)
{
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gqa
