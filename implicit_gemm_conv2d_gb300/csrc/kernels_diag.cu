// kernels_diag.cu -- the bounded-wait self-test: one thread waits on an mbarrier that
// nothing completes, through the same hardware-suspending try_wait the tensor-core kernels
// use, gives up after a short bounded loop, records the timeout in its own status word
// (merged into conv_device_status) and returns, so the timeout path can be exercised
// without faulting or hanging the GPU.
#include "internal.h"
#include "tc_ptx.cuh"

namespace igc {

__device__ unsigned int g_diag_status = 0;

namespace {

__global__ void wait_selftest_kernel(unsigned max_sleeps)
{
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(tc::smem_u32(&bar), 1);
    tc::fence_mbar_init();
    for (unsigned i = 0; i < max_sleeps; ++i)
        if (tc::mbar_try_wait_sleep(tc::smem_u32(&bar), 0u, 1000u)) return;  // no arrival: not reached
    atomicOr(&g_diag_status, CONV_STATUS_WAIT_SELFTEST);
}

}  // namespace

cudaError_t run_wait_selftest(unsigned max_sleeps, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(max_sleeps);
    return cudaGetLastError();
}

cudaError_t diag_read_status(unsigned* out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_diag_status, sizeof(unsigned));
    if (e == cudaSuccess && reset) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbol(g_diag_status, &zero, sizeof(unsigned));
    }
    return e;
}

}  // namespace igc
