// Test hook for the bounded waits of the pipelined kernels.
//
// Every mbarrier wait of the GEMMs gives up after a cycle budget, records bit 0
// of the workspace error word and lets the kernel unwind, so that a stalled
// pipeline becomes an error the host reads (w4a8_device_error) instead of a
// hung GPU. This kernel runs that wait on a barrier nothing ever completes,
// with a short budget, so tests can check the whole path on a real device and
// that the context stays usable afterwards.
#include "internal.h"
#include "ptx.cuh"

namespace w4a8 {

__global__ void __launch_bounds__(32) selftest_wait_timeout_kernel(uint32_t* err, long long budget)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait_for(smem_u32(&bar), 0, budget))
        set_error(err, kErrBitTimeout);
}

cudaError_t launch_selftest_wait_timeout(uint32_t* err, cudaStream_t s)
{
    // about 10 ms at the GPU's clock: the same loop the kernels run, cut short
    selftest_wait_timeout_kernel<<<1, 32, 0, s>>>(err, 20000000LL);
    return cudaGetLastError();
}

}  // namespace w4a8
