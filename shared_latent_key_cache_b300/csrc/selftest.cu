// selftest.cu -- li_selftest_wait_timeout: exercises, on the GPU, the bounded
// wait that every kernel of the library uses, without withholding work from a
// real kernel.
//
// One CTA allocates tensor memory, then waits on an mbarrier that nothing ever
// arrives on, through the same mbar_wait as the scan, absorption and top-k
// kernels.  When the limit runs out the wait latches LI_ERR_TIMEOUT in the
// device status word and returns; the CTA frees its tensor memory and exits,
// so the context stays usable.  Nothing faults, traps or hangs.
#include <cuda_runtime.h>

#include "li_internal.cuh"
#include "ptx.cuh"

namespace li {
namespace {

__global__ void __launch_bounds__(64, 1) selftest_wait_kernel(uint64_t limit_ns, int *status)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1u);
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 32u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();
    // phase 0 of `bar` never completes: this wait must give up after limit_ns
    const bool ok = mbar_wait(&bar, 0u, &abort_flag, status, limit_ns);
    (void)ok;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 32u);
    }
}

} // namespace
} // namespace li

extern "C" int li_selftest_wait_timeout(unsigned int limit_us, void *stream)
{
    if (limit_us == 0 || limit_us > 1000000u)
        return LI_ERR_INVALID_ARG;
    int *status = li::device_status_ptr();
    if (status == nullptr)
        return LI_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t limit_ns = static_cast<uint64_t>(limit_us) * 1000u;
    cudaError_t e = li::launch_pdl(li::selftest_wait_kernel, dim3(1), dim3(64), 0, s, limit_ns, status);
    return e == cudaSuccess ? LI_OK : LI_ERR_CUDA;
}
