// gdn_selftest.cu -- a diagnostic kernel for the library's failure path: it
// waits on an mbarrier that nothing ever completes, through the same bounded
// wait every pipelined kernel of libgdn uses. The wait gives up after its limit
// (2 s), the kernel records GDN_ERR_TIMEOUT in its device error word and
// returns normally, so the CUDA context stays usable and gdn_device_error
// reports the timeout. No fault, trap or unbounded loop is involved.
#include "gdn_async.cuh"
#include "gdn_common.cuh"

namespace gdn {

__device__ unsigned int g_selftest_error;

__global__ void __launch_bounds__(32) wait_timeout_kernel(int *waited_ok)
{
    __shared__ alignas(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);                  // one arrival expected; none ever comes
        fence_mbar_init();
    }
    __syncwarp();
    bool ok = true;
    if (threadIdx.x == 0) ok = mbar_wait_bounded(smem_u32(&bar), 0u);
    if (threadIdx.x == 0) {
        if (waited_ok) *waited_ok = ok ? 1 : 0;
        if (!ok) atomicExch(&g_selftest_error, (unsigned int)GDN_ERR_TIMEOUT);
    }
}

cudaError_t launch_wait_timeout(cudaStream_t s)
{
    wait_timeout_kernel<<<1, 32, 0, s>>>(nullptr);
    return cudaGetLastError();
}

// Reads and clears this file's device error word (synchronous on `s`).
// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *selftest_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_selftest_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
