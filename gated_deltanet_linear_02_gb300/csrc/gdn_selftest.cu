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
cudaError_t take_selftest_error(unsigned int *word, cudaStream_t s)
{
    unsigned int zero = 0;
    cudaError_t e =
        cudaMemcpyFromSymbolAsync(word, g_selftest_error, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && *word != 0)
        e = cudaMemcpyToSymbolAsync(g_selftest_error, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace gdn
