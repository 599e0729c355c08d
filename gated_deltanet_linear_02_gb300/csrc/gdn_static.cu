// gdn_static.cu -- gdn_prefill_static: gdn_prefill with its scratch memory
// taken from a fixed, file-scope device array instead of a caller-provided
// workspace.
//
// Some callers cannot allocate device memory at the point where they run a
// prefill. Examples: code inside a framework that owns every device
// allocation, plugins that receive only input and output buffers, and serving
// loops that forbid allocation after start-up. This entry point needs no
// workspace argument. It runs the same kernels as gdn_prefill, with
// GDN_STATIC_SCRATCH_BYTES of device memory that the library reserves once per
// device when it is loaded.
//
// In host code the symbol g_prefill_scratch is only a host-side stand-in, not a
// device address. So on each device's first call this file asks the runtime
// for the array's device address (cudaGetSymbolAddress, with that device
// current), caches it, and passes that address to the kernels.
#include <mutex>
#include <stdio.h>

#include "gdn_common.cuh"

namespace {

__device__ __align__(256) unsigned char g_prefill_scratch[GDN_STATIC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void *g_scratch_dev[MAX_DEVICES] = {nullptr};

}  // namespace

namespace gdn {
void record_error(const char *msg);   // sets the text gdn_last_error() returns
}

extern "C" gdn_status gdn_prefill_static(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                                         const void *beta, const int32_t *cu_seqlens, int N, int T_total,
                                         const void *conv_state_in, void *conv_state_out,
                                         const float *ssm_state_in, float *ssm_state_out, void *out,
                                         gdn_dtype act, gdn_dtype out_dt, int chunk_size, void *stream)
{
    const size_t need = gdn_prefill_workspace_size(N, T_total, act, chunk_size);
    // Nothing to run, or arguments gdn_prefill rejects on their own: it reports
    // them (with the same status and message as a direct call) without touching
    // CUDA. So does a call with a null or misaligned pointer, which gdn_prefill
    // checks before it looks at the workspace below.
    if (N == 0 || need == 0)
        return gdn_prefill(p, qkv, z, alpha, beta, cu_seqlens, N, T_total, conv_state_in, conv_state_out,
                           ssm_state_in, ssm_state_out, out, act, out_dt, chunk_size, nullptr, 0, stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        gdn::record_error("gdn_prefill_static: no current CUDA device");
        return GDN_ERR_CUDA;
    }
    void *scratch = nullptr;
    {
        // The address is looked up once per device and kept for the life of the
        // process. It assumes the device's primary context is never reset
        // (cudaDeviceReset): after a reset the array has a new address.
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_scratch_dev[dev] == nullptr) {
            void *ptr = nullptr;
            const cudaError_t e = cudaGetSymbolAddress(&ptr, g_prefill_scratch);
            if (e != cudaSuccess || ptr == nullptr) {
                char msg[256];
                snprintf(msg, sizeof(msg), "gdn_prefill_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
                gdn::record_error(msg);
                return GDN_ERR_CUDA;
            }
            g_scratch_dev[dev] = ptr;
        }
        scratch = g_scratch_dev[dev];
    }
    // gdn_prefill validates every argument first, then the scratch size: the
    // chunked form runs in windows sized to the scratch, the exact scan needs
    // room for all of its tokens. The kernels write every scratch byte they
    // later read, so stale contents from the previous call need no clearing.
    return gdn_prefill(p, qkv, z, alpha, beta, cu_seqlens, N, T_total, conv_state_in, conv_state_out, ssm_state_in,
                       ssm_state_out, out, act, out_dt, chunk_size, scratch, (size_t)GDN_STATIC_SCRATCH_BYTES,
                       stream);
}

extern "C" size_t gdn_static_scratch_bytes(void) { return (size_t)GDN_STATIC_SCRATCH_BYTES; }
