// gdn_common.cuh -- shared device helpers of libgdn (sm_103a).
//
// Dimensions are those of the SSM layers in "qwen35moe -- Forward-Pass Design
// (Pantheon port)", section "Config (mini)". The conv stream is laid out
// q (16 heads x 128) | k (16 x 128) | v (32 x 128), head-major.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/gdn.h"

namespace gdn {

constexpr int HV = GDN_NUM_V_HEADS;      // 32 value heads
constexpr int HK = GDN_NUM_K_HEADS;      // 16 key/query heads
constexpr int DK = GDN_HEAD_DIM;         // 128 key dim (rows of S)
constexpr int DV = GDN_HEAD_DIM;         // 128 value dim (columns of S)
constexpr int KC = GDN_CONV_K;           // conv width 4
constexpr int CC = GDN_CONV_CHANNELS;    // 8192 conv channels
constexpr int DI = GDN_D_INNER;          // 4096 = HV * DV
constexpr int Q_OFF = 0;                 // q channels [0, 2048)
constexpr int K_OFF = HK * DK;           // k channels [2048, 4096)
constexpr int V_OFF = 2 * HK * DK;       // v channels [4096, 8192)
static_assert(V_OFF + HV * DV == CC, "conv channel split");

typedef __nv_bfloat16 bf16;

__device__ __forceinline__ float to_f(float x) { return x; }
// bf16 -> fp32 is exact: a bf16 is the top half of the fp32 bit pattern, so
// the widening is a 16-bit shift on the integer pipe.
__device__ __forceinline__ float to_f(bf16 x) { return __uint_as_float((uint32_t)__bfloat16_as_ushort(x) << 16); }

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ bf16 from_f<bf16>(float x) { return __float2bfloat16_rn(x); }

// SiLU(x) = x * sigmoid(x) (the conv activation and the output gate silu(z)).
// 4 consecutive elements (8-byte aligned for bf16, 16-byte for fp32) as one
// vector load or store
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const bf16 *p)
{
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                       __uint_as_float(u.y & 0xFFFF0000u));
}
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(bf16 *p, float4 v)
{
    const uint32_t lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.x)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.y)) << 16);
    const uint32_t hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.z)) |
                        ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v.w)) << 16);
    *reinterpret_cast<uint2 *>(p) = make_uint2(lo, hi);
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// SiLU with the fast exponential and division intrinsics (a few ulp). Used only
// where the result becomes a tf32 tensor-core operand, whose rounding is about
// 1e3 times coarser.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

// softplus with a linear tail above 20, the same reading the oracle takes.
__device__ __forceinline__ float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Sum over aligned groups of `W` lanes (W a power of two <= 32).
template <int W> __device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Decay and beta gates of one (token, V-head), section "Decay gate":
// returns a = exp(g) with g = -exp(A_log) * softplus(alpha + dt_bias), and
// beta = sigmoid(beta_logit).
__device__ __forceinline__ void gates_f(float A_log, float dt_bias, float alpha, float beta_logit,
                                        float &a, float &b)
{
    const float g = -expf(A_log) * softplus_f(alpha + dt_bias);
    a = expf(g);
    b = 1.0f / (1.0f + expf(-beta_logit));
}

// Launches kernel<<<grid, block, smem, s>>>(args...) with programmatic stream
// serialization allowed: the kernel may start before the one ahead of it in the
// stream has finished, and must call grid_dep_wait() (gdn_async.cuh) before it
// touches that kernel's results.
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace gdn
