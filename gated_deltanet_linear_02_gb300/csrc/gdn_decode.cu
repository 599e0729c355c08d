// gdn_decode.cu -- single-token kernels: the conv step and the fused decode step.
//
// Decode is a batched, HBM-bound sweep over the fp32 states. Each 128x128
// state of one (sequence, V-head) is 64 KiB and makes up 97% of the bytes.
// So the kernel reads every state exactly once with 128-bit streaming loads,
// issued before anything else. It does every other step of the SSM block on
// chip while those loads are in flight, and writes the state back once. The
// SSM block is the one in "qwen35moe -- Forward-Pass Design (Pantheon port)",
// sections "Causal conv1d", "Decay gate", "Per-token recurrence" and "Output
// path".
//
// Work split: one CTA per (sequence, V-head), 256 threads. Warp w owns rows
// j in [16w, 16w+16) of S^T (value index j; each row is the 128 keys i,
// contiguous). Lane l holds keys [4l, 4l+4) of each of its rows in registers.
// All of pred_j, delta_j and y_j depend on row j alone, so the rows need no
// exchange, only warp-shuffle dot products.
//
// V-heads vh and vh+16 read the same q/k channels, because of the interleaved
// GQA repeat (V-head vh uses K-head vh % 16). Both CTAs must read those
// conv_state channels before one of them shifts the state. The two CTAs form
// a 2-CTA cluster for this: each arrives on the cluster barrier as soon as it
// has read, and waits on it only at its very end. Then the vh < 16 CTA writes
// the shared q/k rows. The v rows belong to one CTA and are written at once.
#include "gdn_common.cuh"

namespace gdn {

// ------------------------------------------------------------------ conv step

template <typename TA>
__global__ void __launch_bounds__(256) conv_step_kernel(const float *__restrict__ conv_w,
                                                        const TA *__restrict__ x_in,
                                                        TA *__restrict__ x_out,
                                                        TA *__restrict__ conv_state)
{
    const int c = blockIdx.x * blockDim.x + threadIdx.x;   // channel
    const size_t b = blockIdx.y;                           // sequence
    const float4 w = __ldg(reinterpret_cast<const float4 *>(conv_w) + c);
    TA *st = conv_state + b * (size_t)(KC - 1) * CC;
    const TA s0 = st[c], s1 = st[CC + c], s2 = st[2 * CC + c];
    const TA x = x_in[b * CC + c];
    const float u = w.x * to_f(s0) + w.y * to_f(s1) + w.z * to_f(s2) + w.w * to_f(x);
    x_out[b * CC + c] = from_f<TA>(silu_f(u));
    st[c] = s1;
    st[CC + c] = s2;
    st[2 * CC + c] = x;
}

// ---------------------------------------------------------------- decode step

struct DecodeArgs {
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    float norm_eps, l2_eps;
    const void *qkv, *z, *alpha, *beta;
    void *conv_state;
    float *ssm_state;
    void *out;
};

constexpr int DEC_THREADS = 256;
constexpr int DEC_ROWS_PER_WARP = DV / (DEC_THREADS / 32);   // 16

__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

template <typename TA, typename TO>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DEC_THREADS, 2)
decode_step_kernel(const DecodeArgs a)
{
    const int kh = blockIdx.x >> 1;          // K-head shared by the cluster pair
    const int half = blockIdx.x & 1;         // 0: vh = kh, 1: vh = kh + 16
    const int vh = kh + HK * half;
    const size_t b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // (1) Stream this warp's 16 state rows into registers first: 64 KiB per CTA
    //     in flight while the prologue below runs.
    float *S = a.ssm_state + (b * HV + vh) * (size_t)(DV * DK);
    float4 st[DEC_ROWS_PER_WARP];
#pragma unroll
    for (int r = 0; r < DEC_ROWS_PER_WARP; ++r)
        st[r] = __ldcs(reinterpret_cast<const float4 *>(S + (size_t)(warp * DEC_ROWS_PER_WARP + r) * DK) + lane);

    __shared__ float s_q[DK], s_k[DK], s_v[DV], s_y[DV];
    __shared__ float s_red[16];
    __shared__ float s_gate[2];

    // (2) Causal conv + SiLU ("Causal conv1d"): thread t convolves q channel t
    //     (t < 128) or k channel t-128 of K-head kh, and t < 128 also v channel t
    //     of V-head vh.
    const TA *x = static_cast<const TA *>(a.qkv) + b * CC;
    TA *cs = static_cast<TA *>(a.conv_state) + b * (size_t)(KC - 1) * CC;
    const int cA = (tid < DK) ? (Q_OFF + kh * DK + tid) : (K_OFF + kh * DK + tid - DK);
    const float4 wA = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + cA);
    const TA a0 = cs[cA], a1 = cs[CC + cA], a2 = cs[2 * CC + cA], ax = x[cA];
    const float xA = silu_f(wA.x * to_f(a0) + wA.y * to_f(a1) + wA.z * to_f(a2) + wA.w * to_f(ax));
    float xV = 0.0f;
    if (tid < DV) {
        const int cV = V_OFF + vh * DV + tid;
        const float4 wV = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + cV);
        const TA v0 = cs[cV], v1 = cs[CC + cV], v2 = cs[2 * CC + cV], vx = x[cV];
        xV = silu_f(wV.x * to_f(v0) + wV.y * to_f(v1) + wV.z * to_f(v2) + wV.w * to_f(vx));
        // v channels belong to this CTA alone: shift them now.
        cs[cV] = v1;
        cs[CC + cV] = v2;
        cs[2 * CC + cV] = vx;
    }
    // Our reads of the shared q/k conv_state are done (their values feed xA).
    cluster_arrive_release();

    // (3) L2 norms of q and k over the head dim ("L2-normalize q and k over head
    //     dim (not RMS)"): warps 0-3 hold q, warps 4-7 hold k.
    {
        const float ss = warp_sum(xA * xA);
        if (lane == 0) s_red[warp] = ss;
    }
    if (tid == 0) {
        const float al = to_f(static_cast<const TA *>(a.alpha)[b * HV + vh]);
        const float be = to_f(static_cast<const TA *>(a.beta)[b * HV + vh]);
        float ga, gb;
        gates_f(a.A_log[vh], a.dt_bias[vh], al, be, ga, gb);
        s_gate[0] = ga;
        s_gate[1] = gb;
    }
    __syncthreads();
    if (tid < DK) {
        const float inv = rsqrtf(s_red[0] + s_red[1] + s_red[2] + s_red[3] + a.l2_eps);
        s_q[tid] = xA * inv;
        s_v[tid] = xV;
    } else {
        const float inv = rsqrtf(s_red[4] + s_red[5] + s_red[6] + s_red[7] + a.l2_eps);
        s_k[tid - DK] = xA * inv;
    }
    __syncthreads();

    // (4) Recurrence (a)-(d) on this warp's rows; rows are independent.
    const float4 k4 = reinterpret_cast<const float4 *>(s_k)[lane];
    const float4 q4 = reinterpret_cast<const float4 *>(s_q)[lane];
    const float dec = s_gate[0], beta = s_gate[1];
    const float scale = rsqrtf((float)DK);
#pragma unroll
    for (int r = 0; r < DEC_ROWS_PER_WARP; ++r) {
        const int j = warp * DEC_ROWS_PER_WARP + r;
        float4 s = st[r];
        s.x *= dec; s.y *= dec; s.z *= dec; s.w *= dec;                       // (a)
        const float pred = warp_sum(s.x * k4.x + s.y * k4.y + s.z * k4.z + s.w * k4.w);   // (b)
        const float delta = (s_v[j] - pred) * beta;
        s.x += k4.x * delta; s.y += k4.y * delta; s.z += k4.z * delta; s.w += k4.w * delta;  // (c)
        const float yq = warp_sum(s.x * q4.x + s.y * q4.y + s.z * q4.z + s.w * q4.w);       // (d)
        __stcs(reinterpret_cast<float4 *>(S + (size_t)j * DK) + lane, s);
        if (lane == 0) s_y[j] = yq * scale;
    }
    __syncthreads();

    // (5) Gated RMSNorm over this head's 128 outputs, times silu(z) ("Output path").
    float y = 0.0f;
    if (tid < DV) {
        y = s_y[tid];
        const float ss = warp_sum(y * y);
        if (lane == 0) s_red[8 + warp] = ss;
    }
    __syncthreads();
    if (tid < DV) {
        const float ms = (s_red[8] + s_red[9] + s_red[10] + s_red[11]) * (1.0f / DV);
        const float rr = rsqrtf(ms + a.norm_eps);
        const float zz = to_f(static_cast<const TA *>(a.z)[b * DI + vh * DV + tid]);
        static_cast<TO *>(a.out)[b * DI + vh * DV + tid] = from_f<TO>(y * rr * a.norm_w[tid] * silu_f(zz));
    }

    // (6) Shift the shared q/k conv_state rows once both CTAs of the pair have read them.
    cluster_wait_acquire();
    if (half == 0) {
        cs[cA] = a1;
        cs[CC + cA] = a2;
        cs[2 * CC + cA] = ax;
    }
}

// ------------------------------------------------------------------ launchers

cudaError_t launch_conv_step(const float *conv_w, const void *x_in, void *x_out, void *conv_state,
                             int B, gdn_dtype act, cudaStream_t s)
{
    dim3 grid(CC / 256, B);
    if (act == GDN_F32)
        conv_step_kernel<float><<<grid, 256, 0, s>>>(conv_w, (const float *)x_in, (float *)x_out,
                                                     (float *)conv_state);
    else
        conv_step_kernel<bf16><<<grid, 256, 0, s>>>(conv_w, (const bf16 *)x_in, (bf16 *)x_out,
                                                    (bf16 *)conv_state);
    return cudaGetLastError();
}

cudaError_t launch_decode_step(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                               const void *beta, void *conv_state, float *ssm_state, void *out, int B,
                               gdn_dtype act, gdn_dtype out_dt, cudaStream_t s)
{
    DecodeArgs a;
    a.conv_w = p->conv_w; a.A_log = p->A_log; a.dt_bias = p->dt_bias; a.norm_w = p->norm_w;
    a.norm_eps = p->norm_eps; a.l2_eps = p->l2_eps;
    a.qkv = qkv; a.z = z; a.alpha = alpha; a.beta = beta;
    a.conv_state = conv_state; a.ssm_state = ssm_state; a.out = out;
    dim3 grid(HV, B);   // x = 2*kh + half; consecutive pairs form the clusters
    if (act == GDN_F32) {
        if (out_dt == GDN_F32) decode_step_kernel<float, float><<<grid, DEC_THREADS, 0, s>>>(a);
        else decode_step_kernel<float, bf16><<<grid, DEC_THREADS, 0, s>>>(a);
    } else {
        if (out_dt == GDN_F32) decode_step_kernel<bf16, float><<<grid, DEC_THREADS, 0, s>>>(a);
        else decode_step_kernel<bf16, bf16><<<grid, DEC_THREADS, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace gdn
