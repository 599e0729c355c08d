// gdn_scan.cu -- exact per-token prefill (chunk_size 1): packed varlen
// sequences through the SSM block of "qwen35moe -- Forward-Pass Design
// (Pantheon port)", with every step in fp32.
//
// There are four launches, ordered on one stream:
//   1. prep:      one CTA per token. It runs the causal conv and SiLU over all
//                 8192 channels, using the sequence's own conv_state for the
//                 first three positions. It L2-normalises q and k per head, and
//                 computes the gates a = exp(g) and beta for the 32 V-heads.
//                 Results go to the workspace as fp32.
//   2. scan:      one CTA per (sequence, V-head, block of 32 value rows j). It
//                 walks the tokens in order and keeps its 32 rows of S^T in
//                 registers for the whole sequence. Each warp owns 4 rows and
//                 each lane holds 4 keys per row, so pred and y are warp-shuffle
//                 dot products. The state is read once and written once.
//   3. norm:      one CTA per token. It applies the gated RMSNorm with silu(z)
//                 per V-head and writes out.
//   4. conv out:  the last three raw inputs of each sequence, taken from its
//                 tail or from conv_state_in, become conv_state_out.
// Kernel 4 runs last, so conv_state_out may alias conv_state_in.
#include "gdn_async.cuh"
#include "gdn_common.cuh"

namespace gdn {

struct ScanWs {          // carve-up of the workspace, per token row
    float *x;            // [T][8192]: q^ | k^ (L2-normalised) | v (after SiLU)
    float *g;            // [T][32][2]: a = exp(g), beta
    float *y;            // [T][4096]: y before the gated norm (scale applied)
};

constexpr size_t SCAN_BYTES_PER_TOKEN = sizeof(float) * ((size_t)CC + 2 * HV + DI);

// cu_seqlens entry clamped into [lo, hi]: a malformed table then only
// garbles the offending sequences and never sends an index out of bounds.
__device__ __forceinline__ int cu_at(const int32_t *__restrict__ cu, int i, int lo, int hi)
{
    return min(max(__ldg(cu + i), lo), hi);
}

// Sequence that owns packed row t: the n with cu[n] <= t < cu[n+1].
__device__ __forceinline__ int seq_of_row(const int32_t *__restrict__ cu, int N, int t)
{
    int lo = 0, hi = N;   // invariant: cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
    }
    return lo;
}

template <typename TA> struct Vec8;   // 8 activations in one or two 16-byte loads
template <> struct Vec8<float> {
    static __device__ __forceinline__ void load(const float *p, float v[8])
    {
        const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};
template <> struct Vec8<bf16> {
    static __device__ __forceinline__ void load(const bf16 *p, float v[8])
    {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const bf16 *h = reinterpret_cast<const bf16 *>(&u);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __bfloat162float(h[e]);
    }
};

// ------------------------------------------------------------------ 1. prep
// 256 threads x 32 channels; thread th owns channels [32th, 32th+32), so one
// 128-channel head spans 4 consecutive lanes.
template <typename TA>
__global__ void __launch_bounds__(256) scan_prep_kernel(
    const float *__restrict__ conv_w, const float *__restrict__ A_log, const float *__restrict__ dt_bias,
    float l2_eps, const TA *__restrict__ qkv, const TA *__restrict__ alpha, const TA *__restrict__ beta,
    const int32_t *__restrict__ cu, int N, const TA *__restrict__ conv_state_in, ScanWs ws)
{
    const int t = blockIdx.x;
    const int th = threadIdx.x;
    const int n = seq_of_row(cu, N, t);
    const int start = cu_at(cu, n, 0, t);
    const int pos = t - start;   // position inside the sequence

    float xh[32];
    float ss = 0.0f;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        const int c0 = th * 32 + blk * 8;
        float win[4][8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {        // window element m is position pos - 3 + m
            const int pp = pos - 3 + m;
            if (pp >= 0) {
                Vec8<TA>::load(qkv + (size_t)(start + pp) * CC + c0, win[m]);
            } else if (conv_state_in != nullptr) {
                Vec8<TA>::load(conv_state_in + ((size_t)n * (KC - 1) + (pp + 3)) * CC + c0, win[m]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) win[m][e] = 0.0f;
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 w = __ldg(reinterpret_cast<const float4 *>(conv_w) + c0 + e);
            const float u = w.x * win[0][e] + w.y * win[1][e] + w.z * win[2][e] + w.w * win[3][e];
            const float v = silu_f(u);
            xh[blk * 8 + e] = v;
            ss += v * v;
        }
    }
    // L2 norm of q and k heads (threads 0..127); v (threads 128..255) stays as is.
    ss = group_sum<4>(ss);
    const float inv = (th < 2 * HK * DK / 32) ? rsqrtf(ss + l2_eps) : 1.0f;
    float *dst = ws.x + (size_t)t * CC + th * 32;
#pragma unroll
    for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4 *>(dst + e) =
            make_float4(xh[e] * inv, xh[e + 1] * inv, xh[e + 2] * inv, xh[e + 3] * inv);
    if (th < HV) {
        float ga, gb;
        gates_f(A_log[th], dt_bias[th], to_f(alpha[(size_t)t * HV + th]), to_f(beta[(size_t)t * HV + th]),
                ga, gb);
        ws.g[((size_t)t * HV + th) * 2 + 0] = ga;
        ws.g[((size_t)t * HV + th) * 2 + 1] = gb;
    }
}

// ------------------------------------------------------------------ 2. scan
constexpr int SCAN_ROWS_PER_CTA = 32;
constexpr int SCAN_ROWS_PER_WARP = 4;

__global__ void __launch_bounds__(256) scan_recurrence_kernel(const int32_t *__restrict__ cu, int T_total,
                                                              const float *__restrict__ S_in,
                                                              float *__restrict__ S_out, ScanWs ws)
{
    const int n = blockIdx.x, vh = blockIdx.y, kh = vh % HK;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j0 = blockIdx.z * SCAN_ROWS_PER_CTA + warp * SCAN_ROWS_PER_WARP;
    const size_t sbase = ((size_t)n * HV + vh) * (DV * DK);

    float4 st[SCAN_ROWS_PER_WARP];
#pragma unroll
    for (int r = 0; r < SCAN_ROWS_PER_WARP; ++r)
        st[r] = S_in ? __ldcs(reinterpret_cast<const float4 *>(S_in + sbase + (size_t)(j0 + r) * DK) + lane)
                     : make_float4(0.f, 0.f, 0.f, 0.f);

    const int t0 = cu_at(cu, n, 0, T_total), t1 = cu_at(cu, n + 1, t0, T_total);
    const float scale = rsqrtf((float)DK);

    // software pipeline: operands of token t+1 load while token t computes
    float4 k4, q4, nk4, nq4;
    float v[SCAN_ROWS_PER_WARP], nv[SCAN_ROWS_PER_WARP];
    float2 gt, ngt;
    auto load_tok = [&](int t, float4 &kk, float4 &qq, float *vv, float2 &gg) {
        const float *x = ws.x + (size_t)t * CC;
        kk = *reinterpret_cast<const float4 *>(x + K_OFF + kh * DK + lane * 4);
        qq = *reinterpret_cast<const float4 *>(x + Q_OFF + kh * DK + lane * 4);
#pragma unroll
        for (int r = 0; r < SCAN_ROWS_PER_WARP; ++r) vv[r] = x[V_OFF + vh * DV + j0 + r];
        gg = *reinterpret_cast<const float2 *>(ws.g + ((size_t)t * HV + vh) * 2);
    };
    if (t0 < t1) load_tok(t0, k4, q4, v, gt);
    for (int t = t0; t < t1; ++t) {
        if (t + 1 < t1) load_tok(t + 1, nk4, nq4, nv, ngt);
        const float dec = gt.x, beta = gt.y;
#pragma unroll
        for (int r = 0; r < SCAN_ROWS_PER_WARP; ++r) {
            float4 s = st[r];
            s.x *= dec; s.y *= dec; s.z *= dec; s.w *= dec;
            const float pred = warp_sum(s.x * k4.x + s.y * k4.y + s.z * k4.z + s.w * k4.w);
            const float delta = (v[r] - pred) * beta;
            s.x += k4.x * delta; s.y += k4.y * delta; s.z += k4.z * delta; s.w += k4.w * delta;
            const float yq = warp_sum(s.x * q4.x + s.y * q4.y + s.z * q4.z + s.w * q4.w);
            st[r] = s;
            if (lane == r) ws.y[(size_t)t * DI + vh * DV + j0 + r] = yq * scale;
        }
        k4 = nk4; q4 = nq4; gt = ngt;
#pragma unroll
        for (int r = 0; r < SCAN_ROWS_PER_WARP; ++r) v[r] = nv[r];
    }
    if (S_out) {
#pragma unroll
        for (int r = 0; r < SCAN_ROWS_PER_WARP; ++r)
            __stcs(reinterpret_cast<float4 *>(S_out + sbase + (size_t)(j0 + r) * DK) + lane, st[r]);
    }
}

// ------------------------------------------------------------------ 3. norm
// One CTA per token, 8 warps x 4 V-heads; lane l owns j in [4l, 4l+4).
template <typename TA, typename TO>
__global__ void __launch_bounds__(256) scan_norm_kernel(const float *__restrict__ norm_w, float norm_eps,
                                                        const TA *__restrict__ z, TO *__restrict__ out,
                                                        ScanWs ws)
{
    const size_t t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dep_wait();                                   // y comes from the kernel ahead
    grid_dep_launch();
    if (norm_w == nullptr) {                           // no norm weights: out is y itself
#pragma unroll
        for (int hh = 0; hh < HV / 8; ++hh) {
            const size_t o = t * DI + (warp * (HV / 8) + hh) * DV + lane * 4;
            store4(out + o, *reinterpret_cast<const float4 *>(ws.y + o));
        }
        return;
    }
    const float4 w = *reinterpret_cast<const float4 *>(norm_w + lane * 4);
#pragma unroll
    for (int hh = 0; hh < HV / 8; ++hh) {
        const int vh = warp * (HV / 8) + hh;
        const size_t o = t * DI + vh * DV + lane * 4;      // 4 consecutive elements: one vector access each
        const float4 y = *reinterpret_cast<const float4 *>(ws.y + o);
        const float4 zz = load4(z + o);
        const float ms = warp_sum(y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w) * (1.0f / DV);
        const float rr = rsqrtf(ms + norm_eps);
        store4(out + o, make_float4(y.x * rr * w.x * silu_f(zz.x), y.y * rr * w.y * silu_f(zz.y),
                                    y.z * rr * w.z * silu_f(zz.z), y.w * rr * w.w * silu_f(zz.w)));
    }
}

// ------------------------------------------------------------ 4. conv state
// conv_state_out[n][m] = raw input at sequence position L-3+m, or the old row
// (L-3+m)+3 of conv_state_in when that position is before the sequence start.
template <typename TA>
__global__ void __launch_bounds__(256) conv_state_out_kernel(const int32_t *__restrict__ cu, int T_total,
                                                             const TA *__restrict__ qkv,
                                                             const TA *cs_in, TA *cs_out)
{
    const int n = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    grid_dep_wait();                                   // cs_out may alias cs_in, which earlier kernels read
    const int start = cu_at(cu, n, 0, T_total), L = cu_at(cu, n + 1, start, T_total) - start;
    TA nv[KC - 1];
#pragma unroll
    for (int m = 0; m < KC - 1; ++m) {
        const int p = L - (KC - 1) + m;
        if (p >= 0) nv[m] = qkv[(size_t)(start + p) * CC + c];
        else nv[m] = cs_in ? cs_in[((size_t)n * (KC - 1) + (p + KC - 1)) * CC + c] : from_f<TA>(0.0f);
    }
#pragma unroll
    for (int m = 0; m < KC - 1; ++m) cs_out[((size_t)n * (KC - 1) + m) * CC + c] = nv[m];
}

// ----------------------------------------------------------------- launcher

size_t scan_workspace_bytes(int T_total) { return SCAN_BYTES_PER_TOKEN * (size_t)T_total; }

cudaError_t launch_prefill_scan(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                                const void *beta, const int32_t *cu, int N, int T_total,
                                const void *cs_in, void *cs_out, const float *S_in, float *S_out,
                                void *out, gdn_dtype act, gdn_dtype out_dt, void *ws_base,
                                cudaStream_t s)
{
    ScanWs ws;
    ws.x = static_cast<float *>(ws_base);
    ws.g = ws.x + (size_t)T_total * CC;
    ws.y = ws.g + (size_t)T_total * HV * 2;
    if (T_total > 0) {
        if (act == GDN_F32)
            scan_prep_kernel<float><<<T_total, 256, 0, s>>>(p->conv_w, p->A_log, p->dt_bias, p->l2_eps,
                                                            (const float *)qkv, (const float *)alpha,
                                                            (const float *)beta, cu, N,
                                                            (const float *)cs_in, ws);
        else
            scan_prep_kernel<bf16><<<T_total, 256, 0, s>>>(p->conv_w, p->A_log, p->dt_bias, p->l2_eps,
                                                           (const bf16 *)qkv, (const bf16 *)alpha,
                                                           (const bf16 *)beta, cu, N, (const bf16 *)cs_in,
                                                           ws);
    }
    scan_recurrence_kernel<<<dim3(N, HV, DV / SCAN_ROWS_PER_CTA), 256, 0, s>>>(cu, T_total, S_in, S_out, ws);
    if (T_total > 0) {
        if (act == GDN_F32) {
            if (out_dt == GDN_F32)
                scan_norm_kernel<float, float><<<T_total, 256, 0, s>>>(p->norm_w, p->norm_eps,
                                                                       (const float *)z, (float *)out, ws);
            else
                scan_norm_kernel<float, bf16><<<T_total, 256, 0, s>>>(p->norm_w, p->norm_eps,
                                                                      (const float *)z, (bf16 *)out, ws);
        } else {
            if (out_dt == GDN_F32)
                scan_norm_kernel<bf16, float><<<T_total, 256, 0, s>>>(p->norm_w, p->norm_eps,
                                                                      (const bf16 *)z, (float *)out, ws);
            else
                scan_norm_kernel<bf16, bf16><<<T_total, 256, 0, s>>>(p->norm_w, p->norm_eps,
                                                                     (const bf16 *)z, (bf16 *)out, ws);
        }
    }
    if (cs_out) {
        if (act == GDN_F32)
            conv_state_out_kernel<float><<<dim3(CC / 256, N), 256, 0, s>>>(cu, T_total, (const float *)qkv,
                                                                           (const float *)cs_in,
                                                                           (float *)cs_out);
        else
            conv_state_out_kernel<bf16><<<dim3(CC / 256, N), 256, 0, s>>>(cu, T_total, (const bf16 *)qkv,
                                                                          (const bf16 *)cs_in,
                                                                          (bf16 *)cs_out);
    }
    return cudaGetLastError();
}

}  // namespace gdn

namespace gdn {

// The gated RMSNorm . silu(z) over a [T][4096] fp32 buffer of y (scale
// applied), for the chunked path (bf16 activations).
// pdl: launched with programmatic stream serialization (the kernels wait for
// the kernel ahead before reading its results).
cudaError_t launch_gated_norm_bf16(const float *norm_w, float norm_eps, const void *z, const float *y, void *out,
                                   int T_total, gdn_dtype out_dt, cudaStream_t s, bool pdl)
{
    if (T_total <= 0) return cudaSuccess;
    ScanWs ws;
    ws.x = nullptr;
    ws.g = nullptr;
    ws.y = const_cast<float *>(y);
    const bf16 *zb = (const bf16 *)z;
    if (out_dt == GDN_F32) {
        if (pdl) return launch_pdl(scan_norm_kernel<bf16, float>, dim3(T_total), dim3(256), 0, s, norm_w, norm_eps, zb,
                                   (float *)out, ws);
        scan_norm_kernel<bf16, float><<<T_total, 256, 0, s>>>(norm_w, norm_eps, zb, (float *)out, ws);
    } else {
        if (pdl) return launch_pdl(scan_norm_kernel<bf16, bf16>, dim3(T_total), dim3(256), 0, s, norm_w, norm_eps, zb,
                                   (bf16 *)out, ws);
        scan_norm_kernel<bf16, bf16><<<T_total, 256, 0, s>>>(norm_w, norm_eps, zb, (bf16 *)out, ws);
    }
    return cudaGetLastError();
}

// conv_state_out for the chunked path (bf16 activations); same rule as above.
cudaError_t launch_conv_state_out_bf16(const int32_t *cu, int N, int T_total, const void *qkv, const void *cs_in,
                                       void *cs_out, cudaStream_t s, bool pdl)
{
    if (N <= 0) return cudaSuccess;
    if (pdl)
        return launch_pdl(conv_state_out_kernel<bf16>, dim3(CC / 256, N), dim3(256), 0, s, cu, T_total,
                          (const bf16 *)qkv, (const bf16 *)cs_in, (bf16 *)cs_out);
    conv_state_out_kernel<bf16><<<dim3(CC / 256, N), 256, 0, s>>>(cu, T_total, (const bf16 *)qkv,
                                                                  (const bf16 *)cs_in, (bf16 *)cs_out);
    return cudaGetLastError();
}

}  // namespace gdn
