// gdn_decode_multi.cu -- a short run of T consecutive tokens (1 <= T <= 8) for
// each of B independent sequences, in one sweep over the states.
//
// This is the step between single-token decode and chunked prefill: a short
// suffix per sequence, such as the draft tokens of a speculative step. The
// mixer is the SSM block of "qwen35moe -- Forward-Pass Design (Pantheon port)"
// (sections "Causal conv1d", "Decay gate", "Per-token recurrence", "Output
// path"), applied to the T tokens in order. Run token by token, the state would
// cross HBM 2T times. Here every 128x128 state row is read once, takes its T
// updates in registers and is written once, so the state bytes per token fall
// by a factor of T.
//
// Structure. One persistent CTA per SM with 16 warps streams the states
// through six 32 KiB shared-memory slots with TMA bulk copies, a full mbarrier
// per slot. There is no producer warp: the last warp to release a slot (a
// shared counter per slot) issues the copy of the unit that goes there next,
// which keeps the CTA at 512 threads and so 128 registers a thread. An item is
// (sequence b, K-head kh) with both V-heads kh and kh + 16. In an
// item's prologue each thread convolves one channel over the window
// [conv_state (3 rows), x_0 .. x_{T-1}] and shifts T rows into conv_state. The
// q and k rows are L2-normalised per token, and the gates come per token and
// V-head. In the sweep, lanes 8r..8r+7 of a warp hold state row r (16 keys
// each) of both halves of a state (rows r' and 64 + r' of the two slots of
// one head), so that each k and q load of a token serves two rows. The warp's
// rows apply tokens 0..T-1 in order: decay, pred, delta, write, read. The output stage applies the gated RMSNorm per token.
#include "gdn_async.cuh"
#include "gdn_common.cuh"

namespace gdn {

__device__ unsigned int g_multi_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

constexpr int MT_MAX = GDN_DECODE_MAX_T;                    // tokens per sequence, at most
// The kernel is instantiated for a token capacity MT of 4 or 8: a call with
// T <= 4 takes the smaller one, whose per-token arrays use fewer registers.
constexpr int MD_WARPS = 16;
constexpr int MD_THREADS = 32 * MD_WARPS;
constexpr int MD_SLOT_ROWS = 64;                            // rows j of S^T per staging slot
constexpr int MD_UNITS = DV / MD_SLOT_ROWS;                 // slots per state (2)
constexpr int MD_SLOTS = 6;
constexpr uint32_t MD_SLOT_BYTES = MD_SLOT_ROWS * DK * sizeof(float);   // 32 KiB
static_assert(MD_SLOT_ROWS / MD_WARPS == 4, "a warp computes 4 rows of a slot at once, 8 lanes per row");

struct MultiArgs {
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    float norm_eps, l2_eps;
    const void *qkv, *z, *alpha, *beta;   // [B][T][...]
    void *conv_state;
    float *ssm_state;
    void *out;                            // [B][T][4096]
    int n_items;                          // B * 16
    int T;
};

template <int MT>
struct MultiSmem {
    alignas(128) float slot[MD_SLOTS][MD_SLOT_ROWS * DK];   // TMA destinations
    alignas(16) float q[MT][DK];                     // L2-normalised q of each token (float4 reads)
    alignas(16) float k[MT][DK];
    alignas(16) float v[MT][2][DV];
    alignas(16) float y[MT][2][DV];
    alignas(8) uint64_t full[MD_SLOTS];
    int released[MD_SLOTS];                          // warps done with the slot's current unit
    float red[MT][8];                                // per token: q sums (warps 0..3), k sums (4..7)
    float ored[MT][8];                               // per token: y^2 sums of head 0 (warps 0..3), head 1 (4..7)
    float gate[MT][2][2];                            // per token and V-head: decay exp(g), beta
    int pending[MD_SLOTS];
    int abort;
};
template <int MT>
constexpr size_t md_smem() { return sizeof(MultiSmem<MT>) + 128; }
static_assert(md_smem<MT_MAX>() <= 232448, "decode_multi shared memory");

// Loads unit u (u = (2 m + h) * MD_UNITS + part) of this CTA into slot u % MD_SLOTS.
// Caller: one thread; the unit's item exists and the slot is free.
template <int MT>
__device__ __forceinline__ void multi_issue_load(MultiSmem<MT> &sm, const MultiArgs &a, int u)
{
    const int item = blockIdx.x + (u / (2 * MD_UNITS)) * gridDim.x;
    const int h = (u / MD_UNITS) & 1, part = u % MD_UNITS;
    const int b = item / HK, kh = item % HK, vh = kh + HK * h;
    const char *src = reinterpret_cast<const char *>(a.ssm_state + ((size_t)b * HV + vh) * (DV * DK)) +
                      (size_t)part * MD_SLOT_BYTES;
    const int slot = u % MD_SLOTS;
    sm.pending[slot] = u;
    const uint32_t bar = smem_u32(&sm.full[slot]);
    const uint32_t dst = smem_u32(sm.slot[slot]);
    mbar_arrive_expect_tx(bar, MD_SLOT_BYTES);
    bulk_g2s(dst, src, MD_SLOT_BYTES / 2, bar);
    bulk_g2s(dst + MD_SLOT_BYTES / 2, src + MD_SLOT_BYTES / 2, MD_SLOT_BYTES / 2, bar);
}

// conv channel of thread tid within item (., kh): q | k of K-head kh, v of vh = kh, v of vh = kh + 16
__device__ __forceinline__ int multi_channel(int kh, int tid)
{
    if (tid < 128) return Q_OFF + kh * DK + tid;
    if (tid < 256) return K_OFF + kh * DK + (tid - 128);
    if (tid < 384) return V_OFF + kh * DV + (tid - 256);
    return V_OFF + (kh + HK) * DV + (tid - 384);
}

// An item's global prologue inputs held by thread tid, loaded one item ahead:
// its channel's conv_state rows, its T inputs and taps; for tid < 256 the z of
// output column (V-head kh + 16 (tid >> 7), j = tid & 127) of every token; for
// tid < 2T the gate inputs of token tid >> 1 and V-head kh + 16 (tid & 1).
template <typename TA, int MT> struct MultiIn {
    TA s[KC - 1];
    TA x[MT];
    TA zc[MT];
    TA al, be;
    float4 w;
    float A_log, dt_bias;
};

template <typename TA, int MT>
__device__ __forceinline__ MultiIn<TA, MT> multi_load(const MultiArgs &a, int item, int tid)
{
    MultiIn<TA, MT> p;
    const size_t b = item / HK;
    const int kh = item % HK, T = a.T;
    const int c = multi_channel(kh, tid);
    const TA *x = static_cast<const TA *>(a.qkv) + b * (size_t)T * CC;
    const TA *cs = static_cast<const TA *>(a.conv_state) + b * (size_t)(KC - 1) * CC;
    p.w = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + c);
#pragma unroll
    for (int r = 0; r < KC - 1; ++r) p.s[r] = cs[(size_t)r * CC + c];
#pragma unroll
    for (int t = 0; t < MT; ++t) p.x[t] = t < T ? x[(size_t)t * CC + c] : from_f<TA>(0.0f);
    const TA *zb = static_cast<const TA *>(a.z) + b * (size_t)T * DI + (size_t)(kh + HK * (tid >> 7)) * DV + (tid & 127);
#pragma unroll
    for (int t = 0; t < MT; ++t) p.zc[t] = (tid < 2 * DV && t < T) ? zb[(size_t)t * DI] : from_f<TA>(0.0f);
    p.al = p.be = from_f<TA>(0.0f);
    p.A_log = p.dt_bias = 0.0f;
    if (tid < 2 * T) {
        const int t = tid >> 1, vh = kh + HK * (tid & 1);
        p.al = static_cast<const TA *>(a.alpha)[(b * T + t) * HV + vh];
        p.be = static_cast<const TA *>(a.beta)[(b * T + t) * HV + vh];
        p.A_log = a.A_log[vh];
        p.dt_bias = a.dt_bias[vh];
    }
    return p;
}

__device__ __forceinline__ void multi_sync() { __syncthreads(); }

template <int MT>
__device__ __forceinline__ bool multi_unit_exists(const MultiArgs &a, int u)
{
    return blockIdx.x + (u / (2 * MD_UNITS)) * (int)gridDim.x < a.n_items;
}

// Lane 0 of a warp that has finished reading unit u in slot u % MD_SLOTS. The
// sixteenth warp to get here frees the slot and loads unit u + MD_SLOTS into it.
// The fences order every warp's reads of the slot before the counter updates,
// and the last update before the copy, which the proxy fence hands to TMA.
template <int MT>
__device__ __forceinline__ void multi_release(MultiSmem<MT> &sm, const MultiArgs &a, int u)
{
    const int slot = u % MD_SLOTS;
    __threadfence_block();
    if (atomicAdd(&sm.released[slot], 1) != MD_WARPS - 1) return;
    __threadfence_block();
    sm.released[slot] = 0;
    sm.pending[slot] = -1;
    const int nu = u + MD_SLOTS;
    if (sm.abort || !multi_unit_exists<MT>(a, nu)) return;
    fence_proxy_async_smem();
    multi_issue_load(sm, a, nu);
}

template <typename TA, typename TO, int MT>
__global__ void __launch_bounds__(MD_THREADS, 1) decode_multi_kernel(const MultiArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    MultiSmem<MT> &sm = *reinterpret_cast<MultiSmem<MT> *>(smem_aligned128(smem_raw));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int T = a.T;
    const volatile int &aborted = sm.abort;

    if (tid == 0) {
        for (int i = 0; i < MD_SLOTS; ++i) {
            mbar_init(smem_u32(&sm.full[i]), 1);
            sm.released[i] = 0;
            sm.pending[i] = -1;
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_wait();                                   // inputs and states may come from the kernel ahead
    grid_dep_launch();

    if (tid == 0)                                      // the first MD_SLOTS units
        for (int u = 0; u < MD_SLOTS && multi_unit_exists<MT>(a, u); ++u) multi_issue_load(sm, a, u);

    const float scale = rsqrtf((float)DK);
    MultiIn<TA, MT> pin;
    if ((int)blockIdx.x < a.n_items) pin = multi_load<TA, MT>(a, blockIdx.x, tid);
    for (int m = 0;; ++m) {
        const int item = blockIdx.x + m * gridDim.x;
        if (item >= a.n_items) break;
        const size_t b = item / HK;
        const int kh = item % HK;

        // ---- prologue: conv + SiLU of the item's 512 channels for each token,
        //      conv_state shifted by T rows, L2 norms per token, gates per token
        {
            TA *cs = static_cast<TA *>(a.conv_state) + b * (size_t)(KC - 1) * CC;
            const int c = multi_channel(kh, tid);
            float win[MT + KC - 1];                      // raw inputs, oldest first
#pragma unroll
            for (int r = 0; r < KC - 1; ++r) win[r] = to_f(pin.s[r]);
#pragma unroll
            for (int t = 0; t < MT; ++t) win[KC - 1 + t] = to_f(pin.x[t]);
            float xh[MT];
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= T) break;
                xh[t] = silu_f(pin.w.x * win[t] + pin.w.y * win[t + 1] + pin.w.z * win[t + 2] + pin.w.w * win[t + 3]);
            }
            // new conv_state: the last three raw inputs, rows T .. T+2 of the window,
            // shifted in token by token (static indices keep the inputs in registers)
            TA ns[KC - 1];
#pragma unroll
            for (int r = 0; r < KC - 1; ++r) ns[r] = pin.s[r];
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t < T) {
#pragma unroll
                    for (int r = 0; r < KC - 2; ++r) ns[r] = ns[r + 1];
                    ns[KC - 2] = pin.x[t];
                }
            }
#pragma unroll
            for (int r = 0; r < KC - 1; ++r) cs[(size_t)r * CC + c] = ns[r];   // this CTA owns channel c of sequence b
            if (tid < 256) {
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    if (t >= T) break;
                    const float ss = warp_sum(xh[t] * xh[t]);
                    if (lane == 0) sm.red[t][warp] = ss;
                }
            }
            if (tid < 2 * T) {
                float ga, gb;
                gates_f(pin.A_log, pin.dt_bias, to_f(pin.al), to_f(pin.be), ga, gb);
                sm.gate[tid >> 1][tid & 1][0] = ga;
                sm.gate[tid >> 1][tid & 1][1] = gb;
            }
            multi_sync();
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= T) break;
                if (tid < 128)
                    sm.q[t][tid] = xh[t] * rsqrtf(sm.red[t][0] + sm.red[t][1] + sm.red[t][2] + sm.red[t][3] + a.l2_eps);
                else if (tid < 256)
                    sm.k[t][tid - 128] =
                        xh[t] * rsqrtf(sm.red[t][4] + sm.red[t][5] + sm.red[t][6] + sm.red[t][7] + a.l2_eps);
                else
                    sm.v[t][(tid - 256) >> 7][tid & 127] = xh[t];
            }
            multi_sync();
        }
        TA zcur[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) zcur[t] = pin.zc[t];
        if (item + (int)gridDim.x < a.n_items) pin = multi_load<TA, MT>(a, item + gridDim.x, tid);

        // ---- the two states: each row takes tokens 0..T-1 in order
        // Each lane group holds two rows of one head, row jl of part 0 and of
        // part 1, so that every k and q load of a token serves both.
        const int rr = lane >> 3, g = lane & 7;         // row of the warp's four; float4 group within it
        static_assert(MD_UNITS == 2, "a head is two slots");
        for (int h = 0; h < 2; ++h) {
            const int u0 = 2 * MD_UNITS * m + MD_UNITS * h;   // units u0 (rows 0..63), u0 + 1 (rows 64..127)
            const int s0 = u0 % MD_SLOTS, s1 = (u0 + 1) % MD_SLOTS;
            if (aborted) continue;                       // skip the work, keep the barriers in step
            if (!mbar_wait_bounded(smem_u32(&sm.full[s0]), (uint32_t)((u0 / MD_SLOTS) & 1)) ||
                !mbar_wait_bounded(smem_u32(&sm.full[s1]), (uint32_t)(((u0 + 1) / MD_SLOTS) & 1))) {
                sm.abort = 1;
                continue;
            }
            const int vh = kh + HK * h;
            float *Sg = a.ssm_state + (b * HV + vh) * (size_t)(DV * DK);
            const int jl = warp * 4 + rr;                // row within each slot
            const int j0 = jl, j1 = MD_SLOT_ROWS + jl;
            const float4 *src0 = reinterpret_cast<const float4 *>(sm.slot[s0]) + jl * (DK / 4) + g;
            const float4 *src1 = reinterpret_cast<const float4 *>(sm.slot[s1]) + jl * (DK / 4) + g;
            float4 st0[4], st1[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                st0[c] = src0[8 * c];
                st1[c] = src1[8 * c];
            }
            __syncwarp();                                // the rows are in registers: free both slots
            if (lane == 0) {
                multi_release(sm, a, u0);
                multi_release(sm, a, u0 + 1);
            }
            for (int t = 0; t < T; ++t) {
                const float dec = sm.gate[t][h][0], beta = sm.gate[t][h][1];
                const float4 *k4 = reinterpret_cast<const float4 *>(sm.k[t]) + g;
                float pa0 = 0.0f, pb0 = 0.0f, pa1 = 0.0f, pb1 = 0.0f;
                float4 kk[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    kk[c] = k4[8 * c];
                    st0[c].x *= dec; st0[c].y *= dec; st0[c].z *= dec; st0[c].w *= dec;             // (a)
                    st1[c].x *= dec; st1[c].y *= dec; st1[c].z *= dec; st1[c].w *= dec;
                    pa0 = fmaf(st0[c].x, kk[c].x, fmaf(st0[c].y, kk[c].y, pa0));
                    pb0 = fmaf(st0[c].z, kk[c].z, fmaf(st0[c].w, kk[c].w, pb0));
                    pa1 = fmaf(st1[c].x, kk[c].x, fmaf(st1[c].y, kk[c].y, pa1));
                    pb1 = fmaf(st1[c].z, kk[c].z, fmaf(st1[c].w, kk[c].w, pb1));
                }
                const float pred0 = group_sum<8>(pa0 + pb0), pred1 = group_sum<8>(pa1 + pb1);         // (b)
                const float d0 = (sm.v[t][h][j0] - pred0) * beta, d1 = (sm.v[t][h][j1] - pred1) * beta;
                const float4 *q4 = reinterpret_cast<const float4 *>(sm.q[t]) + g;
                float ya0 = 0.0f, yb0 = 0.0f, ya1 = 0.0f, yb1 = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 qq = q4[8 * c];
                    st0[c].x = fmaf(kk[c].x, d0, st0[c].x); st0[c].y = fmaf(kk[c].y, d0, st0[c].y);   // (c)
                    st0[c].z = fmaf(kk[c].z, d0, st0[c].z); st0[c].w = fmaf(kk[c].w, d0, st0[c].w);
                    st1[c].x = fmaf(kk[c].x, d1, st1[c].x); st1[c].y = fmaf(kk[c].y, d1, st1[c].y);
                    st1[c].z = fmaf(kk[c].z, d1, st1[c].z); st1[c].w = fmaf(kk[c].w, d1, st1[c].w);
                    ya0 = fmaf(st0[c].x, qq.x, fmaf(st0[c].y, qq.y, ya0));
                    yb0 = fmaf(st0[c].z, qq.z, fmaf(st0[c].w, qq.w, yb0));
                    ya1 = fmaf(st1[c].x, qq.x, fmaf(st1[c].y, qq.y, ya1));
                    yb1 = fmaf(st1[c].z, qq.z, fmaf(st1[c].w, qq.w, yb1));
                }
                const float y0 = group_sum<8>(ya0 + yb0), y1 = group_sum<8>(ya1 + yb1);                 // (d)
                if (g == 0) {
                    sm.y[t][h][j0] = y0 * scale;
                    sm.y[t][h][j1] = y1 * scale;
                }
            }
            float4 *dst0 = reinterpret_cast<float4 *>(Sg + (size_t)j0 * DK) + g;
            float4 *dst1 = reinterpret_cast<float4 *>(Sg + (size_t)j1 * DK) + g;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                __stcs(dst0 + 8 * c, st0[c]);
                __stcs(dst1 + 8 * c, st1[c]);
            }
        }
        multi_sync();                                    // all rows of y are in, and the abort flag agrees
        if (aborted) break;

        // ---- gated RMSNorm of both heads for every token, times silu(z) ("Output path")
        if (tid < 256) {
            const int h = tid >> 7, j = tid & 127;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= T) break;
                const float yv = sm.y[t][h][j];
                const float ss = warp_sum(yv * yv);
                if (lane == 0) sm.ored[t][warp] = ss;
            }
        }
        multi_sync();
        if (tid < 256) {
            const int h = tid >> 7, j = tid & 127;
            const float nw = a.norm_w[j];
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                if (t >= T) break;
                const float *r4 = sm.ored[t] + 4 * h;
                const float rr2 = rsqrtf((r4[0] + r4[1] + r4[2] + r4[3]) * (1.0f / DV) + a.norm_eps);
                const size_t o = (b * T + t) * (size_t)DI + (size_t)(kh + HK * h) * DV + j;
                static_cast<TO *>(a.out)[o] = from_f<TO>(sm.y[t][h][j] * rr2 * nw * silu_f(to_f(zcur[t])));
            }
        }
        // the next prologue writes q/k/v/red/gate, none of which the lines above read
    }
    if (aborted && tid == 0) atomicExch(&g_multi_error, (unsigned int)GDN_ERR_TIMEOUT);
    multi_sync();                                        // no release is still running
    if (aborted && tid == 0)   // let the copies still in flight land before shared memory is released
        for (int i = 0; i < MD_SLOTS; ++i)
            if (sm.pending[i] >= 0) mbar_wait_bounded(smem_u32(&sm.full[i]), (uint32_t)((sm.pending[i] / MD_SLOTS) & 1));
}

int sm_count();

template <typename TA, typename TO, int MT>
static cudaError_t launch_multi_mt(const MultiArgs &a, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(decode_multi_kernel<TA, TO, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)md_smem<MT>());
    if (e != cudaSuccess) return e;
    const int n_sm = sm_count();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    const int grid = a.n_items < n_sm ? a.n_items : n_sm;
    return launch_pdl(decode_multi_kernel<TA, TO, MT>, dim3(grid), dim3(MD_THREADS), md_smem<MT>(), s, a);
}

template <typename TA, typename TO>
static cudaError_t launch_multi_t(const MultiArgs &a, cudaStream_t s)
{
    return a.T <= 4 ? launch_multi_mt<TA, TO, 4>(a, s) : launch_multi_mt<TA, TO, MT_MAX>(a, s);
}

cudaError_t launch_decode_multi(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                                const void *beta, void *conv_state, float *ssm_state, void *out, int B, int T,
                                gdn_dtype act, gdn_dtype out_dt, cudaStream_t s)
{
    MultiArgs a;
    a.conv_w = p->conv_w; a.A_log = p->A_log; a.dt_bias = p->dt_bias; a.norm_w = p->norm_w;
    a.norm_eps = p->norm_eps; a.l2_eps = p->l2_eps;
    a.qkv = qkv; a.z = z; a.alpha = alpha; a.beta = beta;
    a.conv_state = conv_state; a.ssm_state = ssm_state; a.out = out;
    a.n_items = B * HK;
    a.T = T;
    if (act == GDN_F32)
        return out_dt == GDN_F32 ? launch_multi_t<float, float>(a, s) : launch_multi_t<float, bf16>(a, s);
    return out_dt == GDN_F32 ? launch_multi_t<bf16, float>(a, s) : launch_multi_t<bf16, bf16>(a, s);
}

// Reads and clears this file's device error word (synchronous on `s`).
cudaError_t take_multi_error(unsigned int *word, cudaStream_t s)
{
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_multi_error, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && *word != 0)
        e = cudaMemcpyToSymbolAsync(g_multi_error, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace gdn
