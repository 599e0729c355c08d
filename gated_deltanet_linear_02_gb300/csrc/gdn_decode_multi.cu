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
// through six 32 KiB shared-memory slots, a full mbarrier per slot. There is
// no producer warp: the last warp to finish with a slot (a shared counter per
// slot) issues its copies, which keeps the CTA at 512 threads and so 128
// registers a thread. An item is (sequence b, K-head kh) with both V-heads kh
// and kh + 16. In an item's prologue each thread convolves one channel over the
// window [conv_state (3 rows), x_0 .. x_{T-1}] and shifts T rows into
// conv_state; then warp w L2-normalises q or k of one token, and the gates come
// per token and V-head. In the sweep, head h is one pass over its two slots:
// a group of 16 lanes holds four of its rows (8 keys a lane), so each k and q
// load of a token serves four rows, and applies tokens 0..T-1 in order: decay,
// pred, delta, write, read. The new rows go back into their slot, and a TMA
// bulk store drains the slot to HBM while the warps go on; one pass later,
// when the store has read the slot, the next unit is loaded there. The output stage gives warp w the
// gated RMSNorm of one (token, head) row.
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
static_assert(MD_SLOT_ROWS / MD_WARPS == 4, "a warp holds 4 rows of each slot, 16 lanes per row");

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
    int owed[MD_WARPS][2];                           // loads a warp owes (multi_release), -1 for none
    float gate[MT][2][3];                            // per token and V-head: decay exp(g), beta, 1 / exp(g)
    int pending[MD_SLOTS];
    int abort;
};
template <int MT>
constexpr size_t md_smem() { return sizeof(MultiSmem<MT>) + 128; }
static_assert(md_smem<MT_MAX>() <= 232448, "decode_multi shared memory");

// Loads unit u (u = (2 m + h) * MD_UNITS + part) of this CTA into slot u % MD_SLOTS.
// Caller: one thread; the unit's item exists and the slot is free.
// Rows [64 part, 64 part + 64) of the state of unit u.
__device__ __forceinline__ char *multi_unit_ptr(const MultiArgs &a, int u)
{
    const int item = blockIdx.x + (u / (2 * MD_UNITS)) * gridDim.x;
    const int h = (u / MD_UNITS) & 1, part = u % MD_UNITS;
    const int b = item / HK, kh = item % HK, vh = kh + HK * h;
    return reinterpret_cast<char *>(a.ssm_state + ((size_t)b * HV + vh) * (DV * DK)) + (size_t)part * MD_SLOT_BYTES;
}

template <int MT>
__device__ __forceinline__ void multi_issue_load(MultiSmem<MT> &sm, const MultiArgs &a, int u)
{
    const char *src = multi_unit_ptr(a, u);
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

// Four consecutive activations as loaded (converted only when used, so that a
// prefetch does not wait for its data).
template <typename TA> struct Raw4;
template <> struct Raw4<float> { using type = float4; };
template <> struct Raw4<bf16> { using type = uint2; };
__device__ __forceinline__ float4 raw4_f(float4 v) { return v; }
__device__ __forceinline__ float4 raw4_f(uint2 u) { return load4(reinterpret_cast<const bf16 *>(&u)); }

// An item's global prologue inputs held by thread tid, loaded one item ahead:
// its channel's conv_state rows, its T inputs and taps; for warp w < 2T the z
// of token w >> 1, V-head kh + 16 (w & 1), columns 4 lane .. 4 lane + 3; for
// tid < 2T the gate inputs of token tid >> 1 and V-head kh + 16 (tid & 1).
template <typename TA, int MT> struct MultiIn {
    TA s[KC - 1];
    TA x[MT];
    typename Raw4<TA>::type z;
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
    const int w = tid >> 5;
    p.z = typename Raw4<TA>::type{};
    if (w < 2 * T)
        p.z = *reinterpret_cast<const typename Raw4<TA>::type *>(
            static_cast<const TA *>(a.z) + (b * T + (w >> 1)) * (size_t)DI + (size_t)(kh + HK * (w & 1)) * DV + 4 * (tid & 31));
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

// Gamma below this is folded into S^: 1/Gamma stays far inside the fp32 range.
constexpr float MD_RENORM = 0x1p-60f;

__device__ __forceinline__ void scale4(float4 &v, float s)
{
    v.x *= s; v.y *= s; v.z *= s; v.w *= s;
}
__device__ __forceinline__ void axpy4(float4 &v, const float4 &x, float s)
{
    v.x = fmaf(x.x, s, v.x); v.y = fmaf(x.y, s, v.y); v.z = fmaf(x.z, s, v.z); v.w = fmaf(x.w, s, v.w);
}
__device__ __forceinline__ float dot4(const float4 &v, const float4 &x, float acc)
{
    return fmaf(v.w, x.w, fmaf(v.z, x.z, fmaf(v.y, x.y, fmaf(v.x, x.x, acc))));
}

// Sums four values p[0..3] over the 16 lanes of a half-warp (g = lane & 15)
// in five shuffles, halving the set at each step: lanes whose bit 3 is clear
// keep p[0], p[1] and send p[2], p[3] to their partner, and so on. Returns the
// total of p[g >> 2] (each total lands in four lanes).
// Packed pairs of fp32 (fma.rn.f32x2: two fused multiply-adds per instruction,
// each rounded as fmaf). A float4 is two pairs, (x, y) and (z, w).
__device__ __forceinline__ uint64_t pk2(float a, float b)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk2(uint64_t r, float &a, float &b)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// v0 . x0 + v1 . x1 over 8 elements, as two interleaved partial sums
__device__ __forceinline__ float dot8x2(const float4 &v0, const float4 &v1, const float4 &x0, const float4 &x1)
{
    uint64_t acc = fma2(pk2(v0.x, v0.y), pk2(x0.x, x0.y), 0ull);
    acc = fma2(pk2(v0.z, v0.w), pk2(x0.z, x0.w), acc);
    acc = fma2(pk2(v1.x, v1.y), pk2(x1.x, x1.y), acc);
    acc = fma2(pk2(v1.z, v1.w), pk2(x1.z, x1.w), acc);
    float lo, hi;
    upk2(acc, lo, hi);
    return lo + hi;
}
// v += x s over a float4, as two pairs
__device__ __forceinline__ void axpy4x2(float4 &v, const float4 &x, uint64_t ss)
{
    const uint64_t a = fma2(pk2(x.x, x.y), ss, pk2(v.x, v.y)), b = fma2(pk2(x.z, x.w), ss, pk2(v.z, v.w));
    upk2(a, v.x, v.y);
    upk2(b, v.z, v.w);
}
__device__ __forceinline__ float group16_reduce4(const float (&p)[4], int g)
{
    const bool hi3 = g & 8, hi2 = g & 4;
    const float a0 = (hi3 ? p[2] : p[0]) + __shfl_xor_sync(0xffffffffu, hi3 ? p[0] : p[2], 8);
    const float a1 = (hi3 ? p[3] : p[1]) + __shfl_xor_sync(0xffffffffu, hi3 ? p[1] : p[3], 8);
    float b = (hi2 ? a1 : a0) + __shfl_xor_sync(0xffffffffu, hi2 ? a0 : a1, 4);
    b += __shfl_xor_sync(0xffffffffu, b, 2);
    return b + __shfl_xor_sync(0xffffffffu, b, 1);
}

template <int MT>
__device__ __forceinline__ bool multi_unit_exists(const MultiArgs &a, int u)
{
    return blockIdx.x + (u / (2 * MD_UNITS)) * (int)gridDim.x < a.n_items;
}

// Lane 0 of a warp whose lanes have written their rows of unit u's new state
// back into slot u % MD_SLOTS and fenced them for the async proxy. The
// sixteenth warp to get here stores the slot to the unit's state with a bulk
// copy and returns unit u + MD_SLOTS, which it loads into the slot later
// (multi_refill), once the copy has surely read the slot; other warps, or
// when there is no such unit, get -1. The block fences order every warp's
// writes before the counter updates, and the last update before the copies.
template <int MT>
__device__ __forceinline__ int multi_release(MultiSmem<MT> &sm, const MultiArgs &a, int u)
{
    const int slot = u % MD_SLOTS;
    __threadfence_block();
    if (atomicAdd(&sm.released[slot], 1) != MD_WARPS - 1) return -1;
    __threadfence_block();
    sm.released[slot] = 0;
    sm.pending[slot] = -1;
    const uint32_t src = smem_u32(sm.slot[slot]);
    char *dst = multi_unit_ptr(a, u);
    bulk_s2g(dst, src, MD_SLOT_BYTES / 2);
    bulk_s2g(dst + MD_SLOT_BYTES / 2, src + MD_SLOT_BYTES / 2, MD_SLOT_BYTES / 2);
    bulk_commit();
    const int nu = u + MD_SLOTS;
    return sm.abort || !multi_unit_exists<MT>(a, nu) ? -1 : nu;
}

// The load multi_release returned, issued by the same thread one pass later:
// its own bulk stores have read the slot by then (the wait is a formality).
template <int MT>
__device__ __forceinline__ void multi_refill(MultiSmem<MT> &sm, const MultiArgs &a, int nu)
{
    bulk_wait_read();
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
        for (int w = 0; w < MD_WARPS; ++w) sm.owed[w][0] = sm.owed[w][1] = -1;
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_wait();                                   // inputs and states may come from the kernel ahead
    grid_dep_launch();

    if (tid == 0)                                      // the first MD_SLOTS units
        for (int u = 0; u < MD_SLOTS && multi_unit_exists<MT>(a, u); ++u) multi_issue_load(sm, a, u);

    const float scale = rsqrtf((float)DK);
    // norm weights of columns 4 lane .. 4 lane + 3 (none: the output is y itself,
    // and the norm runs in the output projection, gdn_gated_out_proj)
    const float4 nw = a.norm_w ? load4(a.norm_w + 4 * lane) : make_float4(1.f, 1.f, 1.f, 1.f);
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
            float xh[MT];                                // every slot computed, so tokens interleave
#pragma unroll
            for (int t = 0; t < MT; ++t)
                xh[t] = silu_f(pin.w.x * win[t] + pin.w.y * win[t + 1] + pin.w.z * win[t + 2] + pin.w.w * win[t + 3]);
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
            float *dst = tid < 128 ? &sm.q[0][tid] : tid < 256 ? &sm.k[0][tid - 128] : &sm.v[0][(tid - 256) >> 7][tid & 127];
            const int tstride = tid < 256 ? DK : 2 * DV;
#pragma unroll
            for (int t = 0; t < MT; ++t)
                if (t < T) dst[t * tstride] = xh[t];
            if (tid < 2 * T) {
                float ga, gb;
                gates_f(pin.A_log, pin.dt_bias, to_f(pin.al), to_f(pin.be), ga, gb);
                sm.gate[tid >> 1][tid & 1][0] = ga;
                sm.gate[tid >> 1][tid & 1][1] = gb;
                sm.gate[tid >> 1][tid & 1][2] = 1.0f / ga;   // inf for a decay of 0: then Gamma is renormalised
            }
            multi_sync();
            if (warp < 2 * T) {                          // L2 norm of q_t (w even) or k_t (w odd), t = w >> 1
                float4 *vec = reinterpret_cast<float4 *>((warp & 1) ? sm.k[warp >> 1] : sm.q[warp >> 1]) + lane;
                float4 v4 = *vec;
                const float r = rsqrtf(warp_sum(dot4(v4, v4, 0.0f)) + a.l2_eps);
                scale4(v4, r);
                *vec = v4;
            }
            multi_sync();
        }
        const typename Raw4<TA>::type zcur = pin.z;
        if (item + (int)gridDim.x < a.n_items) pin = multi_load<TA, MT>(a, item + gridDim.x, tid);

        // ---- the two states: each row takes tokens 0..T-1 in order.
        // Head h is one pass over its two slots. A group of 16 lanes holds four
        // of its rows, jl and jl + 32 of each slot, 8 keys a lane, so every k
        // and q load of a token serves four rows. The state is kept as
        // Gamma * S^ with Gamma the running product of the head's decays: the
        // decay costs one multiply per token instead of one per element, and
        // S^ is rescaled only when Gamma falls below MD_RENORM (and at the
        // end). In this form, with Gamma_t = Gamma_{t-1} exp(g_t),
        //   pred = Gamma_t (S^ k),  S^ += k (beta (v - pred) / Gamma_t),
        //   y = Gamma_t (S^ q) / sqrt(d_k).
        static_assert(MD_UNITS == 2 && MD_SLOT_ROWS == 2 * 32 && MD_WARPS * 2 == 32, "row mapping");
        const int g = lane & 15;                         // float4 columns g and g + 16 of each row
        const int jl = warp * 2 + (lane >> 4);           // rows jl, jl + 32 of each slot
        const int qown = g >> 2;                         // the row this lane reduces (see row_of)
        auto row_of = [&](int q) { return (q >> 1) * MD_SLOT_ROWS + jl + 32 * (q & 1); };   // row j of the head
        const int jown = row_of(qown);
        for (int h = 0; h < 2; ++h) {
            const int u0 = 2 * MD_UNITS * m + MD_UNITS * h;   // units u0 (rows 0..63), u0 + 1 (rows 64..127)
            if (lane == 0) {                             // units of later passes, owed since the last one
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (sm.owed[warp][i] >= 0 && !aborted) multi_refill(sm, a, sm.owed[warp][i]);
                    sm.owed[warp][i] = -1;
                }
            }
            if (aborted) continue;                       // skip the work, keep the barriers in step
            if (!mbar_wait_bounded(smem_u32(&sm.full[u0 % MD_SLOTS]), (uint32_t)((u0 / MD_SLOTS) & 1)) ||
                !mbar_wait_bounded(smem_u32(&sm.full[(u0 + 1) % MD_SLOTS]), (uint32_t)(((u0 + 1) / MD_SLOTS) & 1))) {
                sm.abort = 1;
                continue;
            }
            float4 st[4][2];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 *src = reinterpret_cast<const float4 *>(sm.slot[(u0 + (q >> 1)) % MD_SLOTS]) +
                                    (jl + 32 * (q & 1)) * (DK / 4) + g;
                st[q][0] = src[0];
                st[q][1] = src[16];
            }
            float gam = 1.0f, igam = 1.0f;               // Gamma and 1 / Gamma
            // y of each token is stored during the next one, so that the next
            // token's work need not wait for the reduction behind it
            float y_prev = 0.0f, yscale_prev = 0.0f;
            for (int t = 0; t < T; ++t) {
                float G = gam * sm.gate[t][h][0], iG = igam * sm.gate[t][h][2];
                if (G < MD_RENORM) {                     // fold Gamma into S^ (warp-uniform)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        scale4(st[q][0], G);
                        scale4(st[q][1], G);
                    }
                    G = iG = 1.0f;
                }
                gam = G;
                igam = iG;
                const float4 *k4 = reinterpret_cast<const float4 *>(sm.k[t]) + g;
                const float4 *q4 = reinterpret_cast<const float4 *>(sm.q[t]) + g;
                const float4 k0 = k4[0], k1 = k4[16];
                float p[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) p[q] = dot8x2(st[q][0], st[q][1], k0, k1);
                const float pred = G * group16_reduce4(p, g);
                const float dn = (sm.v[t][h][jown] - pred) * sm.gate[t][h][1] * iG;
                float d[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) d[q] = __shfl_sync(0xffffffffu, dn, (lane & 16) | (q << 2));
                const float4 q0 = q4[0], q1 = q4[16];
                float y[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint64_t dd = pk2(d[q], d[q]);
                    axpy4x2(st[q][0], k0, dd);
                    axpy4x2(st[q][1], k1, dd);
                    y[q] = dot8x2(st[q][0], st[q][1], q0, q1);
                }
                if (t > 0 && (g & 3) == 0) sm.y[t - 1][h][jown] = y_prev * yscale_prev;
                y_prev = group16_reduce4(y, g);
                yscale_prev = G * scale;
            }
            if ((g & 3) == 0) sm.y[T - 1][h][jown] = y_prev * yscale_prev;
            // the new rows go back where they came from; the slots' bulk stores
            // then drain them to HBM while the warps go on
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float4 *dst = reinterpret_cast<float4 *>(sm.slot[(u0 + (q >> 1)) % MD_SLOTS]) +
                              (jl + 32 * (q & 1)) * (DK / 4) + g;
                scale4(st[q][0], gam);
                scale4(st[q][1], gam);
                dst[0] = st[q][0];
                dst[16] = st[q][1];
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                sm.owed[warp][0] = multi_release(sm, a, u0);
                sm.owed[warp][1] = multi_release(sm, a, u0 + 1);
            }
        }
        multi_sync();                                    // all rows of y are in, and the abort flag agrees
        if (aborted) break;

        // ---- gated RMSNorm times silu(z) ("Output path"): warp w < 2T takes
        //      token w >> 1 of V-head kh + 16 (w & 1), columns 4 lane .. 4 lane + 3
        if (warp < 2 * T) {
            const int t = warp >> 1, h = warp & 1;
            const float4 y4 = reinterpret_cast<const float4 *>(sm.y[t][h])[lane];
            const float rr2 = rsqrtf(warp_sum(dot4(y4, y4, 0.0f)) * (1.0f / DV) + a.norm_eps);
            const float4 zf = raw4_f(zcur);
            const float4 o = a.norm_w ? make_float4(y4.x * rr2 * nw.x * silu_f(zf.x), y4.y * rr2 * nw.y * silu_f(zf.y),
                                                    y4.z * rr2 * nw.z * silu_f(zf.z), y4.w * rr2 * nw.w * silu_f(zf.w))
                                      : y4;
            store4(static_cast<TO *>(a.out) + (b * T + t) * (size_t)DI + (size_t)(kh + HK * h) * DV + 4 * lane, o);
        }
        // the next prologue writes q/k/v/gate and the next sweep y only after a barrier
    }
    if (aborted && tid == 0) atomicExch(&g_multi_error, (unsigned int)GDN_ERR_TIMEOUT);
    if (lane == 0) bulk_wait_all();                      // the state stores this lane issued are done
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
// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *multi_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_multi_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
