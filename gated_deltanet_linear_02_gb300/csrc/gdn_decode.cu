// gdn_decode.cu -- single-token kernels: the conv step and the fused decode step.
//
// Decode is a batched, HBM-bound sweep over the fp32 states. Each 128x128
// state of one (sequence, V-head) is 64 KiB and makes up 97% of the bytes.
// The kernel reads every state once and writes it once, and runs every other
// step of the SSM block on chip in between. The SSM block is the one in
// "qwen35moe -- Forward-Pass Design (Pantheon port)", sections "Causal conv1d",
// "Decay gate", "Per-token recurrence" and "Output path".
//
// The decode kernel is persistent: one CTA of 16 warps per SM. Each CTA walks
// the work items (sequence b, K-head kh) in turn. An item covers both V-heads
// that read K-head kh, vh = kh and vh = kh + 16 (the interleaved GQA repeat of
// the watch-list). So the item's q/k conv channels, and their conv_state, are
// touched by this CTA alone. No other CTA reads them, and the state shift
// needs no cross-CTA ordering.
//
// The states stream through a ring of six 32 KiB shared-memory slots, each
// holding 64 rows of one state. A producer warp fills them with TMA bulk copies
// (cp.async.bulk), which complete on a "full" mbarrier per slot; it refills a
// slot as soon as all 16 compute warps have arrived on the slot's "empty"
// mbarrier, so the ring stays as full as the slots allow and no CTA-wide
// barrier sits between slots. Warp w computes 4 rows j of each slot (rows of
// S^T: value index j, 128 contiguous keys i), all four at once: lanes 8r..8r+7
// hold row r, lane 8r+g the keys of float4 groups g, g+8, g+16, g+24. pred_j,
// delta_j and y_j depend on row j alone, so each dot product is a sum within
// the row's 8 lanes (3 shuffle steps, the four rows in parallel). The updated
// row goes straight back to global memory with streaming stores. The compute warps synchronise among
// themselves (a named barrier) only in an item's prologue and its output norm.
// An item's prologue inputs (conv_state, qkv, gates, z) are loaded one item
// ahead, so their latency hides behind the previous item's sweep.
#include "gdn_async.cuh"
#include "gdn_common.cuh"

namespace gdn {

__device__ unsigned int g_decode_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

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
    int n_items;   // B * 16
};

constexpr int DEC_WARPS = 16;                              // compute warps
constexpr int DEC_COMPUTE = 32 * DEC_WARPS;
constexpr int DEC_THREADS = DEC_COMPUTE + 32;              // + the producer warp
constexpr int DEC_SLOT_ROWS = 64;                          // rows j of S^T per staging slot
constexpr int DEC_UNITS = DV / DEC_SLOT_ROWS;              // slots per state (2)
constexpr int DEC_ROWS_PER_WARP = DEC_SLOT_ROWS / DEC_WARPS;   // 4
static_assert(DEC_ROWS_PER_WARP == 4, "a warp computes 4 rows of a slot at once, 8 lanes per row");
constexpr int DEC_SLOTS = 6;
constexpr uint32_t SLOT_BYTES = DEC_SLOT_ROWS * DK * sizeof(float);   // 32 KiB
constexpr int DEC_COPIES = 2;                              // bulk copies per slot

struct DecodeSmem {
    alignas(128) float slot[DEC_SLOTS][DEC_SLOT_ROWS * DK];   // TMA destinations
    alignas(16) float q[DK];                        // read as float4
    alignas(16) float k[DK];
    alignas(16) float v[2][DV];
    alignas(16) float y[2][DV];
    alignas(8) uint64_t full[DEC_SLOTS];
    uint64_t empty[DEC_SLOTS];
    float red[32];
    float gate[2][2];
    int pending[DEC_SLOTS];   // unit number whose load is outstanding in each slot, or -1
    int abort;
};
constexpr size_t DEC_SMEM = sizeof(DecodeSmem) + 128;   // + alignment slack

// Issues the TMA load of this CTA's unit number `u` into slot u % DEC_SLOTS.
// Units walk item by item, V-head by V-head, then slot-sized row blocks:
// u = (2 * m + h) * DEC_UNITS + part. Caller: the producer thread; the unit's
// item exists.
__device__ __forceinline__ void decode_issue_load(DecodeSmem &sm, const DecodeArgs &a, int u)
{
    const int item = blockIdx.x + (u / (2 * DEC_UNITS)) * gridDim.x;
    const int h = (u / DEC_UNITS) & 1, part = u % DEC_UNITS;
    const int b = item / HK, kh = item % HK, vh = kh + HK * h;
    const char *src = reinterpret_cast<const char *>(a.ssm_state + ((size_t)b * HV + vh) * (DV * DK)) +
                      (size_t)part * SLOT_BYTES;
    const int slot = u % DEC_SLOTS;
    sm.pending[slot] = u;
    const uint32_t bar = smem_u32(&sm.full[slot]);
    const uint32_t dst = smem_u32(sm.slot[slot]);
    mbar_arrive_expect_tx(bar, SLOT_BYTES);
#pragma unroll
    for (int c = 0; c < DEC_COPIES; ++c)
        bulk_g2s(dst + c * (SLOT_BYTES / DEC_COPIES), src + c * (SLOT_BYTES / DEC_COPIES), SLOT_BYTES / DEC_COPIES,
                 bar);
}

// Global inputs of one item's prologue held by thread `tid`: its conv channel
// (raw conv_state rows, current input, taps) and, for threads 0 and 1, the
// gate inputs of V-heads kh and kh + 16.
template <typename TA> struct PrologueIn {
    TA s0, s1, s2, xc, al, be, zc;
    float4 w;
    float A_log, dt_bias;
};

// conv channel of thread tid within item (., kh): q | k of K-head kh, v of vh = kh, v of vh = kh + 16
__device__ __forceinline__ int item_channel(int kh, int tid)
{
    if (tid < 128) return Q_OFF + kh * DK + tid;
    if (tid < 256) return K_OFF + kh * DK + (tid - 128);
    if (tid < 384) return V_OFF + kh * DV + (tid - 256);
    return V_OFF + (kh + HK) * DV + (tid - 384);
}

template <typename TA>
__device__ __forceinline__ PrologueIn<TA> prologue_load(const DecodeArgs &a, int item, int tid)
{
    PrologueIn<TA> p;
    const size_t b = item / HK;
    const int kh = item % HK;
    const int c = item_channel(kh, tid);
    const TA *x = static_cast<const TA *>(a.qkv) + b * CC;
    const TA *cs = static_cast<const TA *>(a.conv_state) + b * (size_t)(KC - 1) * CC;
    p.w = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + c);
    p.s0 = cs[c]; p.s1 = cs[CC + c]; p.s2 = cs[2 * CC + c]; p.xc = x[c];
    // threads 0..255 also hold z of output column j = tid & 127 of V-head kh + 16 * (tid >> 7)
    p.zc = tid < 2 * DV ? static_cast<const TA *>(a.z)[b * DI + (size_t)(kh + HK * (tid >> 7)) * DV + (tid & 127)]
                        : from_f<TA>(0.0f);
    p.al = p.be = from_f<TA>(0.0f);
    p.A_log = p.dt_bias = 0.0f;
    if (tid < 2) {
        const int vh = kh + HK * tid;
        p.al = static_cast<const TA *>(a.alpha)[b * HV + vh];
        p.be = static_cast<const TA *>(a.beta)[b * HV + vh];
        p.A_log = a.A_log[vh];
        p.dt_bias = a.dt_bias[vh];
    }
    return p;
}

// Barrier among the 16 compute warps only (the producer warp never joins it).
__device__ __forceinline__ void compute_sync() { asm volatile("bar.sync 1, %0;" ::"n"(DEC_COMPUTE) : "memory"); }

template <typename TA, typename TO>
__global__ void __launch_bounds__(DEC_THREADS, 1) decode_step_kernel(const DecodeArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    // The block is aligned through a generic pointer here, unlike the other
    // kernels (smem_aligned128). Measured at B=256: 169 us per launch this way,
    // 179 us with the shared-window form, whose different instruction
    // schedule costs this kernel more than the 64-bit addresses do.
    DecodeSmem &sm = *reinterpret_cast<DecodeSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~(uintptr_t)127);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const volatile int &aborted = sm.abort;

    if (tid == 0) {
        for (int i = 0; i < DEC_SLOTS; ++i) {
            mbar_init(smem_u32(&sm.full[i]), 1);
            mbar_init(smem_u32(&sm.empty[i]), DEC_WARPS);
            sm.pending[i] = -1;
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dep_wait();                                   // inputs and states may come from the kernel ahead
    grid_dep_launch();

    if (warp == DEC_WARPS) {
        // ---- producer: unit u goes into slot u % DEC_SLOTS once the compute
        //      warps have released that slot's previous unit, u - DEC_SLOTS
        if (lane == 0) {
            for (int u = 0;; ++u) {
                if (blockIdx.x + (u / (2 * DEC_UNITS)) * (int)gridDim.x >= a.n_items) break;
                const int slot = u % DEC_SLOTS;
                if (u >= DEC_SLOTS) {
                    if (!mbar_wait_bounded(smem_u32(&sm.empty[slot]), (uint32_t)((u / DEC_SLOTS - 1) & 1))) sm.abort = 1;
                    sm.pending[slot] = -1;     // its previous load completed before the compute warps released it
                }
                if (aborted) break;
                fence_proxy_async_smem();
                decode_issue_load(sm, a, u);
            }
            // after an abort, let the copies still in flight land before the
            // CTA's shared memory is released
            if (aborted)
                for (int i = 0; i < DEC_SLOTS; ++i)
                    if (sm.pending[i] >= 0)
                        mbar_wait_bounded(smem_u32(&sm.full[i]), (uint32_t)((sm.pending[i] / DEC_SLOTS) & 1));
        }
        return;
    }

    // ---- compute warps
    const float scale = rsqrtf((float)DK);
    PrologueIn<TA> pin;
    if ((int)blockIdx.x < a.n_items) pin = prologue_load<TA>(a, blockIdx.x, tid);
    for (int m = 0;; ++m) {
        const int item = blockIdx.x + m * gridDim.x;
        if (item >= a.n_items) break;
        const size_t b = item / HK;
        const int kh = item % HK;

        // ---- item prologue: conv + SiLU of the item's 512 channels (q and k of
        //      K-head kh, v of both V-heads), state shift, L2 norms, gates. Its
        //      global inputs were loaded one item ahead (pin).
        {
            TA *cs = static_cast<TA *>(a.conv_state) + b * (size_t)(KC - 1) * CC;
            const int c = item_channel(kh, tid);
            const float xh = silu_f(pin.w.x * to_f(pin.s0) + pin.w.y * to_f(pin.s1) + pin.w.z * to_f(pin.s2) +
                                    pin.w.w * to_f(pin.xc));
            cs[c] = pin.s1;                   // this CTA owns channel c of sequence b
            cs[CC + c] = pin.s2;
            cs[2 * CC + c] = pin.xc;
            const float ss = warp_sum(xh * xh);
            if (lane == 0) sm.red[warp] = ss;
            if (tid < 2) {
                float ga, gb;
                gates_f(pin.A_log, pin.dt_bias, to_f(pin.al), to_f(pin.be), ga, gb);
                sm.gate[tid][0] = ga;
                sm.gate[tid][1] = gb;
            }
            compute_sync();
            if (tid < 128) sm.q[tid] = xh * rsqrtf(sm.red[0] + sm.red[1] + sm.red[2] + sm.red[3] + a.l2_eps);
            else if (tid < 256) sm.k[tid - 128] = xh * rsqrtf(sm.red[4] + sm.red[5] + sm.red[6] + sm.red[7] + a.l2_eps);
            else sm.v[(tid - 256) >> 7][tid & 127] = xh;
            compute_sync();
        }
        const TA zcur = pin.zc;
        // the next item's prologue inputs: their latency hides behind this item's sweep
        if (item + (int)gridDim.x < a.n_items) pin = prologue_load<TA>(a, item + gridDim.x, tid);

        // ---- the two states of the item: recurrence (a)-(d) row by row. Each
        //      warp takes its rows of a slot as soon as the slot has landed and
        //      releases the slot when it is done with them.
        const int rr = lane >> 3, g = lane & 7;         // row of the warp's four; float4 group within it
        float4 k4[4], q4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            k4[c] = reinterpret_cast<const float4 *>(sm.k)[8 * c + g];
            q4[c] = reinterpret_cast<const float4 *>(sm.q)[8 * c + g];
        }
        for (int hp = 0; hp < 2 * DEC_UNITS; ++hp) {
            const int h = hp / DEC_UNITS, part = hp % DEC_UNITS;
            const int u = 2 * DEC_UNITS * m + hp;
            const int slot = u % DEC_SLOTS;
            if (aborted) continue;                       // skip the work, keep the barriers in step
            if (!mbar_wait_bounded(smem_u32(&sm.full[slot]), (uint32_t)((u / DEC_SLOTS) & 1))) {
                sm.abort = 1;
                continue;
            }
            const int vh = kh + HK * h;
            float *Sg = a.ssm_state + (b * HV + vh) * (size_t)(DV * DK);
            const float dec = sm.gate[h][0], beta = sm.gate[h][1];
            const int jl = warp * DEC_ROWS_PER_WARP + rr;     // row within the slot
            const int j = part * DEC_SLOT_ROWS + jl;
            const float4 *src = reinterpret_cast<const float4 *>(sm.slot[slot]) + jl * (DK / 4) + g;
            const float vj = sm.v[h][j];
            float4 st[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) st[c] = src[8 * c];
            float pa = 0.0f, pb = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                st[c].x *= dec; st[c].y *= dec; st[c].z *= dec; st[c].w *= dec;                      // (a)
                pa = fmaf(st[c].x, k4[c].x, fmaf(st[c].y, k4[c].y, pa));
                pb = fmaf(st[c].z, k4[c].z, fmaf(st[c].w, k4[c].w, pb));
            }
            const float pred = group_sum<8>(pa + pb);                                                  // (b)
            const float delta = (vj - pred) * beta;
            float ya = 0.0f, yb = 0.0f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                st[c].x = fmaf(k4[c].x, delta, st[c].x); st[c].y = fmaf(k4[c].y, delta, st[c].y);      // (c)
                st[c].z = fmaf(k4[c].z, delta, st[c].z); st[c].w = fmaf(k4[c].w, delta, st[c].w);
                ya = fmaf(st[c].x, q4[c].x, fmaf(st[c].y, q4[c].y, ya));
                yb = fmaf(st[c].z, q4[c].z, fmaf(st[c].w, q4[c].w, yb));
            }
            const float yq = group_sum<8>(ya + yb);                                                    // (d)
            float4 *dst = reinterpret_cast<float4 *>(Sg + (size_t)j * DK) + g;
#pragma unroll
            for (int c = 0; c < 4; ++c) __stcs(dst + 8 * c, st[c]);
            if (g == 0) sm.y[h][j] = yq * scale;
            __syncwarp();                                // this warp's reads of the slot are done
            if (lane == 0) mbar_arrive(smem_u32(&sm.empty[slot]));
        }
        compute_sync();                                  // all rows of y are in, and the abort flag agrees
        if (aborted) break;

        // ---- gated RMSNorm of both heads, times silu(z) ("Output path")
        if (tid < 256) {
            const int h = tid >> 7, j = tid & 127;
            const float y = sm.y[h][j];
            const float ss = warp_sum(y * y);
            if (lane == 0) sm.red[16 + warp] = ss;
        }
        compute_sync();
        if (tid < 256) {
            const int h = tid >> 7, j = tid & 127;
            const float *rr4 = sm.red + 16 + 4 * h;
            const float rr = rsqrtf((rr4[0] + rr4[1] + rr4[2] + rr4[3]) * (1.0f / DV) + a.norm_eps);
            const size_t o = b * DI + (size_t)(kh + HK * h) * DV + j;
            // without norm weights the output is y itself (the norm runs in the
            // output projection, gdn_gated_out_proj)
            static_cast<TO *>(a.out)[o] =
                from_f<TO>(a.norm_w ? sm.y[h][j] * rr * a.norm_w[j] * silu_f(to_f(zcur)) : sm.y[h][j]);
        }
        // the next prologue writes q/k/v/red[0..7]/gate, none of which the lines above read
    }
    if (aborted && tid == 0) atomicExch(&g_decode_error, (unsigned int)GDN_ERR_TIMEOUT);
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

int sm_count()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

template <typename TA, typename TO>
static cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t s)
{
    cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<TA, TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)DEC_SMEM);
    if (e != cudaSuccess) return e;
    const int n_sm = sm_count();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    const int grid = a.n_items < n_sm ? a.n_items : n_sm;
    // programmatic stream serialization: this launch may start while the kernel
    // ahead drains; the kernel waits for it before its first global access
    return launch_pdl(decode_step_kernel<TA, TO>, dim3(grid), dim3(DEC_THREADS), DEC_SMEM, s, a);
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
    a.n_items = B * HK;
    if (act == GDN_F32)
        return out_dt == GDN_F32 ? launch_decode_t<float, float>(a, s) : launch_decode_t<float, bf16>(a, s);
    return out_dt == GDN_F32 ? launch_decode_t<bf16, float>(a, s) : launch_decode_t<bf16, bf16>(a, s);
}

// Reads and clears this file's device error word (synchronous on `s`).
// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *decode_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_decode_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
