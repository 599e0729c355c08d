// gdn_in_conv.cu -- the input projections with the causal conv1d, SiLU and the
// q/k L2 norms applied in the GEMM's epilogue. Sections "Projections" and
// "Causal conv1d" of "qwen35moe -- Forward-Pass Design (Pantheon port)", "SSM
// block -- Gated-Delta-Net": the projections attn_qkv, attn_gate, ssm_alpha and
// ssm_beta of the normed hidden state, then the conv over the 8192-channel
// q|k|v stream with the last three raw inputs of each sequence (conv_state)
// before its first token, SiLU, and the L2 norm of each q and k head.
//
// The raw q|k|v stream never goes to memory: each output tile's fp32
// accumulator is staged in shared memory, and the conv reads the three rows
// above a row from there. The Lily page's "Reduce intermediate and state
// traffic" gives the reason: the fused step saves the stream's write and its
// read back (32 KiB per token).
//
// Design. Output tiles of 256 columns (two heads of q, k or v, or 256 columns
// of z, or alpha|beta) by 128 GEMM rows. Consecutive row tiles overlap by three
// rows: tile i covers rows [125 i - 3, 125 i + 125) and produces rows [125 i,
// 125 i + 125), so every produced row finds its three predecessors in the same
// tile (the rows before row 0 are read as zeros by TMA and never used: a row
// before its sequence's start takes conv_state instead). Per CTA (persistent):
//  - warp 0, lane 0: TMA producer: 64-column K slices of h (128 rows) and of
//    the weight (256 rows) into three 48 KiB stages, 128-byte swizzle;
//  - warp 1, lane 0: MMA issuer: tcgen05.mma kind::f16 (bf16), M=128, N=256,
//    K=16, into two 256-column TMEM accumulators;
//  - warps 2-17: the epilogue. Warp w takes TMEM lane quarter w % 4 (tile rows
//    32 (w % 4) ..) and one quarter of the columns (32). The tile goes to shared
//    memory [128][129] fp32 (rows on distinct banks), one 128-column half at a
//    time. Then per row and column quarter of the half: q|k|v: the conv over rows r-3..r (or conv_state rows before the
//    sequence's start) and SiLU, kept in registers. For q and k the four
//    quarters' sums of squares meet in shared memory for the head's L2 norm.
//    The result is written as fp16 x^, and the raw values of each sequence's
//    last three tokens go to conv_state_out. z, alpha, beta: written as bf16.
// All mbarrier waits are bounded; a wait that gives up records GDN_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_fp16.h>

#include <mutex>

#include "gdn_async.cuh"
#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

namespace gdn {

__device__ unsigned int g_inconv_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

constexpr int IC_BM = 128, IC_ROWS = IC_BM - (KC - 1), IC_BN = 256, IC_BK = 64;
constexpr int IC_HALF = 128;                              // the epilogue takes a tile in two 128-column halves
constexpr int IC_STAGES = 3;
constexpr uint32_t IC_A_BYTES = IC_BM * IC_BK * 2, IC_B_BYTES = IC_BN * IC_BK * 2;
constexpr uint32_t IC_STAGE = IC_A_BYTES + IC_B_BYTES;   // 48 KiB
constexpr int IC_EPI_WARPS = 16;                         // 4 per TMEM lane quarter, 32 columns each
constexpr int IC_THREADS = 64 + 32 * IC_EPI_WARPS;
constexpr int IC_LD = IC_HALF + 1;                        // staged half-tile row stride (floats)
constexpr int IC_N = CC + DI + 2 * HV;                    // 12352 projected columns
constexpr int IC_NT = (IC_N + IC_BN - 1) / IC_BN;         // 49 column tiles
constexpr int IC_K = GDN_HIDDEN;                          // 2048

struct IcSmem {
    alignas(1024) unsigned char stage[IC_STAGES][IC_STAGE];
    float ep[IC_BM][IC_LD];                               // the staged half of the accumulator tile
    float4 cw[IC_HALF];                                   // conv taps of the half's columns
    float red[IC_BM][4];                                  // per-row partial sums of squares (q, k heads)
    alignas(8) uint64_t full[IC_STAGES], empty[IC_STAGES], acc_full[2], acc_empty[2];
    int last_it[IC_STAGES];
    uint32_t tmem;
    int abort;
};
constexpr size_t IC_SMEM = sizeof(IcSmem) + 1024;
static_assert(IC_SMEM <= 232448, "in-projection conv shared memory");

struct IcArgs {
    const float *conv_w;          // [8192][4]
    float l2_eps;
    const int32_t *cu;            // [N + 1]
    int N, M;
    const bf16 *cs_in;            // [N][3][8192] or NULL (zeros)
    bf16 *cs_out;                 // [N][3][8192] or NULL
    __half *xhat;                 // [M][8192]
    bf16 *z, *alpha, *beta;       // [M][4096], [M][32], [M][32]
};

__device__ __forceinline__ float silu_approx(float u)
{
    // u sigmoid(u) = (u / 2)(1 + tanh(u / 2)), one special-function operation
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * u));
    const float hu = 0.5f * u;
    return fmaf(hu, th, hu);
}

// Sequence n holding packed row m: the last n with cu[n] <= m (cu clamped into
// [0, M] and made non-decreasing as read).
__device__ __forceinline__ int seq_of(const int32_t *cu, int N, int M, int m)
{
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (min(max(__ldg(cu + mid), 0), M) <= m) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// The epilogue warps meet at named barrier 1; ic_epi_or also returns the OR
// of a flag over them, so that they leave a loop together or not at all.
__device__ __forceinline__ void ic_epi_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
__device__ __forceinline__ bool ic_epi_or(bool p)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
                 "bar.red.or.pred b, 1, 512, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
                 : "=r"(r) : "r"((uint32_t)p) : "memory");
    return r != 0;
}
static_assert(IC_EPI_WARPS == 16, "the named barriers count 512 epilogue threads");

__global__ void __launch_bounds__(IC_THREADS, 1) in_conv_kernel(const __grid_constant__ CUtensorMap mh,
                                                                const __grid_constant__ CUtensorMap mw,
                                                                const IcArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *blk = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    IcSmem &sm = *reinterpret_cast<IcSmem *>(blk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = a.M;
    const int n_work = ((M + IC_ROWS - 1) / IC_ROWS) * IC_NT;
    const volatile int &aborted = sm.abort;
    constexpr int KB = IC_K / IC_BK;                   // 32 K slices

    if (warp == 1) {
        tc::tmem_alloc(smem_u32(&sm.tmem), 2 * IC_BN);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < IC_STAGES; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1);
            sm.last_it[s] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sm.acc_full[b]), 1);
            mbar_init(smem_u32(&sm.acc_empty[b]), 32 * IC_EPI_WARPS);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem;
    grid_dep_wait();                                   // h may come from the kernel ahead
    grid_dep_launch();

    if (warp == 0) {
        if (lane == 0) {
            int it = 0;
            for (int w = blockIdx.x; w < n_work && !aborted; w += gridDim.x) {
                const int m0 = (w / IC_NT) * IC_ROWS - (KC - 1), nt = w % IC_NT;
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % IC_STAGES;
                    if (it >= IC_STAGES &&
                        !mbar_wait_bounded(smem_u32(&sm.empty[s]), (uint32_t)((it / IC_STAGES - 1) & 1)))
                        sm.abort = 1;
                    if (aborted) break;
                    const uint32_t dst = smem_u32(sm.stage[s]);
                    mbar_arrive_expect_tx(smem_u32(&sm.full[s]), IC_STAGE);
                    tma_load_2d(dst, &mh, kb * IC_BK, m0, smem_u32(&sm.full[s]));   // rows < 0 read as zero
                    tma_load_2d(dst + IC_A_BYTES, &mw, kb * IC_BK, nt * IC_BN, smem_u32(&sm.full[s]));
                    sm.last_it[s] = it;
                }
            }
            if (aborted)
                for (int s = 0; s < IC_STAGES; ++s)
                    if (sm.last_it[s] >= 0)
                        mbar_wait_bounded(smem_u32(&sm.full[s]), (uint32_t)((sm.last_it[s] / IC_STAGES) & 1));
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::instr_desc(tc::FMT_BF16, IC_BM, IC_BN);
            int it = 0, ti = 0;
            for (int w = blockIdx.x; w < n_work && !aborted; w += gridDim.x, ++ti) {
                const int ab = ti & 1;
                if (ti >= 2 && !mbar_wait_bounded(smem_u32(&sm.acc_empty[ab]), (uint32_t)(((ti >> 1) - 1) & 1)))
                    sm.abort = 1;
                tc::fence_after_sync();
                const uint32_t d = tm + (uint32_t)(IC_BN * ab);
                for (int kb = 0; kb < KB; ++kb, ++it) {
                    const int s = it % IC_STAGES;
                    if (!mbar_wait_bounded(smem_u32(&sm.full[s]), (uint32_t)((it / IC_STAGES) & 1))) sm.abort = 1;
                    if (aborted) break;
                    tc::fence_after_sync();
                    const uint32_t a0 = smem_u32(sm.stage[s]);
                    const uint64_t ad = tc::sw128_desc(a0), bd = tc::sw128_desc(a0 + IC_A_BYTES);
#pragma unroll
                    for (int k = 0; k < IC_BK / 16; ++k)
                        tc::mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    tc::mma_commit(smem_u32(&sm.empty[s]));
                }
                if (aborted) break;
                tc::mma_commit(smem_u32(&sm.acc_full[ab]));
            }
        }
    } else {
        // ---- epilogue: warp w (2..17) owns tile rows 32 (w % 4) + lane and
        //      columns [32 cq, 32 cq + 32), cq = (w - 2) / 4
        const int q = warp & 3, r = 32 * q + lane, cq = (warp - 2) >> 2, cb = 32 * cq, t = tid - 64;
        int ti = 0;
        for (int w = blockIdx.x; w < n_work; w += gridDim.x, ++ti) {
            const int ab = ti & 1;
            const int m = (w / IC_NT) * IC_ROWS - (KC - 1) + r, nt = w % IC_NT, c0t = nt * IC_BN;
            const bool got = mbar_wait_bounded(smem_u32(&sm.acc_full[ab]), (uint32_t)((ti >> 1) & 1));
            if (!got) sm.abort = 1;
            if (ic_epi_or(!got || aborted)) break;     // all epilogue warps leave together
            tc::fence_after_sync();
            for (int hh = 0; hh < IC_BN / IC_HALF; ++hh) {
            const int c0 = c0t + IC_HALF * hh;         // first column of this half
            {
                float v[32];
                tc::tmem_ld32(tc::tmem_addr(tm + (uint32_t)(IC_BN * ab), 32 * q, IC_HALF * hh + cb), v);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) sm.ep[r][cb + e] = v[e];
            }
            if (hh == IC_BN / IC_HALF - 1) {
                tc::fence_before_sync();
                mbar_arrive(smem_u32(&sm.acc_empty[ab]));   // the accumulator may be refilled
            }
            if (c0 < CC && t < IC_HALF) sm.cw[t] = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + c0 + t);
            ic_epi_sync();                             // the half and its taps are staged
            const bool live = r >= KC - 1 && m < M;
            if (c0 < CC) {
                // ---- conv + SiLU (+ L2 norm for q and k) of row m, columns c0 + cb ..
                float o[32];
                int n = 0, s0 = 0, s1 = 0;
                if (live) {
                    n = seq_of(a.cu, a.N, M, m);
                    s0 = min(max(__ldg(a.cu + n), 0), M);
                    s1 = min(max(__ldg(a.cu + n + 1), s0), M);
                    const bf16 *csr[KC - 1];           // conv_state rows for taps before the sequence start
#pragma unroll
                    for (int k = 0; k < KC - 1; ++k) {
                        const int pos = m - (KC - 1) + k;
                        csr[k] = (pos >= s0 || !a.cs_in)
                                     ? nullptr
                                     : a.cs_in + ((size_t)n * (KC - 1) + (pos - s0 + KC - 1)) * CC + c0 + cb;
                    }
                    const bool inside[KC - 1] = {m - 3 >= s0, m - 2 >= s0, m - 1 >= s0};
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        float x[KC];
#pragma unroll
                        for (int k = 0; k < KC - 1; ++k)
                            x[k] = inside[k] ? sm.ep[r - (KC - 1) + k][cb + e] : (csr[k] ? to_f(csr[k][e]) : 0.0f);
                        x[KC - 1] = sm.ep[r][cb + e];
                        const float4 wv = sm.cw[cb + e];
                        o[e] = silu_approx(wv.x * x[0] + wv.y * x[1] + wv.z * x[2] + wv.w * x[3]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0.0f;
                }
                float scale = 1.0f;
                if (c0 < V_OFF) {                      // q or k head: L2 norm over its 128 columns
                    float ss = 0.0f;
#pragma unroll
                    for (int e = 0; e < 32; ++e) ss = fmaf(o[e], o[e], ss);
                    sm.red[r][cq] = ss;
                    ic_epi_sync();
                    const float4 p4 = *reinterpret_cast<const float4 *>(sm.red[r]);
                    scale = rsqrtf((p4.x + p4.y) + (p4.z + p4.w) + a.l2_eps);
                }
                if (live) {
                    __half *dst = a.xhat + (size_t)m * CC + c0 + cb;
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint32_t pk[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) pk[e] = tc::pack_half2(o[c + 2 * e] * scale, o[c + 2 * e + 1] * scale);
                        *reinterpret_cast<uint4 *>(dst + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    }
                    // ---- conv_state_out: the raw inputs of the sequence's last three positions
                    if (a.cs_out) {
                        if (m >= s1 - (KC - 1)) {
                            bf16 *d = a.cs_out + ((size_t)n * (KC - 1) + (m - (s1 - (KC - 1)))) * CC + c0 + cb;
#pragma unroll
                            for (int c = 0; c < 32; c += 8) {
                                __align__(16) bf16 o8[8];
#pragma unroll
                                for (int e = 0; e < 8; ++e) o8[e] = from_f<bf16>(sm.ep[r][cb + c + e]);
                                *reinterpret_cast<uint4 *>(d + c) = *reinterpret_cast<const uint4 *>(o8);
                            }
                        }
                        if (m == s0)                   // positions before the start, from conv_state_in
                            for (int j = 0; j < KC - 1; ++j) {
                                const int pos = s1 - (KC - 1) + j;
                                if (pos >= s0) break;
                                bf16 *d = a.cs_out + ((size_t)n * (KC - 1) + j) * CC + c0 + cb;
                                const bf16 *src = a.cs_in ? a.cs_in + ((size_t)n * (KC - 1) + (pos - s0 + KC - 1)) * CC +
                                                                c0 + cb
                                                          : nullptr;
                                for (int c = 0; c < 32; ++c) d[c] = src ? src[c] : from_f<bf16>(0.0f);
                            }
                    }
                }
            } else if (live && c0 < IC_N) {
                // ---- z, alpha, beta: the projection itself, as bf16
                if (c0 < CC + DI || cb < 2 * HV) {
                    bf16 *dst = c0 < CC + DI ? a.z + (size_t)m * DI + (c0 - CC) + cb
                                             : (cb < HV ? a.alpha + (size_t)m * HV + cb : a.beta + (size_t)m * HV + (cb - HV));
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        __align__(16) bf16 o8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o8[e] = from_f<bf16>(sm.ep[r][cb + c + e]);
                        *reinterpret_cast<uint4 *>(dst + c) = *reinterpret_cast<const uint4 *>(o8);
                    }
                }
            }
            ic_epi_sync();                             // every row's reads of the half are done
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tm, 2 * IC_BN);
    if (tid == 0 && sm.abort) atomicExch(&g_inconv_error, (unsigned int)GDN_ERR_TIMEOUT);
}

// conv_state_out of the sequences with no tokens: conv_state_in (zeros without one).
__global__ void __launch_bounds__(256) in_conv_empty_kernel(const int32_t *__restrict__ cu, int M, const bf16 *cs_in,
                                                            bf16 *cs_out)
{
    const int n = blockIdx.x;
    const int s0 = min(max(cu[n], 0), M), s1 = min(max(cu[n + 1], s0), M);
    if (s1 > s0) return;
    for (int i = threadIdx.x; i < (KC - 1) * CC; i += blockDim.x)
        cs_out[(size_t)n * (KC - 1) * CC + i] = cs_in ? cs_in[(size_t)n * (KC - 1) * CC + i] : from_f<bf16>(0.0f);
}

// ------------------------------------------------------------------ launcher

bool make_bf16_sw128_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_rows);
int sm_count();

cudaError_t launch_in_proj_conv(const float *conv_w, float l2_eps, const void *h, const void *w_in,
                                const int32_t *cu, int N, int M, const void *cs_in, void *cs_out, void *xhat,
                                void *z, void *alpha, void *beta, cudaStream_t s)
{
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            cudaError_t e = cudaFuncSetAttribute(in_conv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)IC_SMEM);
            if (e != cudaSuccess) return e;
            attr_set[dev] = true;
        }
    }
    const int n_sm = sm_count();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    cudaError_t e = cudaSuccess;
    if (M > 0) {
        CUtensorMap mh, mw;
        if (!make_bf16_sw128_map(&mh, h, M, IC_K, IC_BM) || !make_bf16_sw128_map(&mw, w_in, IC_N, IC_K, IC_BN))
            return cudaErrorInvalidValue;
        IcArgs a;
        a.conv_w = conv_w; a.l2_eps = l2_eps; a.cu = cu; a.N = N; a.M = M;
        a.cs_in = static_cast<const bf16 *>(cs_in); a.cs_out = static_cast<bf16 *>(cs_out);
        a.xhat = static_cast<__half *>(xhat);
        a.z = static_cast<bf16 *>(z); a.alpha = static_cast<bf16 *>(alpha); a.beta = static_cast<bf16 *>(beta);
        const int n_work = ((M + IC_ROWS - 1) / IC_ROWS) * IC_NT;
        e = launch_pdl(in_conv_kernel, dim3((unsigned)(n_work < n_sm ? n_work : n_sm)), dim3(IC_THREADS), IC_SMEM, s,
                       mh, mw, a);
    }
    if (e == cudaSuccess && cs_out && N > 0)
        e = launch_pdl(in_conv_empty_kernel, dim3((unsigned)N), dim3(256), 0, s, cu, M,
                       static_cast<const bf16 *>(cs_in), static_cast<bf16 *>(cs_out));
    return e;
}

// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *inconv_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_inconv_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
