// gdn_gated_proj.cu -- the gated RMSNorm . silu(z) and the output projection
// after it in one tensor-core GEMM: section "Output path" of "qwen35moe --
// Forward-Pass Design (Pantheon port)", "SSM block -- Gated-Delta-Net":
//   gated[m][h 128 + j] = y[m][h 128 + j] r[m][h] w_j silu(z[m][h 128 + j]),
//   r[m][h] = (mean_j y[m][h 128 + j]^2 + eps)^-1/2,
//   out[m][n] = sum_k gated[m][k] W[n][k]        (cur = ssm_out . gated)
// The gated rows never go to memory: warps of the GEMM's own CTA compute each
// 128-column head of them straight into the A operand tiles in shared memory,
// and the tensor core reads them from there. The Lily page's "Reduce
// intermediate and state traffic" gives the reason: a fused step saves the
// intermediate's write and its read back.
//
// Design. Output tiles of 128 rows x BN columns (BN = 512 for large M, where
// one fp32 accumulator fills all 512 tensor-memory columns, so the A operand is
// built 2048 / 512 = 4 times per row block; BN = 256 with split K for small M).
// Per CTA (22 warps):
//  - warp 0, lane 0: the TMA producer: per head, (bf16 y) the head's 128 rows of
//    y straight into an A slot, in the 128-byte swizzle the tensor core reads,
//    then the head's weight boxes (256 rows x 64 columns) into a ring of four
//    32 KiB stages;
//  - warp 1, lane 0: MMA issuer: per 64-column K slice, four tcgen05.mma
//    (kind::f16, bf16 operands, M=128, N=256, K=16) per 256 output columns;
//  - warps 2-5: the epilogue: one accumulator row per thread, written as out;
//  - warps 6-21: the A producers. Two 32 KiB A slots take alternate heads.
//    Thread (row r, quarter qq) reads its 32 values of y from the slot and holds
//    its 32 values of z, loaded one head ahead. The four quarters of a row meet
//    in two shuffles for the head's mean square. The thread writes its 32 gated
//    values over its y, as bf16 in the same 128-byte-swizzle layout (row r at
//    128 r, 16-byte chunk c at (c xor r % 8) 16), and fences them for the async
//    proxy. (fp32 y: y and z are loaded into registers.)
// Split K (small M): each tile's 32 heads are split S ways over the S CTAs of a
// cluster; the fp32 partial tiles are summed through distributed shared memory.
// All mbarrier waits are bounded; a wait that gives up records GDN_ERR_TIMEOUT.
#include <cuda.h>

#include <mutex>

#include "gdn_async.cuh"
#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

namespace gdn {

__device__ unsigned int g_gproj_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

constexpr int GP_BM = 128, GP_BK = 64;
constexpr int GP_PRODUCER_WARPS = 16;
constexpr int GP_THREADS = 32 * (6 + GP_PRODUCER_WARPS);
constexpr uint32_t GP_SLICE = GP_BM * GP_BK * 2;        // 16 KiB: 128 rows x 64 bf16
constexpr uint32_t GP_A_SLOT = 2 * GP_SLICE;            // one head (128 columns of K)
constexpr uint32_t GP_B_BOX = 256 * GP_BK * 2;          // 32 KiB: 256 weight rows x 64 columns
constexpr int GP_BSTAGES = 4;
constexpr int GP_NA = 2;                                // A slots
constexpr int GP_HEADS = DI / DV;                       // 32 heads along K
constexpr int GP_N = GDN_HIDDEN;                        // 2048 output features

struct GpSmem {
    alignas(1024) unsigned char a[GP_NA][GP_A_SLOT];     // A slots: head i of the CTA's sequence in slot i % GP_NA
    alignas(1024) unsigned char b[GP_BSTAGES][GP_B_BOX];  // weight stages
    float nw[DV];                                        // the norm weights
    alignas(8) uint64_t a_full[GP_NA], a_empty[GP_NA], b_full[GP_BSTAGES], b_empty[GP_BSTAGES];
    uint64_t y_full[GP_NA];                              // bf16 y: the TMA copy of a head's rows landed
    uint64_t acc_full[2], acc_empty[2];
    int last_b[GP_BSTAGES];                               // last weight box loaded into each stage
    int last_y[GP_NA];                                    // last head whose y was loaded into each slot
    uint32_t tmem;
    int abort;
};
constexpr size_t GP_SMEM = sizeof(GpSmem) + 1024;        // + slack to align the block to 1024 bytes
static_assert(GP_SMEM <= 232448, "gated projection shared memory");

struct GpArgs {
    const void *y, *z;          // [M][4096], type TY
    const float *norm_w;        // [128]
    float eps;
    void *out;                  // [M][2048], type TO
    int M, splits;
};

__device__ __forceinline__ float silu_tanh(float z)
{
    // z sigmoid(z) = (z / 2)(1 + tanh(z / 2)), with the hardware tanh
    // approximation (absolute error about 5e-4 on tanh, far below the bf16
    // rounding of the operand it feeds)
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * z));
    const float hz = 0.5f * z;
    return fmaf(hz, th, hz);
}

__device__ __forceinline__ void bf16x8_to_f(const uint4 u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w[e] << 16);
        f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// fp32 y: one producer thread's quarter of a head row (32 columns) of y and z,
// loaded into registers before the thread computes anything. (bf16 y arrives
// by TMA in the operand slot instead.)
struct RowQuarterF32 {
    float4 y[8], z[8];
    __device__ __forceinline__ void load(const float *yr, const float *zr)
    {
#pragma unroll
        for (int c = 0; c < 8; ++c) y[c] = __ldg(reinterpret_cast<const float4 *>(yr) + c);
#pragma unroll
        for (int c = 0; c < 8; ++c) z[c] = __ldg(reinterpret_cast<const float4 *>(zr) + c);
    }
    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int c = 0; c < 8; ++c) y[c] = z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __device__ __forceinline__ void get(int c, float (&yf)[8], float (&zf)[8]) const
    {
        const float4 a = y[2 * c], b = y[2 * c + 1], p = z[2 * c], q = z[2 * c + 1];
        yf[0] = a.x; yf[1] = a.y; yf[2] = a.z; yf[3] = a.w; yf[4] = b.x; yf[5] = b.y; yf[6] = b.z; yf[7] = b.w;
        zf[0] = p.x; zf[1] = p.y; zf[2] = p.z; zf[3] = p.w; zf[4] = q.x; zf[5] = q.y; zf[6] = q.z; zf[7] = q.w;
    }
};

template <typename TY, typename TO, int BN>
__global__ void __launch_bounds__(GP_THREADS, 1) gated_proj_kernel(const __grid_constant__ CUtensorMap mw,
                                                                   const __grid_constant__ CUtensorMap my,
                                                                   const GpArgs a)
{
    constexpr int NACC = 512 / BN;                     // accumulators that fit in 512 columns
    constexpr int NH = BN / 256;                       // N=256 products per K step
    constexpr int PART_LD = BN + 4;                    // fp32 partial row stride (split K)
    static_assert(BN == 256 || BN == 512, "tile width");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *blk = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    GpSmem &sm = *reinterpret_cast<GpSmem *>(blk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = a.M, splits = a.splits;
    const int n_tiles = GP_N / BN;
    const bool split = splits > 1;
    const int n_work = split ? 1 : ((M + GP_BM - 1) / GP_BM) * n_tiles;
    const int w0 = split ? (int)blockIdx.x / splits : (int)blockIdx.x;
    const int wstep = split ? 1 : (int)gridDim.x;
    const int wend = split ? w0 + 1 : n_work;
    const int kh_n = GP_HEADS / splits;                // heads per work item
    const int kh0 = split ? ((int)blockIdx.x % splits) * kh_n : 0;
    const volatile int &aborted = sm.abort;

    if (warp == 1) {
        tc::tmem_alloc(smem_u32(&sm.tmem), 512);
        tc::tmem_relinquish();
    }
    if (tid < DV) sm.nw[tid] = __ldg(a.norm_w + tid);   // a parameter, not produced by the kernel ahead
    if (tid == 0) {
        for (int s = 0; s < GP_BSTAGES; ++s) {
            mbar_init(smem_u32(&sm.b_full[s]), 1);
            mbar_init(smem_u32(&sm.b_empty[s]), 1);
            sm.last_b[s] = -1;
        }
        for (int b = 0; b < GP_NA; ++b) {
            mbar_init(smem_u32(&sm.a_full[b]), GP_PRODUCER_WARPS);
            mbar_init(smem_u32(&sm.y_full[b]), 1);
            mbar_init(smem_u32(&sm.a_empty[b]), 1);
            sm.last_y[b] = -1;
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sm.acc_full[b]), 1);
            mbar_init(smem_u32(&sm.acc_empty[b]), 128);
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = sm.tmem;
    grid_dep_wait();                                   // y and z come from the kernel ahead
    grid_dep_launch();

    if (warp == 0) {
        // ---- TMA producer: per head, (bf16 y) the head's y rows into its A slot
        //      once the slot's previous head has been multiplied, then the
        //      weight boxes of the head
        if (lane == 0) {
            int ib = 0, ia = 0;
            for (int w = w0; w < wend && !aborted; w += wstep) {
                const int nt = w % n_tiles, mt = w / n_tiles;
                for (int hh = kh0; hh < kh0 + kh_n && !aborted; ++hh, ++ia) {
                    if constexpr (sizeof(TY) == 2) {
                        const int sa = ia % GP_NA, u = ia / GP_NA;
                        if (u >= 1 && !mbar_wait_bounded(smem_u32(&sm.a_empty[sa]), (uint32_t)((u - 1) & 1)))
                            sm.abort = 1;
                        if (aborted) break;
                        mbar_arrive_expect_tx(smem_u32(&sm.y_full[sa]), GP_A_SLOT);
                        tma_load_2d(smem_u32(sm.a[sa]), &my, hh * DV, mt * GP_BM, smem_u32(&sm.y_full[sa]));
                        tma_load_2d(smem_u32(sm.a[sa]) + GP_SLICE, &my, hh * DV + GP_BK, mt * GP_BM,
                                    smem_u32(&sm.y_full[sa]));
                        sm.last_y[sa] = ia;
                    }
                    for (int h = 0; h < 2 && !aborted; ++h)
                        for (int nh = 0; nh < NH; ++nh, ++ib) {
                            const int s = ib % GP_BSTAGES;
                            if (ib >= GP_BSTAGES &&
                                !mbar_wait_bounded(smem_u32(&sm.b_empty[s]), (uint32_t)((ib / GP_BSTAGES - 1) & 1)))
                                sm.abort = 1;
                            if (aborted) break;
                            mbar_arrive_expect_tx(smem_u32(&sm.b_full[s]), GP_B_BOX);
                            tma_load_2d(smem_u32(sm.b[s]), &mw, (2 * hh + h) * GP_BK, nt * BN + 256 * nh,
                                        smem_u32(&sm.b_full[s]));
                            sm.last_b[s] = ib;
                        }
                }
            }
            if (aborted) {                             // let the copies in flight land before the CTA exits
                for (int s = 0; s < GP_BSTAGES; ++s)
                    if (sm.last_b[s] >= 0)
                        mbar_wait_bounded(smem_u32(&sm.b_full[s]), (uint32_t)((sm.last_b[s] / GP_BSTAGES) & 1));
                for (int s = 0; s < GP_NA; ++s)
                    if (sm.last_y[s] >= 0)
                        mbar_wait_bounded(smem_u32(&sm.y_full[s]), (uint32_t)((sm.last_y[s] / GP_NA) & 1));
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::instr_desc(tc::FMT_BF16, GP_BM, 256);
            int ib = 0, ia = 0, ti = 0;
            for (int w = w0; w < wend && !aborted; w += wstep, ++ti) {
                const int ab = ti % NACC;
                if (ti >= NACC &&
                    !mbar_wait_bounded(smem_u32(&sm.acc_empty[ab]), (uint32_t)((ti / NACC - 1) & 1)))
                    sm.abort = 1;
                tc::fence_after_sync();
                const uint32_t d = tm + (uint32_t)(BN * ab);
                for (int hh = kh0; hh < kh0 + kh_n && !aborted; ++hh, ++ia) {
                    const int sa = ia % GP_NA;
                    if (!mbar_wait_bounded(smem_u32(&sm.a_full[sa]), (uint32_t)((ia / GP_NA) & 1))) sm.abort = 1;
                    tc::fence_after_sync();
                    for (int h = 0; h < 2 && !aborted; ++h)
                        for (int nh = 0; nh < NH; ++nh, ++ib) {
                            const int s = ib % GP_BSTAGES;
                            if (!mbar_wait_bounded(smem_u32(&sm.b_full[s]), (uint32_t)((ib / GP_BSTAGES) & 1)))
                                sm.abort = 1;
                            if (aborted) break;
                            tc::fence_after_sync();
                            const uint64_t ad = tc::sw128_desc(smem_u32(sm.a[sa]) + (uint32_t)h * GP_SLICE);
                            const uint64_t bd = tc::sw128_desc(smem_u32(sm.b[s]));
#pragma unroll
                            for (int k = 0; k < GP_BK / 16; ++k)   // 16 bf16 = 32 bytes = 2 descriptor units
                                tc::mma_f16(d + 256u * nh, ad + 2u * k, bd + 2u * k, idesc,
                                            (hh > kh0 || h > 0 || k > 0) ? 1u : 0u);
                            tc::mma_commit(smem_u32(&sm.b_empty[s]));
                        }
                    tc::mma_commit(smem_u32(&sm.a_empty[sa]));   // the A slot is free once these have read it
                }
                if (aborted) break;
                tc::mma_commit(smem_u32(&sm.acc_full[ab]));
            }
        }
    } else if (warp >= 6) {
        // ---- A producers: head i of the CTA's sequence goes to slot i % GP_NA.
        //      Thread (row r, quarter qq) owns columns [32 qq, 32 qq + 32) of
        //      row r; the 8 lanes of a quarter-warp hold 8 consecutive rows, so
        //      their 16-byte accesses fall on distinct banks in the swizzle.
        const int p = tid - 6 * 32;                    // 0..511
        const int r = 8 * (p >> 5) + (lane & 7), qq = lane >> 3;
        const int hf = qq >> 1;                        // K slice (64 columns) of the quarter
        const TY *zs = static_cast<const TY *>(a.z);
        const int n_items = ((wend - w0 + wstep - 1) / wstep) * kh_n;
        auto row_of = [&](int i) { return ((w0 + (i / kh_n) * wstep) / n_tiles) * GP_BM + r; };
        auto col_of = [&](int i) { return (size_t)(kh0 + i % kh_n) * DV + 32 * qq; };
        auto chunk_at = [&](int sa, int c) {           // 16-byte chunk c of this thread's quarter in slot sa
            const uint32_t chunk = (uint32_t)(4 * (qq & 1) + c);
            return sm.a[sa] + (uint32_t)hf * GP_SLICE + (uint32_t)r * 128u + ((chunk ^ (uint32_t)(r & 7)) << 4);
        };
        auto gate = [&](const float (&yf)[8], const float (&zf)[8], float rr, int c) {
            const float4 w0v = *reinterpret_cast<const float4 *>(sm.nw + 32 * qq + 8 * c);
            const float4 w1v = *reinterpret_cast<const float4 *>(sm.nw + 32 * qq + 8 * c + 4);
            const float nw[8] = {w0v.x, w0v.y, w0v.z, w0v.w, w1v.x, w1v.y, w1v.z, w1v.w};
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pk[e] = pack_bf16x2(yf[2 * e] * rr * nw[2 * e] * silu_tanh(zf[2 * e]),
                                    yf[2 * e + 1] * rr * nw[2 * e + 1] * silu_tanh(zf[2 * e + 1]));
            return make_uint4(pk[0], pk[1], pk[2], pk[3]);
        };
        if constexpr (sizeof(TY) == 2) {
            // y arrives by TMA in the slot itself (the operand layout); z is
            // loaded into registers one head ahead. The gated values replace y
            // in place: each thread reads and writes only its own chunks.
            uint4 zq[4];
            auto load_z = [&](int i) {
                const int m = row_of(i);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    zq[c] = m < M ? __ldg(reinterpret_cast<const uint4 *>(zs + (size_t)m * DI + col_of(i)) + c)
                                  : make_uint4(0u, 0u, 0u, 0u);
            };
            if (n_items > 0) load_z(0);
#pragma unroll 1
            for (int i = 0; i < n_items && !aborted; ++i) {
                const int sa = i % GP_NA, u = i / GP_NA;
                if (!mbar_wait_sleep(smem_u32(&sm.y_full[sa]), (uint32_t)(u & 1))) sm.abort = 1;
                if (aborted) break;
                float yf[4][8];
                float ss = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    bf16x8_to_f(*reinterpret_cast<const uint4 *>(chunk_at(sa, c)), yf[c]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(yf[c][e], yf[c][e], ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 8);
                ss += __shfl_xor_sync(0xffffffffu, ss, 16);
                const float rr = rsqrtf(ss * (1.0f / DV) + a.eps);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float zf[8];
                    bf16x8_to_f(zq[c], zf);
                    *reinterpret_cast<uint4 *>(chunk_at(sa, c)) = gate(yf[c], zf, rr, c);
                }
                fence_proxy_async_smem();              // the tensor core reads these through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.a_full[sa]));
                // the next head's z after the fence, which would otherwise wait for these loads
                if (i + 1 < n_items) load_z(i + 1);
            }
        } else {
            // fp32 y and z: both loaded into registers, the slot waited for here
            const float *ys = static_cast<const float *>(a.y);
            const float *zf32 = static_cast<const float *>(a.z);
#pragma unroll 1
            for (int i = 0; i < n_items && !aborted; ++i) {
                const int m = row_of(i);
                RowQuarterF32 rq;
                if (m < M) rq.load(ys + (size_t)m * DI + col_of(i), zf32 + (size_t)m * DI + col_of(i));
                else rq.zero();
                float ss = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float yf[8], zf[8];
                    rq.get(c, yf, zf);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(yf[e], yf[e], ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 8);
                ss += __shfl_xor_sync(0xffffffffu, ss, 16);
                const float rr = rsqrtf(ss * (1.0f / DV) + a.eps);
                const int sa = i % GP_NA, u = i / GP_NA;
                if (u >= 1 && !mbar_wait_sleep(smem_u32(&sm.a_empty[sa]), (uint32_t)((u - 1) & 1))) sm.abort = 1;
                if (aborted) break;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float yf[8], zf[8];
                    rq.get(c, yf, zf);
                    *reinterpret_cast<uint4 *>(chunk_at(sa, c)) = gate(yf, zf, rr, c);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sm.a_full[sa]));
            }
        }
    } else {
        // ---- epilogue: warp w (2..5) owns TMEM lanes 32 (w % 4) .. + 31, one row each
        const int q = warp & 3;
        const int row = 32 * q + lane;
        int ti = 0;
        if (split) {                                   // this CTA's fp32 partial tile to shared memory
            if (!mbar_wait_bounded(smem_u32(&sm.acc_full[0]), 0)) sm.abort = 1;
            tc::fence_after_sync();
            if (!aborted) {
                float *part = reinterpret_cast<float *>(sm.a[0]) + row * PART_LD;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    float v[32];
                    tc::tmem_ld32(tc::tmem_addr(tm, 32 * q, c), v);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        reinterpret_cast<float4 *>(part + c)[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                }
            }
        }
        for (int w = w0; w < wend && !split; w += wstep, ++ti) {
            const int ab = ti % NACC;
            if (!mbar_wait_bounded(smem_u32(&sm.acc_full[ab]), (uint32_t)((ti / NACC) & 1))) sm.abort = 1;
            if (aborted) break;
            tc::fence_after_sync();
            const int m = (w / n_tiles) * GP_BM + row, nt = w % n_tiles;
            TO *dst = static_cast<TO *>(a.out) + (size_t)m * GP_N + (size_t)nt * BN;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                float v[32];
                tc::tmem_ld32(tc::tmem_addr(tm + (uint32_t)(BN * ab), 32 * q, c), v);
                tc::wait_ld();
                if (m < M) {
                    if constexpr (sizeof(TO) == 4) {
                        float4 *d4 = reinterpret_cast<float4 *>(dst + c);
#pragma unroll
                        for (int e = 0; e < 8; ++e) d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                    } else {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + c);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            d4[e] = make_uint4(pack_bf16x2(v[8 * e], v[8 * e + 1]), pack_bf16x2(v[8 * e + 2], v[8 * e + 3]),
                                               pack_bf16x2(v[8 * e + 4], v[8 * e + 5]), pack_bf16x2(v[8 * e + 6], v[8 * e + 7]));
                    }
                }
            }
            tc::fence_before_sync();
            mbar_arrive(smem_u32(&sm.acc_empty[ab]));  // the MMA warp may refill this accumulator
        }
    }
    if (split) {
        // ---- the cluster's reduction: CTA r writes rows [r 128/S, (r+1) 128/S)
        //      of the tile, each the sum of the S partials
        cluster_sync_all();                            // every partial of the cluster is staged
        if (warp >= 2 && warp < 6 && !aborted) {
            const int t = tid - 64;                    // 0..127
            const int rows = GP_BM / splits, r0 = ((int)blockIdx.x % splits) * rows;
            const int mt = w0 / n_tiles, nt = w0 % n_tiles;
            const uint32_t pbase = smem_u32(sm.a[0]);
            for (int f = t; f < rows * (BN / 4); f += 128) {
                const int rr = r0 + f / (BN / 4), col = 4 * (f % (BN / 4));
                const uint32_t off = pbase + (uint32_t)((rr * PART_LD + col) * 4);
                float4 p4[8];                          // all S remote loads in flight before the sum
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    if (s < splits) p4[s] = ld_cluster_f32x4(mapa_shared(off, (uint32_t)s));
                float4 acc = p4[0];
#pragma unroll
                for (int s = 1; s < 8; ++s)
                    if (s < splits) {
                        acc.x += p4[s].x; acc.y += p4[s].y; acc.z += p4[s].z; acc.w += p4[s].w;
                    }
                const int m = mt * GP_BM + rr, n = nt * BN + col;
                if (m < M) {
                    TO *dst = static_cast<TO *>(a.out) + (size_t)m * GP_N + n;
                    if constexpr (sizeof(TO) == 4) {
                        *reinterpret_cast<float4 *>(dst) = acc;
                    } else {
                        *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
                    }
                }
            }
        }
        cluster_sync_all();                            // no CTA leaves while others read its partial
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tm, 512);
    if (tid == 0 && sm.abort) atomicExch(&g_gproj_error, (unsigned int)GDN_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ launcher

bool make_bf16_sw128_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_rows);
int sm_count();

template <typename TY, typename TO, int BN>
static bool gp_attr()
{
    return cudaFuncSetAttribute(gated_proj_kernel<TY, TO, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)GP_SMEM) == cudaSuccess;
}

// Per device, once: the shared-memory attribute of every instance, and how many
// clusters of 2, 4 and 8 CTAs can be resident at once.
struct GpDevice {
    int max_clusters[3];
};

static const GpDevice *gp_device()
{
    static GpDevice info[64];
    static bool ready[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
        if (!gp_attr<bf16, bf16, 256>() || !gp_attr<bf16, float, 256>() || !gp_attr<float, bf16, 256>() ||
            !gp_attr<float, float, 256>() || !gp_attr<bf16, bf16, 512>() || !gp_attr<bf16, float, 512>() ||
            !gp_attr<float, bf16, 512>() || !gp_attr<float, float, 512>())
            return nullptr;
        for (int k = 0; k < 3; ++k) {
            const int cs = 2 << k;
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(cs);
            q.blockDim = dim3(GP_THREADS);
            q.dynamicSmemBytes = GP_SMEM;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = (unsigned)cs;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, gated_proj_kernel<bf16, bf16, 256>, &q) != cudaSuccess) {
                cudaGetLastError();                    // a refused query: never split this far
                n = 0;
            }
            info[dev].max_clusters[k] = n;
        }
        ready[dev] = true;
    }
    return &info[dev];
}

template <typename TY, typename TO>
static cudaError_t launch_gp_typed(const CUtensorMap &mw, const CUtensorMap &my, const GpArgs &args, int bn,
                                   int grid, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(GP_THREADS);
    cfg.dynamicSmemBytes = GP_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)args.splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = args.splits > 1 ? 2 : 1;
    if (bn == 512) return cudaLaunchKernelEx(&cfg, gated_proj_kernel<TY, TO, 512>, mw, my, args);
    return cudaLaunchKernelEx(&cfg, gated_proj_kernel<TY, TO, 256>, mw, my, args);
}

cudaError_t launch_gated_out_proj(const float *norm_w, float eps, const void *y, const void *z, const void *w,
                                  void *out, int M, gdn_dtype act, gdn_dtype out_dt, cudaStream_t s)
{
    if (M <= 0) return cudaSuccess;
    const int n_sm = sm_count();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    const GpDevice *gd = gp_device();
    if (!gd) return cudaErrorInvalidDevice;
    CUtensorMap mw, my;
    if (!make_bf16_sw128_map(&mw, w, GP_N, DI, 256)) return cudaErrorInvalidValue;
    // bf16 y is read by TMA in the operand layout (fp32 y: the map is not used)
    if (!make_bf16_sw128_map(&my, act == GDN_BF16 ? y : w, act == GDN_BF16 ? M : GP_N, DI, GP_BM))
        return cudaErrorInvalidValue;
    const int m_tiles = (M + GP_BM - 1) / GP_BM;
    GpArgs args;
    args.y = y; args.z = z; args.norm_w = norm_w; args.eps = eps; args.out = out; args.M = M; args.splits = 1;
    int bn = 512, grid;
    if (m_tiles * (GP_N / 512) * 2 > n_sm) {           // enough 512-wide tiles to fill the GPU
        const int n_work = m_tiles * (GP_N / 512);
        grid = n_work < n_sm ? n_work : n_sm;
    } else {
        // 256-wide tiles; split K (2, 4 or 8 ways) while the tiles fill less than
        // half of the SMs, and only as far as every cluster can be resident at once
        bn = 256;
        const int n_work = m_tiles * (GP_N / 256);
        int sp = 1;
        while (sp < 8 && n_work * sp * 2 <= n_sm && gd->max_clusters[sp == 1 ? 0 : sp == 2 ? 1 : 2] >= n_work)
            sp *= 2;
        args.splits = sp;
        grid = sp > 1 ? n_work * sp : (n_work < n_sm ? n_work : n_sm);
    }
    if (act == GDN_F32)
        return out_dt == GDN_F32 ? launch_gp_typed<float, float>(mw, my, args, bn, grid, s)
                                 : launch_gp_typed<float, bf16>(mw, my, args, bn, grid, s);
    return out_dt == GDN_F32 ? launch_gp_typed<bf16, float>(mw, my, args, bn, grid, s)
                             : launch_gp_typed<bf16, bf16>(mw, my, args, bn, grid, s);
}

// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *gproj_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_gproj_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
