// gdn_gemm.cu -- the dense projections around the mixer on 5th-generation
// tensor cores: y[m][n] = sum_k x[m][k] w[n][k], bf16 operands, fp32
// accumulation. Both are in "qwen35moe -- Forward-Pass Design (Pantheon port)",
// section "SSM block -- Gated-Delta-Net":
//  - the input projections (from the normed x, K = n_embd 2048): attn_qkv ->
//    qkv [8192], attn_gate -> z [4096], ssm_alpha -> alpha [32], ssm_beta -> beta
//    [32], computed as one GEMM over the stacked weight [12352][2048], whose
//    epilogue writes each column range to its own array;
//  - the output projection "cur = ssm_out . gated" (section "Output path"),
//    4096 -> 2048.
//
// Design. A persistent grid walks output tiles of 128 rows x 256 columns, or
// x 128 columns when the 256-wide tiles would fill less than half the GPU (the
// last column tile may be partial: weight rows past N read as zero and their
// columns are not stored). Per CTA:
//  - warp 0, lane 0: the TMA producer. 2-D tensor-map copies bring 64-wide K
//    slices of x (128 x 64) and w (256 x 64) into a ring of four shared-memory
//    stages in the 128-byte-swizzle layout the tensor core reads directly.
//  - warp 1, lane 0: the MMA issuer. Per K slice, four tcgen05.mma (kind::f16,
//    M=128, N=256, K=16) accumulate into one of two 256-column fp32
//    accumulators in tensor memory; commits release the stage, and after the
//    last slice, the accumulator.
//  - warps 2..5: the epilogue. Each thread owns one accumulator row (its TMEM
//    lane) and writes its outputs 32 columns at a time to the array that owns
//    those columns, while the MMA warp already fills the other accumulator with
//    the next tile.
// Split K. When the tiles are too few to fill the GPU (a decode batch), each
// tile's K range is split S ways (S = 2, 4 or 8) over the S CTAs of a
// cluster, one tile per CTA. Each CTA stages its fp32 partial tile in the
// shared memory its stages no longer need; after a cluster barrier, CTA r sums
// rows [r 128/S, (r+1) 128/S) over all S partials through distributed shared
// memory and writes them.
// All mbarrier waits are bounded; a wait that gives up records GDN_ERR_TIMEOUT.
#include <cuda.h>

#include <mutex>

#include "gdn_async.cuh"
#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

namespace gdn {

__device__ unsigned int g_gemm_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

constexpr int GM_BM = 128, GM_BK = 64;
constexpr uint32_t GM_A_BYTES = GM_BM * GM_BK * 2;        // 16 KiB
constexpr int GM_THREADS = 192;                   // TMA warp, MMA warp, 4 epilogue warps
static_assert(GM_BK == 64, "K slices are the 64-column boxes of make_bf16_sw128_map");

// Tile width BN = 256 (large M), or 128 when the 256-wide tiles would leave
// most SMs idle (a decode batch): twice the tiles, each half as long to issue.
template <int BN>
struct GemmCfg {
    static constexpr int STAGES = BN == 256 ? 4 : 6;
    static constexpr uint32_t B_BYTES = BN * GM_BK * 2;
    static constexpr uint32_t STAGE_BYTES = GM_A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = 2 * BN;         // two accumulators
    static constexpr int PART_LD = BN + 4;                // fp32 partial row stride (floats): rows fall on other banks
    static_assert(GM_BM * PART_LD * 4 <= STAGES * STAGE_BYTES, "split-K partial fits the stages");
    static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1024-byte aligned");
};

// Where the GEMM's output columns go: columns [c0[s], c0[s+1]) are written to
// ptr[s] as rows of ld[s] elements (column c lands at ptr[s][m * ld[s] + c - c0[s]]).
// Every boundary is a multiple of 32, so a 32-column chunk has one owner.
struct ProjOut {
    void *ptr[4];
    int c0[5];
    int ld[4];
    int nseg;
};

// Address of output element (m, n): the segment holding column n is picked by
// a compare chain with static indices, so the kernel parameter stays in the
// constant bank (a runtime index would copy the struct to local memory).
template <typename TO>
__device__ __forceinline__ TO *proj_out_addr(const ProjOut &out, int m, int n)
{
    void *p = out.ptr[0];
    int ld = out.ld[0], c0 = out.c0[0];
#pragma unroll
    for (int i = 1; i < 4; ++i)
        if (i < out.nseg && n >= out.c0[i]) {
            p = out.ptr[i];
            ld = out.ld[i];
            c0 = out.c0[i];
        }
    return static_cast<TO *>(p) + (size_t)m * ld + (n - c0);
}

template <int BN>
struct GemmSmem {
    static constexpr int STAGES = GemmCfg<BN>::STAGES;
    alignas(1024) unsigned char stage[STAGES][GemmCfg<BN>::STAGE_BYTES];   // A tile | B tile, 1024-byte aligned
    alignas(8) uint64_t full[STAGES], empty[STAGES];
    uint64_t acc_full[2], acc_empty[2];
    int last_it[STAGES];                          // last K slice loaded into each stage (for an abort)
    uint32_t tmem;
    int abort;
};
template <int BN>
constexpr size_t gm_smem() { return sizeof(GemmSmem<BN>) + 1024; }   // + slack to align the block to 1024 bytes

template <typename TO, int BN>
__global__ void __launch_bounds__(GM_THREADS, 1) proj_kernel(const __grid_constant__ CUtensorMap mx,
                                                             const __grid_constant__ CUtensorMap mw,
                                                             const ProjOut out, int M, int N, int K, int splits)
{
    using Cfg = GemmCfg<BN>;
    constexpr int GM_BN = BN, GM_STAGES = Cfg::STAGES, GM_PART_LD = Cfg::PART_LD;
    constexpr uint32_t GM_TMEM_COLS = Cfg::TMEM_COLS, GM_STAGE_BYTES = Cfg::STAGE_BYTES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *blk = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    GemmSmem<BN> &sm = *reinterpret_cast<GemmSmem<BN> *>(blk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_tiles = (N + GM_BN - 1) / GM_BN;
    // persistent mode: CTAs stride over the tiles with all K slices each;
    // split mode: CTA = (tile blockIdx.x / splits, K split blockIdx.x % splits)
    const bool split = splits > 1;
    const int n_work = split ? 1 : ((M + GM_BM - 1) / GM_BM) * n_tiles;
    const int w0 = split ? (int)blockIdx.x / splits : (int)blockIdx.x;
    const int wstep = split ? 1 : (int)gridDim.x;
    const int wend = split ? w0 + 1 : n_work;
    const int kbn = K / GM_BK / splits;                // K slices per work item
    const int kb0 = split ? ((int)blockIdx.x % splits) * kbn : 0;
    const volatile int &aborted = sm.abort;

    if (warp == 1) {
        tc::tmem_alloc(smem_u32(&sm.tmem), GM_TMEM_COLS);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int s = 0; s < GM_STAGES; ++s) {
            mbar_init(smem_u32(&sm.full[s]), 1);
            mbar_init(smem_u32(&sm.empty[s]), 1);
            sm.last_it[s] = -1;
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
    grid_dep_wait();                                   // the operands may come from the kernel ahead
    grid_dep_launch();

    if (warp == 0) {
        // ---- TMA producer
        if (lane == 0) {
            int it = 0;                                // K slices issued so far, over all tiles
            for (int w = w0; w < wend && !aborted; w += wstep) {
                const int mt = w / n_tiles, nt = w % n_tiles;
                for (int kb = kb0; kb < kb0 + kbn; ++kb, ++it) {
                    const int s = it % GM_STAGES;
                    if (it >= GM_STAGES &&
                        !mbar_wait_bounded(smem_u32(&sm.empty[s]), (uint32_t)((it / GM_STAGES - 1) & 1)))
                        sm.abort = 1;
                    if (aborted) break;
                    const uint32_t dst = smem_u32(sm.stage[s]);
                    mbar_arrive_expect_tx(smem_u32(&sm.full[s]), GM_STAGE_BYTES);
                    tma_load_2d(dst, &mx, kb * GM_BK, mt * GM_BM, smem_u32(&sm.full[s]));
                    tma_load_2d(dst + GM_A_BYTES, &mw, kb * GM_BK, nt * GM_BN, smem_u32(&sm.full[s]));
                    sm.last_it[s] = it;
                }
            }
            if (aborted)                               // let the copies in flight land before the CTA exits
                for (int s = 0; s < GM_STAGES; ++s)
                    if (sm.last_it[s] >= 0)
                        mbar_wait_bounded(smem_u32(&sm.full[s]), (uint32_t)((sm.last_it[s] / GM_STAGES) & 1));
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::instr_desc(tc::FMT_BF16, GM_BM, GM_BN);
            int it = 0, ti = 0;
            for (int w = w0; w < wend && !aborted; w += wstep, ++ti) {
                const int ab = ti & 1;
                if (ti >= 2 && !mbar_wait_bounded(smem_u32(&sm.acc_empty[ab]), (uint32_t)(((ti >> 1) - 1) & 1)))
                    sm.abort = 1;
                tc::fence_after_sync();
                const uint32_t d = tm + (uint32_t)(GM_BN * ab);
                for (int kb = 0; kb < kbn; ++kb, ++it) {
                    const int s = it % GM_STAGES;
                    if (!mbar_wait_bounded(smem_u32(&sm.full[s]), (uint32_t)((it / GM_STAGES) & 1))) sm.abort = 1;
                    if (aborted) break;
                    tc::fence_after_sync();
                    const uint32_t a0 = smem_u32(sm.stage[s]);
                    const uint64_t ad = tc::sw128_desc(a0), bd = tc::sw128_desc(a0 + GM_A_BYTES);
#pragma unroll
                    for (int k = 0; k < GM_BK / 16; ++k)      // K step of 16 bf16 = 32 bytes = 2 descriptor units
                        tc::mma_f16(d, ad + 2u * k, bd + 2u * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
                    tc::mma_commit(smem_u32(&sm.empty[s]));   // the stage is free once these have read it
                }
                if (aborted) break;
                tc::mma_commit(smem_u32(&sm.acc_full[ab]));
            }
        }
    } else {
        // ---- epilogue: thread (lane quarter warp % 4, lane) owns accumulator row 32 q + lane
        const int q = warp & 3;
        const int row = 32 * q + lane;
        int ti = 0;
        if (split) {                                   // stage this CTA's fp32 partial tile in shared memory
            if (!mbar_wait_bounded(smem_u32(&sm.acc_full[0]), 0)) sm.abort = 1;
            tc::fence_after_sync();
            float *part = reinterpret_cast<float *>(sm.stage[0]) + row * GM_PART_LD;
            for (int c = 0; c < GM_BN; c += 64) {      // four TMEM loads per wait
                float v[64];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, c + 16 * k), *reinterpret_cast<float(*)[16]>(v + 16 * k));
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    reinterpret_cast<float4 *>(part + c)[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
            }
        }
        for (int w = w0; w < wend && !split; w += wstep, ++ti) {
            const int ab = ti & 1;
            const int mt = w / n_tiles, nt = w % n_tiles;
            if (!mbar_wait_bounded(smem_u32(&sm.acc_full[ab]), (uint32_t)((ti >> 1) & 1))) sm.abort = 1;
            if (aborted) break;
            tc::fence_after_sync();
            const int m = mt * GM_BM + row;
#pragma unroll 2
            for (int c = 0; c < GM_BN; c += 32) {
                float v[32];
                tc::tmem_ld16(tc::tmem_addr(tm + (uint32_t)(GM_BN * ab), 32 * q, c), *reinterpret_cast<float(*)[16]>(v));
                tc::tmem_ld16(tc::tmem_addr(tm + (uint32_t)(GM_BN * ab), 32 * q, c + 16),
                              *reinterpret_cast<float(*)[16]>(v + 16));
                tc::wait_ld();
                const int n = nt * GM_BN + c;          // first output column of this chunk
                TO *dst = proj_out_addr<TO>(out, m, n);
                if (m < M && n < N) {
                    if (sizeof(TO) == 4) {
                        float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
                        for (int e = 0; e < 8; ++e) d4[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
                    } else {
                        __align__(16) bf16 o[32];
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = from_f<bf16>(v[e]);
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                        for (int e = 0; e < 4; ++e) d4[e] = reinterpret_cast<const uint4 *>(o)[e];
                    }
                }
            }
            tc::fence_before_sync();
            mbar_arrive(smem_u32(&sm.acc_empty[ab]));  // the MMA warp may refill this accumulator
        }
    }
    if (split) {
        // ---- the cluster's reduction: CTA r writes rows [r 128/S, (r+1) 128/S) of
        //      the tile, each the sum of the S partials
        cluster_sync_all();                            // every partial of the cluster is staged
        if (warp >= 2 && !aborted) {
            const int t = tid - 64;                    // 0..127
            const int rows = GM_BM / splits, r0 = ((int)blockIdx.x % splits) * rows;
            const int mt = w0 / n_tiles, nt = w0 % n_tiles;
            const uint32_t pbase = smem_u32(sm.stage[0]);
            for (int f = t; f < rows * (GM_BN / 4); f += 128) {
                const int rr = r0 + f / (GM_BN / 4), col = 4 * (f % (GM_BN / 4));
                const uint32_t off = pbase + (uint32_t)((rr * GM_PART_LD + col) * 4);
                float4 p4[8];                          // all S remote loads in flight before the sum
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r < splits) p4[r] = ld_cluster_f32x4(mapa_shared(off, (uint32_t)r));
                float4 acc = p4[0];
#pragma unroll
                for (int r = 1; r < 8; ++r)
                    if (r < splits) {
                        acc.x += p4[r].x; acc.y += p4[r].y; acc.z += p4[r].z; acc.w += p4[r].w;
                    }
                const int m = mt * GM_BM + rr, n = nt * GM_BN + col;
                if (m < M && n < N) {
                    TO *dst = proj_out_addr<TO>(out, m, n);
                    if (sizeof(TO) == 4) {
                        *reinterpret_cast<float4 *>(dst) = acc;
                    } else {
                        __align__(8) bf16 o4[4] = {from_f<bf16>(acc.x), from_f<bf16>(acc.y), from_f<bf16>(acc.z),
                                                   from_f<bf16>(acc.w)};
                        *reinterpret_cast<uint2 *>(dst) = *reinterpret_cast<const uint2 *>(o4);
                    }
                }
            }
        }
        cluster_sync_all();                            // no CTA leaves while others read its partial
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tm, GM_TMEM_COLS);
    if (tid == 0 && sm.abort) atomicExch(&g_gemm_error, (unsigned int)GDN_ERR_TIMEOUT);
}

// ------------------------------------------------------------------ launcher

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime.
static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

static bool encode_bf16_2d(CUtensorMap *map, const void *base, long long rows, int cols, int box_cols, int box_rows,
                           CUtensorMapSwizzle swz)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 matrix [rows][cols] read in boxes of 64 columns x box_rows
// rows, 128-byte swizzle; elements past either end read as zero.
bool make_bf16_sw128_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_rows)
{
    return encode_bf16_2d(map, base, rows, cols, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_bf16_plain_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_cols, int box_rows)
{
    return encode_bf16_2d(map, base, rows, cols, box_cols, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

int sm_count();

// Per-device set-up of the projection kernels, done once: the shared-memory
// attribute, and how many clusters of 2, 4 and 8 CTAs can be resident at once,
// for each tile width.
struct ProjDevice {
    int max_clusters[2][3];   // [BN == 128][cluster size 2, 4, 8]
};

template <int BN>
static bool proj_setup(int (&max_clusters)[3])
{
    if (cudaFuncSetAttribute(proj_kernel<float, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gm_smem<BN>()) != cudaSuccess ||
        cudaFuncSetAttribute(proj_kernel<bf16, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gm_smem<BN>()) != cudaSuccess)
        return false;
    for (int k = 0; k < 3; ++k) {
        const int cs = 2 << k;
        cudaLaunchConfig_t q = {};
        q.gridDim = dim3(cs);
        q.blockDim = dim3(GM_THREADS);
        q.dynamicSmemBytes = gm_smem<BN>();
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = (unsigned)cs;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        q.attrs = qa;
        q.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, proj_kernel<bf16, BN>, &q) != cudaSuccess) {
            cudaGetLastError();                        // a refused query: never split this far
            n = 0;
        }
        max_clusters[k] = n;
    }
    return true;
}

static const ProjDevice *proj_device()
{
    static ProjDevice dev_info[64];
    static bool ready[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ready[dev]) {
        if (!proj_setup<256>(dev_info[dev].max_clusters[0]) || !proj_setup<128>(dev_info[dev].max_clusters[1]))
            return nullptr;
        ready[dev] = true;
    }
    return &dev_info[dev];
}

template <int BN>
static cudaError_t launch_proj_bn(const void *x, const void *w, const ProjOut &out, int M, int N, int K,
                                  gdn_dtype out_dt, cudaStream_t s, int n_sm, const int (&max_clusters)[3])
{
    CUtensorMap mx, mw;
    if (!make_bf16_sw128_map(&mx, x, M, K, GM_BM) || !make_bf16_sw128_map(&mw, w, N, K, BN))
        return cudaErrorInvalidValue;
    const int n_work = ((M + GM_BM - 1) / GM_BM) * ((N + BN - 1) / BN);
    // Split K (2, 4 or 8 ways) while the tiles fill less than half of the SMs,
    // and only as far as every cluster of that size can be resident at once:
    // a cluster that waits for another to finish costs a whole tile's time.
    int splits = 1;
    while (splits < 8 && n_work * splits * 2 <= n_sm && (K / GM_BK) % (splits * 2) == 0 &&
           max_clusters[splits == 1 ? 0 : splits == 2 ? 1 : 2] >= n_work)
        splits *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(splits > 1 ? n_work * splits : (n_work < n_sm ? n_work : n_sm));
    cfg.blockDim = dim3(GM_THREADS);
    cfg.dynamicSmemBytes = gm_smem<BN>();
    cfg.stream = s;
    // programmatic stream serialization (the kernel waits for the kernel ahead
    // before its first global access), plus the cluster shape when splitting K
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 2 : 1;
    return out_dt == GDN_F32 ? cudaLaunchKernelEx(&cfg, proj_kernel<float, BN>, mx, mw, out, M, N, K, splits)
                             : cudaLaunchKernelEx(&cfg, proj_kernel<bf16, BN>, mx, mw, out, M, N, K, splits);
}

// y[M][N] = x[M][K] w[N][K]^T with the output columns routed by `out`.
static cudaError_t launch_proj(const void *x, const void *w, const ProjOut &out, int M, int N, int K,
                               gdn_dtype out_dt, cudaStream_t s)
{
    if (M <= 0) return cudaSuccess;
    const int n_sm = sm_count();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    const ProjDevice *pd = proj_device();
    if (!pd) return cudaErrorInvalidDevice;
    const int n_work256 = ((M + GM_BM - 1) / GM_BM) * ((N + 255) / 256);
    if (n_work256 * 2 <= n_sm)                         // 256-wide tiles would leave most SMs idle
        return launch_proj_bn<128>(x, w, out, M, N, K, out_dt, s, n_sm, pd->max_clusters[1]);
    return launch_proj_bn<256>(x, w, out, M, N, K, out_dt, s, n_sm, pd->max_clusters[0]);
}

cudaError_t launch_out_proj(const void *x, const void *w, void *y, int M, gdn_dtype out_dt, cudaStream_t s)
{
    ProjOut o = {};
    o.ptr[0] = y;
    o.c0[0] = 0;
    o.c0[1] = GDN_HIDDEN;
    o.ld[0] = GDN_HIDDEN;
    o.nseg = 1;
    return launch_proj(x, w, o, M, GDN_HIDDEN, DI, out_dt, s);
}

// The input projections: columns 0..8191 -> qkv, 8192..12287 -> z,
// 12288..12319 -> alpha, 12320..12351 -> beta.
cudaError_t launch_in_proj(const void *h, const void *w_in, void *qkv, void *z, void *alpha, void *beta, int M,
                           gdn_dtype act, cudaStream_t s)
{
    ProjOut o = {};
    o.ptr[0] = qkv; o.ptr[1] = z; o.ptr[2] = alpha; o.ptr[3] = beta;
    o.c0[0] = 0; o.c0[1] = CC; o.c0[2] = CC + DI; o.c0[3] = CC + DI + HV; o.c0[4] = CC + DI + 2 * HV;
    o.ld[0] = CC; o.ld[1] = DI; o.ld[2] = HV; o.ld[3] = HV;
    o.nseg = 4;
    return launch_proj(h, w_in, o, M, CC + DI + 2 * HV, GDN_HIDDEN, act, s);
}

// Reads and clears this file's device error word (synchronous on `s`).
// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *gemm_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_gemm_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
