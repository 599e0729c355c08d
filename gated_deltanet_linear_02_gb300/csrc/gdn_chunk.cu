// gdn_chunk.cu -- chunked (WY / UT-transform) prefill on tcgen05 tensor cores,
// for bf16 activations with fp32 state (chunk_size 64).
//
// The recurrence is the per-token delta rule of "qwen35moe -- Forward-Pass
// Design (Pantheon port)", section "Per-token recurrence". The pages say only
// that prefill may be evaluated as a token scan or reorganised into blocks
// ("Optimizing on-device inference for Apple silicon", the section on the three
// workload shapes). The block form used here is an exact re-association of
// that recurrence, written out by plain algebra. Within a chunk of n <= 64
// tokens entering with state S0, let G_r = sum_{s<=r} g_s and gamma_r = exp(G_r):
//   L    = strict_lower(exp(G_r - G_s) k_r.k_s),   T = (I + diag(b) L)^-1 diag(b)
//   U    = T V,  W = T diag(gamma) K,  Vnew = U - W S0   (= the per-token deltas)
//   Y    = scale (diag(gamma) Q S0 + (Mask o Q K^T) Vnew),  Mask_rs = exp(G_r-G_s), s<=r
//   Send = gamma_n S0 + K^T diag(exp(G_n - G_s)) Vnew
// Every exponent is <= 0 (r >= s); the inverse decay is never formed.
//
// Two kernels:
//  prep  (one CTA per (chunk, K-head); both V-heads of the GQA pair). This is
//        the S-independent part: conv + SiLU, L2 norms, gates, K K^T and Q K^T
//        (tf32 MMAs), the unit-lower triangular inverse for T (fp32, two
//        levels of 32x32 blocks), then U and W (tf32 MMAs). It writes per (chunk, V-head)
//        operand tiles to the workspace, already in the shared-memory layout
//        the carry kernel feeds to its MMAs.
//  carry (one CTA per (sequence, V-head, block of 32 value columns)). This is
//        the sequential chain over the chunks, for the CTA's columns of S (the
//        columns are independent). The state block lives in tensor memory
//        (fp32) and as a bf16 copy in shared memory. Per chunk: MMA (W S0, Q S0)
//        -> Vnew = U - W S0 -> MMA (P Vnew, K^T Vnew into the state) -> state
//        copy and decay. y goes to a buffer, and the gated RMSNorm . silu(z)
//        over each head's 128 columns runs as a separate kernel.
// Operand precision: the products whose rounding reaches the tolerance budget
// (U = T V, Q K^T, P Vnew, the state update) use tf32 operands, rounded to
// nearest when stored. W S0 and Q S0 take bf16 operands (kind::f16). All
// accumulation is fp32.
#include "gdn_async.cuh"
#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

#include <algorithm>

namespace gdn {

__device__ unsigned int g_chunk_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

constexpr int CH = 64;                    // chunk length

// Per (chunk, V-head) blob in the workspace. W | Q~ are contiguous (one bulk
// copy), and P | K~^T are contiguous (another bulk copy).
constexpr uint32_t BLOB_W = 0;         // W [t][i], bf16, K-major (Kd 128)        16 KiB
constexpr uint32_t BLOB_Q = 16384;     // Q~ = diag(gamma) Q [t][i], bf16, K-major  16 KiB
constexpr uint32_t BLOB_P = 32768;     // P = Mask o Q K^T [t][s], tf32, K-major    16 KiB
constexpr uint32_t BLOB_KT = 49152;    // K~^T [i][t], K~ = diag(exp(G_n-G_t)) K    32 KiB
constexpr uint32_t BLOB_U = 81920;     // U [t][j], fp32 row-major                  32 KiB
constexpr uint32_t BLOB_G = 114688;    // gamma_n of the chunk (fp32)
constexpr size_t BLOB_BYTES = 114944;

struct ChunkArgs {
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    float norm_eps, l2_eps;
    const bf16 *qkv, *z, *alpha, *beta;
    const int32_t *cu;
    int N, T_total, max_chunks;
    const bf16 *cs_in;
    const float *S_in;
    float *S_out;
    void *out;
    int32_t *chunk_off;       // [N+1]: first global chunk of each sequence
    int4 *chunk_info;         // [max_chunks]: {sequence, chunk in it, its first row, tokens}; -1 = unused
    unsigned char *blobs;     // [max_chunks][32] x BLOB_BYTES
    float *ybuf;              // [T_total][4096]: y before the gated norm (scale applied)
};

__device__ __forceinline__ int cu_clamp(const int32_t *cu, int i, int lo, int hi)
{
    return min(max(__ldg(cu + i), lo), hi);
}

// ------------------------------------------------------------------ schedule
// chunk_off[n] = sum over m < n of ceil(L_m / 64), clamped to max_chunks.
__global__ void __launch_bounds__(1024) chunk_schedule_kernel(const int32_t *__restrict__ cu, int N, int T_total,
                                                              int max_chunks, int32_t *__restrict__ chunk_off,
                                                              int4 *__restrict__ chunk_info)
{
    __shared__ int warp_part[32];
    grid_dep_launch();                                 // the prep kernel may be scheduled now
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (N + 1023) / 1024;
    const int lo = min(tid * per, N), hi = min(lo + per, N);
    int sum = 0;
    for (int n = lo; n < hi; ++n) {
        const int a = cu_clamp(cu, n, 0, T_total), b = cu_clamp(cu, n + 1, a, T_total);
        sum += (b - a + CH - 1) / CH;
    }
    // exclusive prefix sum of the per-thread chunk counts: inclusive scan within
    // each warp, then a scan of the 32 warp totals by warp 0
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) warp_part[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_part[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += v;
        }
        warp_part[lane] = w;                            // inclusive over warps
    }
    __syncthreads();
    const int all = warp_part[31];
    const int total = min(all, max_chunks);
    if (tid == 0) chunk_off[N] = total;
    int run = (warp ? warp_part[warp - 1] : 0) + incl - sum;
    for (int n = lo; n < hi; ++n) {
        chunk_off[n] = min(run, max_chunks);
        const int a = cu_clamp(cu, n, 0, T_total), b = cu_clamp(cu, n + 1, a, T_total);
        const int nch = (b - a + CH - 1) / CH;
        for (int c = 0; c < nch && run + c < max_chunks; ++c)   // {sequence, chunk in it, start row, tokens}
            chunk_info[run + c] = make_int4(n, c, a, min(CH, b - a - CH * c));
        run += nch;
    }
    for (int g = total + tid; g < max_chunks; g += blockDim.x) chunk_info[g] = make_int4(-1, 0, 0, 0);
}

// -------------------------------------------------------------------- prep
constexpr int P1_THREADS = 512;
constexpr int NW1 = P1_THREADS / 32;   // 16 warps: 4 per lane quarter of the tensor memory
constexpr uint32_t S1_QS = 0;          // q^ tf32 [t][i] Kd128; later (Gamma K)^T of head 0 [i][s] Kd64
constexpr uint32_t S1_KS = 32768;      // k^ tf32 [t][i] Kd128
constexpr uint32_t S1_VT0 = 65536;     // v^T tf32 [j][s] Kd64, head 0
constexpr uint32_t S1_VT1 = 98304;     //                    head 1
constexpr uint32_t S1_LB0 = 131072;    // beta_r * L[r][s], fp32 [64][64], 16-byte groups swizzled (lb_at), head 0
constexpr uint32_t S1_LB1 = 147456;    //                                                                    head 1
constexpr uint32_t S1_TS0 = 163840;    // T tf32 [t][s] Kd64, head 0
constexpr uint32_t S1_TS1 = 180224;    //                     head 1
constexpr uint32_t S1_GK1 = 196608;    // (Gamma K)^T tf32 [i][s] Kd64, head 1
constexpr uint32_t S1_SMALL = 229376;
// Float index of L[t][s] in a [64][64] tile whose 16-byte groups are XOR-swizzled
// by the row: rows written one per lane spread over the banks, and a row still
// reads as float4 groups of 4 consecutive s.
__device__ __forceinline__ int lb_at(int t, int s) { return t * CH + (((s >> 2) ^ (t & 15)) << 2) + (s & 3); }
// Raw bf16 inputs of the chunk, staged before the conv by four 2-D TMA copies,
// one per 128-channel block (q, k, v of head 0, v of head 1): 67 rows
// (positions -3..63) of 136 channels. The 8 extra channels pad each row to
// 272 bytes, which spreads consecutive rows over the banks. The staging
// overlays the L / T / (Gamma K)^T area, which is written only after the conv.
constexpr uint32_t S1_RAW = 131072;
constexpr int RAW_ROWS = CH + KC - 1;
constexpr int RAW_COLS = 136;
constexpr int RAW_ROWB = RAW_COLS * 2;                              // 272-byte rows
constexpr uint32_t RAW_BOX_BYTES = RAW_ROWS * RAW_ROWB;             // 18,224
constexpr uint32_t RAW_SEG = (RAW_BOX_BYTES + 127) / 128 * 128;    // 128-byte aligned block stride
// conv taps of the 512 channels (4 blocks x 128 channels x 16 B), staged with the rows
constexpr uint32_t S1_CW = S1_RAW + 4 * RAW_SEG;
static_assert(S1_CW % 128 == 0 && S1_CW + 4 * 2048 <= S1_SMALL, "staging overlap");
struct P1Small {
    float G[2][CH];     // chunk-local cumulative log-decay per V-head
    float B[2][CH];     // beta
    float gam[2][CH];   // exp(G)
    float ktf[2][CH];   // exp(G_n - G_t), the row factor of K~
    uint64_t bar;       // tensor-core completions
    uint64_t bar_ld;    // the staging copies
    uint32_t tmem;
    int abort;
};
constexpr size_t P1_SMEM = S1_SMALL + sizeof(P1Small) + 128;
// tensor-memory columns of the prep kernel
constexpr uint32_t T1_KK = 0, T1_QK = 64, T1_U = 128, T1_W = 256, T1_COLS = 512;

template <int ES> __device__ __forceinline__ uint32_t km(int r, int k, int Kd) { return tc::kmajor_offset<ES>(r, k, Kd); }

__global__ void __launch_bounds__(P1_THREADS, 1) chunk_prep_kernel(const __grid_constant__ CUtensorMap qkv_map,
                                                                  const ChunkArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = smem_aligned128(smem_raw);
    P1Small &ss = *reinterpret_cast<P1Small *>(sm + S1_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = smem_u32(sm);
    float *Qs = reinterpret_cast<float *>(sm + S1_QS);
    float *Ks = reinterpret_cast<float *>(sm + S1_KS);

    grid_dep_wait();                                   // chunk_info comes from the schedule kernel
    grid_dep_launch();
    // Persistent: CTA b takes items b, b + grid, ... (item = chunk * 16 + K-head),
    // skipping unused chunk slots. The next item's raw rows are staged while the
    // current item writes its outputs.
    const int n_items = a.max_chunks * HK;
    auto next_valid = [&](int it) {
        while (it < n_items && __ldg(a.chunk_info + it / HK).x < 0) it += (int)gridDim.x;
        return it;
    };
    // ---- B1. stage an item's raw q|k|v inputs of chunk positions -3..63 (the
    //      512 channels of its K-head pair) and their conv taps: one thread
    //      issues four 2-D tensor copies and four 2 KiB bulk copies on one
    //      mbarrier. Rows past the chunk's last token hold whatever follows (the
    //      next sequence, or zeros past the end); only outputs of valid tokens
    //      are kept, and those never read such rows.
    auto stage = [&](int it) {                         // caller: thread 0
        const int4 c = __ldg(a.chunk_info + it / HK);
        const int k2 = it % HK;
        const int ch[4] = {Q_OFF + k2 * DK, K_OFF + k2 * DK, V_OFF + k2 * DV, V_OFF + (k2 + HK) * DV};
        const uint32_t bl = smem_u32(&ss.bar_ld);
        mbar_arrive_expect_tx(bl, 4 * RAW_BOX_BYTES + 4 * 2048);
#pragma unroll
        for (int sg = 0; sg < 4; ++sg) {
            tma_load_2d(sbase + S1_RAW + sg * RAW_SEG, &qkv_map, ch[sg], c.z + CH * c.y - (KC - 1), bl);
            bulk_g2s(sbase + S1_CW + sg * 2048, a.conv_w + (size_t)ch[sg] * KC, 2048, bl);
        }
    };
    if (warp == 0) {
        tc::tmem_alloc(smem_u32(&ss.tmem), T1_COLS);
        tc::tmem_relinquish();
    }
    int item = next_valid((int)blockIdx.x);
    int done = 0;                                      // items finished by this CTA
    bool staged = false;                               // thread 0: a staging copy is in flight
    float al_next = 0.0f, be_next = 0.0f;              // threads < 128: the next item's gate logits
    if (tid == 0) {
        mbar_init(smem_u32(&ss.bar), 1);
        mbar_init(smem_u32(&ss.bar_ld), 1);
        ss.abort = 0;
        fence_mbar_init();
        if (item < n_items) {
            stage(item);
            staged = true;
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = ss.tmem;

    for (; item < n_items; ++done) {
    const int g = item / HK, kh = item % HK;
    const int4 ci = __ldg(a.chunk_info + g);
    const int n = ci.x;                                // sequence
    const int lc = ci.y;                               // chunk index inside the sequence
    const int seq0 = ci.z;                             // the sequence's first row
    const int t0 = seq0 + CH * lc;
    const int nv = ci.w;                               // valid tokens in this chunk (1..64)
    const int nit = next_valid(item + (int)gridDim.x);
    // first channel of segment sg: q, k of K-head kh, v of V-heads kh and kh + 16
    auto chan0 = [kh](int sg) {
        return sg == 0 ? Q_OFF + kh * DK : sg == 1 ? K_OFF + kh * DK : V_OFF + (kh + (sg - 2) * HK) * DV;
    };
    // gates of both V-heads; padded tokens get g = 0, beta = 0. After the first
    // item the logits were loaded ahead, during the previous item's stores.
    if (tid < 2 * CH) {
        const int h = tid >> 6, p = tid & 63, vh = kh + HK * h;
        float gg = 0.0f, bb = 0.0f;
        if (p < nv) {
            const float al = done == 0 ? to_f(a.alpha[(size_t)(t0 + p) * HV + vh]) : al_next;
            const float be = done == 0 ? to_f(a.beta[(size_t)(t0 + p) * HV + vh]) : be_next;
            gg = -expf(a.A_log[vh]) * softplus_f(al + a.dt_bias[vh]);
            bb = 1.0f / (1.0f + expf(-be));
        }
        ss.G[h][p] = gg;
        ss.B[h][p] = bb;
    }
    __syncthreads();
    if (!mbar_wait_bounded(smem_u32(&ss.bar_ld), (uint32_t)(done & 1))) ss.abort = 1;
    if (tid == 0) staged = false;
    if (lc == 0 && tid < 3 * 4 * 16) {
        // the first chunk of a sequence: positions -3..-1 are its conv_state
        // (zeros without one), not the rows before the sequence
        const int r = tid >> 6, sg = (tid >> 4) & 3, pc = tid & 15;
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (a.cs_in) x = __ldg(reinterpret_cast<const uint4 *>(a.cs_in + ((size_t)n * (KC - 1) + r) * CC + chan0(sg)) + pc);
        *reinterpret_cast<uint4 *>(sm + S1_RAW + sg * RAW_SEG + r * RAW_ROWB + pc * 16) = x;
    }
    __syncthreads();

    // ---- B2. conv + SiLU from the staged rows. q and k go raw into their tf32
    //      tiles (normalised below); v^T follows once the first products are
    //      issued. Lanes map onto the 8 rows of a core matrix, so each 16-byte
    //      store of a warp phase fills one contiguous 128-byte core matrix.
    const unsigned char *raw = sm + S1_RAW;
    // Each pass loads the inputs of four iterations before it stores anything,
    // so the loads of later iterations need not wait behind earlier stores.
    static_assert(NW1 == 16, "a pass's four iterations it0 + 16 k share the tile (it >> 6) and k-group (it & 7)");
#pragma unroll 1
    for (int it0 = warp; it0 < 128; it0 += 4 * NW1) {                // q, k: (tile, row octet, k-group)
        const int tile = it0 >> 6, kgh = it0 & 7;
        const int d = 4 * (kgh * 4 + (lane >> 3));                    // 4 consecutive channels d..d+3
        float4 w4[4];                                                 // their taps, the same for the whole pass
#pragma unroll
        for (int e = 0; e < 4; ++e) w4[e] = reinterpret_cast<const float4 *>(sm + S1_CW + tile * 2048)[d + e];
        uint2 pr[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int p = (((it0 + k * NW1) >> 3) & 7) * 8 + (lane & 7);
#pragma unroll
            for (int m = 0; m < 4; ++m)                               // positions p-3+m = rows p+m
                pr[k][m] = *reinterpret_cast<const uint2 *>(raw + tile * RAW_SEG + (p + m) * RAW_ROWB + d * 2);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int p = (((it0 + k * NW1) >> 3) & 7) * 8 + (lane & 7);
            float x[4][4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const bf16 *hv = reinterpret_cast<const bf16 *>(&pr[k][m]);
#pragma unroll
                for (int e = 0; e < 4; ++e) x[m][e] = to_f(hv[e]);
            }
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 w = w4[e];
                const float u = w.x * x[0][e] + w.y * x[1][e] + w.z * x[2][e] + w.w * x[3][e];
                o[e] = p < nv ? silu_fast(u) : 0.0f;
            }
            *reinterpret_cast<float4 *>(sm + (tile ? S1_KS : S1_QS) + km<4>(p, d, DK)) = make_float4(o[0], o[1], o[2], o[3]);
        }
    }
    __syncthreads();

    // ---- C. L2 norm of the 64 q rows and 64 k rows. A warp takes 8 rows at a
    //      time; lane (row r%8, k-group) reads 8 float4s, and the 4 lanes of a
    //      row combine their sums with two shuffles.
    for (int gi = warp; gi < 16; gi += P1_THREADS / 32) {
        float *tile = gi < 8 ? Qs : Ks;
        const int t = (gi & 7) * 8 + (lane & 7), kgl = lane >> 3;
        float4 v[8];
        float s2 = 0.0f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            v[m] = *reinterpret_cast<const float4 *>(reinterpret_cast<unsigned char *>(tile) + km<4>(t, 4 * (4 * m + kgl), DK));
            s2 += v[m].x * v[m].x + v[m].y * v[m].y + v[m].z * v[m].z + v[m].w * v[m].w;
        }
        s2 += __shfl_xor_sync(0xffffffffu, s2, 8);
        s2 += __shfl_xor_sync(0xffffffffu, s2, 16);
        const float inv = rsqrtf(s2 + a.l2_eps);
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            float4 x = v[m];
            x.x *= inv; x.y *= inv; x.z *= inv; x.w *= inv;
            *reinterpret_cast<float4 *>(reinterpret_cast<unsigned char *>(tile) + km<4>(t, 4 * (4 * m + kgl), DK)) = tc::tf32_rn(x);
        }
    }
    if (warp < 2) {                                   // warp h: inclusive scan of head h's log-decays
        const float g0 = ss.G[warp][2 * lane], g1 = ss.G[warp][2 * lane + 1];
        float run = g0 + g1;                           // lane l holds tokens 2l, 2l+1
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float up = __shfl_up_sync(0xffffffffu, run, o);
            if (lane >= o) run += up;
        }
        ss.G[warp][2 * lane] = run - g1;
        ss.G[warp][2 * lane + 1] = run;
    }
    __syncthreads();
    if (tid < 2 * CH) {
        const int h = tid >> 6, p = tid & 63;
        ss.gam[h][p] = expf(ss.G[h][p]);
        ss.ktf[h][p] = __expf(ss.G[h][CH - 1] - ss.G[h][p]);   // K~ row factor, exponent <= 0
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- D. K K^T and Q K^T (tf32, M=64, N=64, K=128)
    if (tid == 0) {
        tc::fence_after_sync();
        const uint32_t id = tc::instr_desc(tc::FMT_TF32, CH, CH);
        tc::mma_tile<true>(tm + T1_KK, sbase + S1_KS, DK, sbase + S1_KS, DK, DK, id, false);
        tc::mma_tile<true>(tm + T1_QK, sbase + S1_QS, DK, sbase + S1_KS, DK, DK, id, false);
        tc::mma_commit(smem_u32(&ss.bar));
    }
    // The value stream's conv runs while the tensor core computes K K^T and Q K^T:
    // v^T of both heads goes straight into its tiles.
    // Iteration it = (V-head hv, half of the channels, block of 8 tokens): lane
    // (group g = lane >> 3, pair c = lane & 7) convolves channels d, d + 1
    // (d = 64 half + 16 g + 2 c) over tokens p0 .. p0 + 7, from 4-byte loads of
    // 11 staged rows; a warp's load covers 128 contiguous bytes of one row. For
    // the stores, lanes c >= 4 write their odd channel first, so that each
    // quarter-warp's 16-byte stores fill rows 0..7 of two core matrices.
    static_assert(CH == 64 && DV == 128, "v^T tiling of the conv");
#pragma unroll 1
    for (int it = warp; it < 32; it += NW1) {
        const int hv = it >> 4, half = (it >> 3) & 1, p0 = 8 * (it & 7);
        const int c = lane & 7, d = 64 * half + 16 * (lane >> 3) + 2 * c;
        const float4 *cw = reinterpret_cast<const float4 *>(sm + S1_CW + (2 + hv) * 2048);
        const float4 wa = cw[d], wb = cw[d + 1];
        uint32_t xr[11];                                              // positions p0-3 .. p0+7, channels d, d+1
#pragma unroll
        for (int m = 0; m < 11; ++m)
            xr[m] = *reinterpret_cast<const uint32_t *>(raw + (2 + hv) * RAW_SEG + (p0 + m) * RAW_ROWB + d * 2);
        float oa[8], ob[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            float xa[4], xb[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                xa[m] = __uint_as_float(xr[e + m] << 16);             // channel d: the low half
                xb[m] = __uint_as_float(xr[e + m] & 0xFFFF0000u);     // channel d + 1
            }
            const float ua = wa.x * xa[0] + wa.y * xa[1] + wa.z * xa[2] + wa.w * xa[3];
            const float ub = wb.x * xb[0] + wb.y * xb[1] + wb.z * xb[2] + wb.w * xb[3];
            const bool ok = (p0 + e) < nv;
            oa[e] = ok ? tc::tf32_rn(silu_fast(ua)) : 0.0f;
            ob[e] = ok ? tc::tf32_rn(silu_fast(ub)) : 0.0f;
        }
        unsigned char *vt = sm + (hv ? S1_VT1 : S1_VT0);
        const bool odd_first = c >= 4;
#pragma unroll
        for (int sidx = 0; sidx < 2; ++sidx) {
            const bool odd = odd_first != (sidx == 1);
            const float *o = odd ? ob : oa;
#pragma unroll
            for (int tq = 0; tq < 2; ++tq)
                *reinterpret_cast<float4 *>(vt + km<4>(d + (odd ? 1 : 0), p0 + 4 * tq, CH)) =
                    make_float4(o[4 * tq], o[4 * tq + 1], o[4 * tq + 2], o[4 * tq + 3]);
        }
    }
    __syncthreads();                                   // every read of the staged rows is done
    if (!mbar_wait_bounded(smem_u32(&ss.bar), 0)) ss.abort = 1;
    tc::fence_after_sync();

    // the blobs of V-heads kh and kh + 16 (a function of h, not an array, so
    // that a runtime h does not put the pointers in local memory)
    unsigned char *const blob0 = a.blobs + ((size_t)g * HV + kh) * BLOB_BYTES;
    auto blob = [&](int h) { return blob0 + (size_t)h * HK * BLOB_BYTES; };

    // ---- E. P = Mask o QK^T and beta * L from the M=64 accumulators (row t in
    //      TMEM lane 32*(t/16) + t%16), then Q~ and gamma_n. Warp w reads
    //      columns [16 (w / 4), +16) of its lane quarter w % 4.
    {
        const int q = warp & 3, hf = warp >> 2;
        float kk[16], qk[16];
        tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T1_KK + 16 * hf), kk);
        tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T1_QK + 16 * hf), qk);
        tc::wait_ld();
        // Rows live in lanes 0..15. Lanes 16..31 take over columns 8..15 of their row.
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float a1 = __shfl_sync(0xffffffffu, kk[8 + c], lane & 15);
            const float a2 = __shfl_sync(0xffffffffu, qk[8 + c], lane & 15);
            if (lane >= 16) { kk[c] = a1; qk[c] = a2; }
        }
        if (!ss.abort) {
            const int t = 16 * q + (lane & 15);
            const int cbase = 16 * hf + 8 * (lane >> 4);      // this lane's 8 columns
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float Gt = ss.G[h][t], bt = ss.B[h][t];
                float *Lb = reinterpret_cast<float *>(sm + (h ? S1_LB1 : S1_LB0));
#pragma unroll
                for (int c4 = 0; c4 < 2; ++c4) {
                    float pv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int cc = c4 * 4 + e, s = cbase + cc;
                        const float dec = s <= t ? __expf(Gt - ss.G[h][s]) : 0.0f;
                        Lb[lb_at(t, s)] = s < t ? bt * dec * kk[cc] : 0.0f;
                        pv[e] = dec * qk[cc];
                    }
                    *reinterpret_cast<float4 *>(blob(h) + BLOB_P + km<4>(t, cbase + c4 * 4, CH)) =
                        tc::tf32_rn(make_float4(pv[0], pv[1], pv[2], pv[3]));
                }
            }
        }
    }
    // Q~ = diag(gamma) q^ -> bf16 K-major (Kd 128), 8 elements per store
    for (int u = tid; u < 2 * CH * 16; u += P1_THREADS) {   // lanes walk the 8 rows of a core matrix
        const int h = u >> 10, i8 = (u >> 3) & 15, t = ((u >> 7) & 7) * 8 + (u & 7);
        const float gm = ss.gam[h][t];
        const float4 x0 = *reinterpret_cast<const float4 *>(sm + S1_QS + km<4>(t, i8 * 8, DK));
        const float4 x1 = *reinterpret_cast<const float4 *>(sm + S1_QS + km<4>(t, i8 * 8 + 4, DK));
        auto pk = [gm](float lo, float hi) {            // two bf16 in one word, lo first
            const __nv_bfloat162 v = __floats2bfloat162_rn(lo * gm, hi * gm);
            return *reinterpret_cast<const uint32_t *>(&v);
        };
        *reinterpret_cast<uint4 *>(blob(h) + BLOB_Q + km<2>(t, i8 * 8, DK)) =
            make_uint4(pk(x0.x, x0.y), pk(x0.z, x0.w), pk(x1.x, x1.y), pk(x1.z, x1.w));
    }
    if (tid < 2) *reinterpret_cast<float *>(blob(tid) + BLOB_G) = ss.gam[tid][CH - 1];
    tc::fence_before_sync();
    __syncthreads();

    // ---- F. T = (I + A)^-1 diag(b), A = diag(b) L (Lb), in two 32x32 block
    //      levels. With X_b = (I + A_bb)^-1 for the diagonal blocks b = 0, 1:
    //        T_00 = X_0 diag(b_0),  T_11 = X_1 diag(b_1),  T_01 = 0,
    //        T_10 = -X_1 (A_10 T_00)                     (block row 1 of (I + A) T).
    //      Level 1 (threads 0..127: one column of one block of one head) runs
    //      the forward substitutions while warps 4..7 build (Gamma K)^T of head 0;
    //      level 2 spreads the two 32x32x32 products over all threads. The fp32
    //      intermediates T_00, X_1 and M = A_10 T_00 sit in the head-1 (Gamma K)^T
    //      area, which is built last.
    {
        constexpr int XS = 36;                               // X_1 row stride (floats): rows 2 apart hit other banks
        auto t00_of = [&](int h) { return reinterpret_cast<float *>(sm + S1_GK1 + h * 12288); };
        auto x1_of = [&](int h) { return reinterpret_cast<float *>(sm + S1_GK1 + h * 12288 + 4096); };
        auto m_of = [&](int h) { return reinterpret_cast<float *>(sm + S1_GK1 + 24576 + h * 4096); };
        static_assert(24576 + 2 * 4096 <= 32768 && 4096 + 32 * XS * 4 <= 12288, "solve scratch");
        if (tid < 2 * CH) {
            const int h = tid >> 6, b = (tid >> 5) & 1, c = tid & 31;
            const float *Lb = reinterpret_cast<const float *>(sm + (h ? S1_LB1 : S1_LB0));
            float x[32];
#pragma unroll
            for (int r = 0; r < 32; ++r) x[r] = 0.0f;     // x[s >= r] stay 0 while row r is summed
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                float acc[4] = {(r == c) ? 1.0f : 0.0f, 0.0f, 0.0f, 0.0f};   // 4 chains for ILP
#pragma unroll
                for (int s4 = 0; s4 < (r + 3) / 4; ++s4) {      // A[r][s] = 0 for s >= r
                    const float4 l4 = *reinterpret_cast<const float4 *>(Lb + lb_at(32 * b + r, 32 * b + 4 * s4));
                    acc[0] = fmaf(-l4.x, x[4 * s4], acc[0]);
                    acc[1] = fmaf(-l4.y, x[4 * s4 + 1], acc[1]);
                    acc[2] = fmaf(-l4.z, x[4 * s4 + 2], acc[2]);
                    acc[3] = fmaf(-l4.w, x[4 * s4 + 3], acc[3]);
                }
                x[r] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            }
            const float bc = ss.B[h][32 * b + c];
            unsigned char *Ts = sm + (h ? S1_TS1 : S1_TS0);
            float *plain = b ? x1_of(h) : t00_of(h);
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                *reinterpret_cast<float *>(Ts + km<4>(32 * b + r, 32 * b + c, CH)) = tc::tf32_rn(x[r] * bc);
                plain[r * (b ? XS : 32) + c] = b ? x[r] : x[r] * bc;
            }
        } else {
            for (int it = warp - 4; it < 16 * 4; it += NW1 - 4) {      // (Gamma K)^T of head 0 into QS
                const int i = ((it >> 2) & 15) * 8 + (lane & 7), s4 = (it & 3) * 4 + (lane >> 3);
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int sx = s4 * 4 + e;
                    v[e] = ss.gam[0][sx] * *reinterpret_cast<const float *>(sm + S1_KS + km<4>(sx, i, DK));
                }
                *reinterpret_cast<float4 *>(sm + S1_QS + km<4>(i, s4 * 4, CH)) =
                    tc::tf32_rn(make_float4(v[0], v[1], v[2], v[3]));
            }
        }
        __syncthreads();
        // level 2: thread (head, row, column quad) owns row r and columns c0..c0+3
        const int h = tid >> 8, r = ((tid >> 5) & 7) * 4 + (lane >> 3), c0 = 4 * (lane & 7);
        {                                                     // M = A_10 T_00
            const float *Lb = reinterpret_cast<const float *>(sm + (h ? S1_LB1 : S1_LB0));
            const float *T00 = t00_of(h);
            float acc[4] = {};
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(Lb + lb_at(32 + r, k));
                const float ar[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(T00 + (k + e) * 32 + c0);
                    acc[0] = fmaf(ar[e], t4.x, acc[0]);
                    acc[1] = fmaf(ar[e], t4.y, acc[1]);
                    acc[2] = fmaf(ar[e], t4.z, acc[2]);
                    acc[3] = fmaf(ar[e], t4.w, acc[3]);
                }
            }
            *reinterpret_cast<float4 *>(m_of(h) + r * 32 + c0) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        }
        __syncthreads();
        {                                                     // T_10 = -X_1 M; T_01 = 0
            const float *X1 = x1_of(h);
            const float *M = m_of(h);
            float acc[4] = {};
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(X1 + r * XS + k);
                const float ar[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 m4 = *reinterpret_cast<const float4 *>(M + (k + e) * 32 + c0);
                    acc[0] = fmaf(ar[e], m4.x, acc[0]);
                    acc[1] = fmaf(ar[e], m4.y, acc[1]);
                    acc[2] = fmaf(ar[e], m4.z, acc[2]);
                    acc[3] = fmaf(ar[e], m4.w, acc[3]);
                }
            }
            unsigned char *Ts = sm + (h ? S1_TS1 : S1_TS0);
            *reinterpret_cast<float4 *>(Ts + km<4>(32 + r, c0, CH)) =
                tc::tf32_rn(make_float4(-acc[0], -acc[1], -acc[2], -acc[3]));
            *reinterpret_cast<float4 *>(Ts + km<4>(r, 32 + c0, CH)) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
        for (int it = warp; it < 16 * 4; it += P1_THREADS / 32) {      // (Gamma K)^T of head 1
            const int i = ((it >> 2) & 15) * 8 + (lane & 7), s4 = (it & 3) * 4 + (lane >> 3);
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int sx = s4 * 4 + e;
                v[e] = ss.gam[1][sx] * *reinterpret_cast<const float *>(sm + S1_KS + km<4>(sx, i, DK));
            }
            *reinterpret_cast<float4 *>(sm + S1_GK1 + km<4>(i, s4 * 4, CH)) =
                tc::tf32_rn(make_float4(v[0], v[1], v[2], v[3]));
        }
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    // ---- G. U^T = V^T T^T and W^T = (Gamma K)^T T^T per head (tf32, M=128, N=64, K=64)
    if (tid == 0 && !ss.abort) {
        tc::fence_after_sync();
        const uint32_t id = tc::instr_desc(tc::FMT_TF32, 128, CH);
        for (int h = 0; h < 2; ++h) {
            const uint32_t ts = sbase + (h ? S1_TS1 : S1_TS0);
            tc::mma_tile<true>(tm + T1_U + 64 * h, sbase + (h ? S1_VT1 : S1_VT0), CH, ts, CH, CH, id, false);
            tc::mma_tile<true>(tm + T1_W + 64 * h, sbase + (h ? S1_GK1 : S1_QS), CH, ts, CH, CH, id, false);
        }
        tc::mma_commit(smem_u32(&ss.bar));
    }
    // While the tensor core computes U and W: K~^T to the blob (k^ stays intact
    // in its tile until the kernel ends).
    // K~^T [i][t] = exp(G_n - G_t) k^[t][i] -> tf32 K-major (Kd 64), 4 tokens per
    // store; lanes cover 4 whole core matrices, so a warp writes 512 contiguous bytes
    for (int it = warp; it < 2 * 16 * 4; it += P1_THREADS / 32) {
        const int h = it >> 6, i = ((it >> 2) & 15) * 8 + (lane & 7), t4 = (it & 3) * 4 + (lane >> 3);
        float v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int t = t4 * 4 + e;
            v[e] = ss.ktf[h][t] * *reinterpret_cast<const float *>(sm + S1_KS + km<4>(t, i, DK));
        }
        *reinterpret_cast<float4 *>(blob(h) + BLOB_KT + km<4>(i, t4 * 4, CH)) =
            tc::tf32_rn(make_float4(v[0], v[1], v[2], v[3]));
    }
    if (!ss.abort && !mbar_wait_bounded(smem_u32(&ss.bar), 1)) ss.abort = 1;
    tc::fence_after_sync();
    // U and W have been read out of shared memory: the staging area (which
    // overlaps L, T and (Gamma K)^T) takes the next item's rows during H
    if (tid == 0 && nit < n_items && !ss.abort) {
        stage(nit);
        staged = true;
    }
    if (tid < 2 * CH && nit < n_items) {              // and the next item's gate logits
        const int4 c = __ldg(a.chunk_info + nit / HK);
        const int h = tid >> 6, p = tid & 63, vh = nit % HK + HK * h;
        if (p < c.w) {
            const size_t row = (size_t)(c.z + CH * c.y + p) * HV + vh;
            al_next = to_f(a.alpha[row]);
            be_next = to_f(a.beta[row]);
        }
    }

    // ---- H. U -> blob as [t][j] fp32; W -> blob as bf16 K-major [t][i]. Warp w
    //      reads token columns [16 (w / 4), +16) of its lane quarter w % 4.
    //      Its W values fill two runs of 512 bytes of the K-major layout (rows
    //      t >> 3 = 2 hf, 2 hf + 1; columns [32 q, 32 q + 32)), so the warp stages
    //      them in shared memory (the v^T tile, which the U products have read)
    //      and copies its own runs out in 16-byte stores. In the staging copy the
    //      16-byte units of a run are XOR-swizzled (row t & 7 ^ 2 g for column
    //      group g), which puts the lanes' 2-byte stores for one token in four
    //      different bank groups.
    {
        const int q = warp & 3, hf = warp >> 2;
        const int j = 32 * q + lane;
        unsigned char *wst = sm + S1_VT0;                // 16 KiB per head
        auto wst_unit = [](int r8, int g) { return g * 8 + (r8 ^ (2 * g)); };   // staged unit of (t & 7, g)
        for (int h = 0; h < 2; ++h) {
            float u[16], wv[16];
            tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T1_U + 64 * h + 16 * hf), u);
            tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T1_W + 64 * h + 16 * hf), wv);
            tc::wait_ld();
            if (!ss.abort) {
                float *U = reinterpret_cast<float *>(blob(h) + BLOB_U);
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int t = 16 * hf + e;
                    U[t * DV + j] = u[e];
                    *reinterpret_cast<bf16 *>(wst + h * 16384 + (t >> 3) * 2048 + q * 512 +
                                              wst_unit(t & 7, (j >> 3) & 3) * 16 + (j & 7) * 2) = from_f<bf16>(wv[e]);
                }
            }
        }
        __syncwarp();
        if (!ss.abort) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int r = 0; r < 2; ++r) {            // run r (row block 2 hf + r), unit lane of 32
                    const uint32_t run = (uint32_t)((2 * hf + r) * 2048 + q * 512);
                    const int g = lane >> 3, r8 = lane & 7;
                    *reinterpret_cast<uint4 *>(blob(h) + BLOB_W + run + lane * 16) =
                        *reinterpret_cast<const uint4 *>(wst + h * 16384 + run + wst_unit(r8, g) * 16);
                }
        }
    }
    tc::fence_before_sync();
    __syncthreads();                                   // the next item rewrites gates, tiles and TMEM
    if (ss.abort) break;
    item = nit;
    }
    if (tid == 0 && staged)                            // after an abort: the copy in flight lands first
        mbar_wait_bounded(smem_u32(&ss.bar_ld), (uint32_t)(done & 1));
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, T1_COLS);
    if (tid == 0 && ss.abort) atomicExch(&g_chunk_error, (unsigned int)GDN_ERR_TIMEOUT);
}

// ------------------------------------------------------------------- carry
// One CTA per (sequence, V-head, block of 32 value columns j). Columns of S are
// independent (pred_j and y_j read only column j), so the value dimension splits
// exactly across the four CTAs of a V-head. Products per chunk, all written with
// the token or key index as the MMA M dimension and the CTA's 32 columns as N:
//   (1) Vn^(t,j) = W[t][i] S[i][j]          bf16, M=64 (t), N=32, K=128
//       Y(t,j)   = Q~[t][i] S[i][j]         bf16, M=64,     N=32, K=128
//   (2) S(i,j)  += K~^T[i][t] Vnew[t][j]    tf32, M=128 (i), N=32, K=64
//       Y(t,j)  += P[t][s] Vnew[s][j]       tf32, M=64,     N=32, K=64 (issued
//                                            with the next chunk's products)
// The state block S(i,j) lives in tensor memory (fp32, lane = i), plus a bf16
// copy in shared memory as the B operand of (1). Vnew = U - W S goes to shared
// memory as Vnew^T[j][t] (tf32), the B operand of (2). y (scale applied) goes to
// a [T][4096] fp32 buffer, and a separate kernel applies the gated RMSNorm
// across all 128 columns of each head.
//
// Issue. A tcgen05.mma instruction holds its issuing thread for a fixed time of
// some 60 cycles however small the product, while the tensor core accepts such
// instructions from several warps at once; small products then run at the rate
// shared memory feeds their operands. Only Vn^ = W S and the state update are on
// the chunk-to-chunk chain, so each is split along K between two issuer warps
// with separate accumulators (the epilogues add the halves), and each Y product
// is queued right behind a chain product, so that it runs while the epilogue of
// that product does: issuer k's K half of Y = Q~ S behind its half of Vn^, and
// its half of Y += P Vnew behind its half of the state update. Eight more warps
// run the tensor-memory epilogues. The issuers take no part in CTA-wide
// barriers (they would hold them up while an issue blocks): the epilogue warps
// hand over through two mbarriers, "Vnew written" and "next state block
// written", which each epilogue warp arrives on once its lanes have written
// and fenced.
constexpr int P2_EPI_WARPS = 8;
constexpr int P2_THREADS = 32 * (P2_EPI_WARPS + 2);
constexpr int JB = 32;                 // value columns per CTA
constexpr int NJB = DV / JB;           // CTAs per V-head
constexpr uint32_t S2_SS = 0;          // S block bf16, MN-major (N = 32 j, K = 128 i)    8 KiB
constexpr uint32_t S2_VN = 8192;       // Vnew^T block tf32 [32 j][64 t], 128-byte swizzle, chunk c at + 8 KiB (c % 2)
constexpr uint32_t S2_WQ0 = 24576;     // W | Q~ (bf16 [t][i] Kd128, 16 KiB each), stage 0
constexpr uint32_t S2_WQ1 = 57344;     //                                          stage 1
constexpr uint32_t S2_PK0 = 90112;     // P (tf32 [t][s] Kd64) | K~^T (tf32 [i][t] Kd64), stage 0
constexpr uint32_t S2_PK1 = 139264;    //                                                  stage 1
constexpr uint32_t S2_SMALL = 188416;
struct P2Small {
    uint64_t bar_wq[2], bar_pk[2];     // operand loads, per stage
    uint64_t bar_m1[2], bar_m2[2];     // chain products, per issuer
    uint64_t bar_y[2][2];              // all of a chunk's products, per Y buffer and issuer
    uint64_t bar_vn, bar_s;            // epilogue -> issuers: Vnew written; next state block written
    uint64_t bar_yfree;                // epilogue -> issuers: a Y buffer has been drained
    uint32_t tmem;
    int abort;
};
constexpr size_t P2_SMEM = S2_SMALL + sizeof(P2Small) + 128;
// tensor-memory columns (M=64 accumulators use lanes 0-15 of each lane quarter):
// issuer k's half of Vn^ at T2_VN + 32k; the state block S and issuer 1's half
// of its update dS; issuer k's half of Y at T2_Y + 64 (c % 2) + 32k, two
// buffers so that chunk c's y drains while chunk c + 1's products run
constexpr uint32_t T2_VN = 0, T2_S = 64, T2_DS = 96, T2_Y = 128, T2_COLS = 256;

// Caller: one thread. Loads chunk c's W | Q~ or P | K~^T into stage c % 2.
template <bool WQ>
__device__ __forceinline__ void carry_issue(const unsigned char *blob, uint32_t sb, P2Small &ss, int c)
{
    const int st = c & 1;
    if (WQ) {
        mbar_arrive_expect_tx(smem_u32(&ss.bar_wq[st]), 32768);
        bulk_g2s(sb + (st ? S2_WQ1 : S2_WQ0), blob + BLOB_W, 32768, smem_u32(&ss.bar_wq[st]));
    } else {
        mbar_arrive_expect_tx(smem_u32(&ss.bar_pk[st]), 49152);
        bulk_g2s(sb + (st ? S2_PK1 : S2_PK0), blob + BLOB_P, 49152, smem_u32(&ss.bar_pk[st]));
    }
}

// Byte offset of Vnew^T element (j, t) in its tile: K-major with the 128-byte
// swizzle, two atoms of 32 tokens (128-byte rows) x 32 columns j, 4 KiB apart.
// The 16-byte chunk of row j is permuted by XOR with j % 8, so the 16 tokens a
// warp stores for one column land in 16 different banks.
__device__ __forceinline__ uint32_t vn_offset(int j, int t)
{
    return (uint32_t)((t >> 5) * 4096 + j * 128 + ((((t & 31) >> 2) ^ (j & 7)) << 4) + (t & 3) * 4);
}

// D (+)= A B^T over 4 tf32 K steps of 8: A a K-major no-swizzle tile (two core
// matrices, 256 bytes, per step), B the swizzled Vnew^T atom (32 bytes per step).
__device__ __forceinline__ void mma_vn(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       bool accumulate)
{
#pragma unroll
    for (int s = 0; s < 4; ++s)
        tc::mma_tf32(d_tmem, a_desc + 16u * s, b_desc + 2u * s, idesc, (accumulate || s > 0) ? 1u : 0u);
}

// Thread (key row i, column half hf) stores its 16 state values S[i][j], j in
// [16hf, 16hf+16) of the CTA's block, as bf16 into the MN-major state tile:
// two 16-byte stores.
__device__ __forceinline__ void store_s_bf16(unsigned char *sm, int i, int hf, const float (&v)[16])
{
#pragma unroll
    for (int g8 = 0; g8 < 2; ++g8) {
        __align__(16) bf16 o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = from_f<bf16>(v[8 * g8 + e]);
        *reinterpret_cast<uint4 *>(sm + S2_SS + tc::mnmajor_offset_bf16(16 * hf + 8 * g8, i, DK)) =
            *reinterpret_cast<const uint4 *>(o);
    }
}

__global__ void __launch_bounds__(P2_THREADS, 1) chunk_carry_kernel(const ChunkArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = smem_aligned128(smem_raw);
    P2Small &ss = *reinterpret_cast<P2Small *>(sm + S2_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x, vh = blockIdx.y, jb = blockIdx.z;
    const bool issuer = warp >= P2_EPI_WARPS;          // warps 8, 9: lane 0 issues MMAs
    const int ik = warp - P2_EPI_WARPS;                // issuer index (issuer warps only)
    const int q = warp & 3, hf = (warp >> 2) & 1;      // lane quarter; column half (16 of the 32)
    const int i = 32 * q + lane;                       // key row i (M=128 accumulator lane)
    const int t = 16 * q + lane;                       // token row t (M=64 accumulator, lanes < 16)
    const bool trow = lane < 16;
    const int j0 = JB * jb + 16 * hf;                  // first of this thread's 16 value columns
    const size_t sbase_g = ((size_t)n * HV + vh) * (DV * DK);
    grid_dep_wait();                                   // the blobs come from the prep kernel
    grid_dep_launch();
    const int g0 = __ldg(a.chunk_off + n);
    const int nc = max(0, __ldg(a.chunk_off + n + 1) - g0);
    const int seq0 = cu_clamp(a.cu, n, 0, a.T_total);
    const int seqL = cu_clamp(a.cu, n + 1, seq0, a.T_total) - seq0;

    if (nc == 0) {                                     // empty sequence: this block of the state passes through
        if (a.S_out)
            for (int e = tid; e < JB * DK / 4; e += P2_THREADS) {
                const size_t off = sbase_g / 4 + (size_t)JB * jb * (DK / 4) + e;
                const float4 v = a.S_in ? reinterpret_cast<const float4 *>(a.S_in)[off] : make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(a.S_out)[off] = v;
            }
        return;
    }
    const uint32_t sb = smem_u32(sm);
    auto blob_of = [&](int c) { return a.blobs + ((size_t)(g0 + c) * HV + vh) * BLOB_BYTES; };
    auto gamma_of = [&](int c) { return c < nc ? *reinterpret_cast<const float *>(blob_of(c) + BLOB_G) : 0.0f; };
    auto load_u = [&](int c, float4 (&u)[4]) {        // U[t][j0 .. j0+16) of chunk c
        const float4 *U = reinterpret_cast<const float4 *>(blob_of(c) + BLOB_U + ((size_t)t * DV + j0) * 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) u[e] = trow ? U[e] : make_float4(0.f, 0.f, 0.f, 0.f);
    };

    if (warp == 0) {
        tc::tmem_alloc(smem_u32(&ss.tmem), T2_COLS);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int k = 0; k < 2; ++k) {
            mbar_init(smem_u32(&ss.bar_wq[k]), 1);
            mbar_init(smem_u32(&ss.bar_pk[k]), 1);
            mbar_init(smem_u32(&ss.bar_m1[k]), 1);
            mbar_init(smem_u32(&ss.bar_m2[k]), 1);
            mbar_init(smem_u32(&ss.bar_y[0][k]), 1);
            mbar_init(smem_u32(&ss.bar_y[1][k]), 1);
        }
        mbar_init(smem_u32(&ss.bar_vn), P2_EPI_WARPS);   // one arrival per epilogue warp
        mbar_init(smem_u32(&ss.bar_s), P2_EPI_WARPS);
        mbar_init(smem_u32(&ss.bar_yfree), P2_EPI_WARPS);
        ss.abort = 0;
        fence_mbar_init();
        for (int c = 0; c < 2 && c < nc; ++c) {        // both stages in flight from the start
            carry_issue<true>(blob_of(c), sb, ss, c);
            carry_issue<false>(blob_of(c), sb, ss, c);
        }
    }
    float4 u_cur[4], u_nxt[4];
    float gam_c1 = 0.0f;                               // gamma_n of the next chunk
    if (!issuer) {
        load_u(0, u_cur);
        gam_c1 = gamma_of(1);
    }
    tc::fence_before_sync();
    __syncthreads();
    const uint32_t tm = ss.tmem;
    tc::fence_after_sync();

    // initial state block: bf16 copy in shared memory, gamma_n(0) * S in TMEM
    if (!issuer) {
        const float gam0 = gamma_of(0);
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = a.S_in ? a.S_in[sbase_g + (size_t)(j0 + e) * DK + i] : 0.0f;
        store_s_bf16(sm, i, hf, v);
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] *= gam0;
        tc::tmem_st16(tc::tmem_addr(tm, 32 * q, T2_S + 16 * hf), v);
        tc::wait_st();
    }
    fence_proxy_async_smem();
    tc::fence_before_sync();
    __syncthreads();

    const float scale = rsqrtf((float)DK);
    // y of chunk cy (scale applied), token row t -> [T][4096] buffer, once both
    // issuers' products of that chunk have completed. Each Y buffer has its own
    // barriers, which complete every second chunk.
    auto drain_y = [&](int cy) {
        const uint32_t ph = (uint32_t)((cy >> 1) & 1);
        if (!mbar_wait_bounded(smem_u32(&ss.bar_y[cy & 1][0]), ph) || !mbar_wait_bounded(smem_u32(&ss.bar_y[cy & 1][1]), ph))
            ss.abort = 1;
        tc::fence_after_sync();
        float y[16], y1[16];
        const uint32_t yc = T2_Y + 64 * (cy & 1) + 16 * hf;
        tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, yc), y);
        tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, yc + 32), y1);
        tc::wait_ld();
        const int nvy = max(0, min(CH, seqL - CH * cy));
        if (trow && t < nvy && !ss.abort) {
            float4 *dst = reinterpret_cast<float4 *>(a.ybuf + (size_t)(seq0 + CH * cy + t) * DI + (size_t)vh * DV + j0);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                dst[e] = make_float4((y[4 * e] + y1[4 * e]) * scale, (y[4 * e + 1] + y1[4 * e + 1]) * scale,
                                     (y[4 * e + 2] + y1[4 * e + 2]) * scale, (y[4 * e + 3] + y1[4 * e + 3]) * scale);
        }
    };
    const uint32_t id1 = tc::instr_desc(tc::FMT_BF16, CH, JB) | (1u << 16);   // B (the state) MN-major
    const uint32_t id2s = tc::instr_desc(tc::FMT_TF32, 128, JB), id2y = tc::instr_desc(tc::FMT_TF32, CH, JB);
    const volatile int &aborted = ss.abort;
    if (issuer) {
        if (lane == 0) {
            for (int c = 0; c < nc; ++c) {
                const int st = c & 1;
                const uint32_t spar = (uint32_t)((c >> 1) & 1);   // phase of this stage's load barriers
                const uint32_t wq = sb + (st ? S2_WQ1 : S2_WQ0), pk = sb + (st ? S2_PK1 : S2_PK0);
                const uint32_t vnb = sb + S2_VN + 8192u * st;     // this chunk's Vnew^T buffer
                const uint32_t ycol = T2_Y + 64 * st + 32 * ik;
                // (1) K half i in [64k, 64k+64) of Vn^ = W S, committed alone, then
                //     the same half of Y = Q~ S. Chunk 0's state block was written
                //     before the loop; later ones are announced on bar_s.
                if (c > 0 && !mbar_wait_bounded(smem_u32(&ss.bar_s), (uint32_t)((c - 1) & 1))) ss.abort = 1;
                if (!mbar_wait_bounded(smem_u32(&ss.bar_wq[st]), spar)) ss.abort = 1;
                if (aborted) break;
                tc::fence_after_sync();
                const uint64_t bs = tc::smem_desc(sb + S2_SS + 1024u * ik, 128u, (uint32_t)DK * 16u);
                tc::mma_steps<false>(tm + T2_VN + 32 * ik, tc::kmajor_desc<2>(wq, 64 * ik, DK), bs, 4, id1, false);
                tc::mma_commit(smem_u32(&ss.bar_m1[ik]));
                // this Y buffer last held chunk c - 2, drained after chunk c - 1's state block
                if (c >= 2 && !mbar_wait_bounded(smem_u32(&ss.bar_yfree), (uint32_t)((c - 2) & 1))) ss.abort = 1;
                if (aborted) break;
                tc::fence_after_sync();
                tc::mma_steps<false>(tm + ycol, tc::kmajor_desc<2>(wq + 16384, 64 * ik, DK), bs, 4, id1, false);
                // (2) K half t in [32k, 32k+32) of the state update, into S (k = 0)
                //     or dS (k = 1), committed alone, then the same half of Y += P Vnew
                if (!mbar_wait_bounded(smem_u32(&ss.bar_vn), (uint32_t)(c & 1))) ss.abort = 1;
                if (!mbar_wait_bounded(smem_u32(&ss.bar_pk[st]), spar)) ss.abort = 1;
                if (aborted) break;
                tc::fence_after_sync();
                const uint64_t vn = tc::sw128_desc(vnb + 4096u * ik);   // tokens [32k, 32k+32): atom k
                mma_vn(tm + (ik ? T2_DS : T2_S), tc::kmajor_desc<4>(pk + 16384, 32 * ik, CH), vn, id2s, ik == 0);
                tc::mma_commit(smem_u32(&ss.bar_m2[ik]));
                mma_vn(tm + ycol, tc::kmajor_desc<4>(pk, 32 * ik, CH), vn, id2y, true);
                tc::mma_commit(smem_u32(&ss.bar_y[st][ik]));
            }
        }
    } else {
        float sdec[16];                                // state block to decay into TMEM before this chunk's update
        float gam_dec = 0.0f;                          // its decay: gamma_n of the chunk about to update it
        for (int c = 0; c < nc; ++c) {
            const int st = c & 1;
            const uint32_t par = (uint32_t)(c & 1);   // phase of the per-chunk MMA barriers
            if (c > 0) {                               // previous state block decays for this chunk's update
#pragma unroll
                for (int e = 0; e < 16; ++e) sdec[e] *= gam_dec;
                tc::tmem_st16(tc::tmem_addr(tm, 32 * q, T2_S + 16 * hf), sdec);
            }
            if (c + 1 < nc) load_u(c + 1, u_nxt);      // latency hides behind this chunk's chain
            const float gam_c2 = gamma_of(c + 2);
            if (!mbar_wait_bounded(smem_u32(&ss.bar_m1[0]), par) || !mbar_wait_bounded(smem_u32(&ss.bar_m1[1]), par))
                ss.abort = 1;
            if (aborted) break;
            tc::fence_after_sync();
            // Vnew = U - W S for token row t, columns j0..j0+16 -> Vnew^T tf32 tile
            {
                float d[16], d1[16];
                tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T2_VN + 16 * hf), d);
                tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T2_VN + 32 + 16 * hf), d1);
                tc::wait_ld();
                if (trow) {
                    const float *u = reinterpret_cast<const float *>(u_cur);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        *reinterpret_cast<float *>(sm + S2_VN + 8192u * st + vn_offset(16 * hf + e, t)) =
                            tc::tf32_rn(u[e] - (d[e] + d1[e]));
                }
            }
            tc::wait_st();
            fence_proxy_async_smem();                  // each thread: its stores -> the tensor core
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ss.bar_vn));
            if (!mbar_wait_bounded(smem_u32(&ss.bar_m2[0]), par) || !mbar_wait_bounded(smem_u32(&ss.bar_m2[1]), par))
                ss.abort = 1;
            if (aborted) break;
            tc::fence_after_sync();
            // chunk c - 1's P | K~^T stage was last read by its Y += P Vnew, which
            // completed before this chunk's state update (same issuers, in order)
            if (tid == 0 && c > 0 && c + 1 < nc) carry_issue<false>(blob_of(c + 1), sb, ss, c + 1);
            // W | Q~ of this stage were last read by Y = Q~ S, issued before each state update
            if (tid == 0 && c + 2 < nc) carry_issue<true>(blob_of(c + 2), sb, ss, c + 2);
            // state block S + dS: bf16 copy for the next chunk (its decay waits
            // for the next chunk's Vnew), or the final state out
            {
                float ds[16];
                tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T2_S + 16 * hf), sdec);
                tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, T2_DS + 16 * hf), ds);
                tc::wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) sdec[e] += ds[e];
            }
            if (c + 1 < nc) {
                store_s_bf16(sm, i, hf, sdec);
                fence_proxy_async_smem();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ss.bar_s));
            } else if (a.S_out) {
#pragma unroll
                for (int e = 0; e < 16; ++e) a.S_out[sbase_g + (size_t)(j0 + e) * DK + i] = sdec[e];
            }
            if (c > 0) {                               // y of the previous chunk, off the chain
                drain_y(c - 1);
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ss.bar_yfree));
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) u_cur[e] = u_nxt[e];
            gam_dec = gam_c1;
            gam_c1 = gam_c2;
        }
        if (!aborted) drain_y(nc - 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, T2_COLS);
    if (tid == 0 && ss.abort) atomicExch(&g_chunk_error, (unsigned int)GDN_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- launcher

cudaError_t launch_conv_state_out_bf16(const int32_t *cu, int N, int T_total, const void *qkv, const void *cs_in,
                                       void *cs_out, cudaStream_t s, bool pdl);
int sm_count();
cudaError_t launch_gated_norm_bf16(const float *norm_w, float norm_eps, const void *z, const float *y, void *out,
                                   int T_total, gdn_dtype out_dt, cudaStream_t s, bool pdl);

static size_t off_info(int N) { return ((size_t)(N + 1) * sizeof(int32_t) + 255) & ~(size_t)255; }
static size_t off_blobs(int N, int T_total)
{
    return off_info(N) + ((((size_t)T_total / CH + (size_t)N) * sizeof(int4) + 255) & ~(size_t)255);
}
static size_t off_ybuf(int N, int T_total)
{
    return off_blobs(N, T_total) + ((size_t)T_total / CH + (size_t)N) * HV * BLOB_BYTES;
}

// Workspace of the chunked path: chunk offsets | chunk descriptors | per-(chunk, V-head) blobs | y buffer.
size_t chunk_workspace_bytes(int N, int T_total)
{
    return off_ybuf(N, T_total) + (size_t)T_total * DI * sizeof(float);
}

cudaError_t launch_prefill_chunked(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                                   const void *beta, const int32_t *cu, int N, int T_total, const void *cs_in,
                                   void *cs_out, const float *S_in, float *S_out, void *out, gdn_dtype out_dt,
                                   void *ws_body, cudaStream_t s)
{
    ChunkArgs a;
    a.conv_w = p->conv_w; a.A_log = p->A_log; a.dt_bias = p->dt_bias; a.norm_w = p->norm_w;
    a.norm_eps = p->norm_eps; a.l2_eps = p->l2_eps;
    a.qkv = (const bf16 *)qkv; a.z = (const bf16 *)z; a.alpha = (const bf16 *)alpha; a.beta = (const bf16 *)beta;
    a.cu = cu; a.N = N; a.T_total = T_total;
    a.max_chunks = T_total / CH + N;
    a.cs_in = (const bf16 *)cs_in; a.S_in = S_in; a.S_out = S_out; a.out = out;
    a.chunk_off = static_cast<int32_t *>(ws_body);
    a.chunk_info = reinterpret_cast<int4 *>(static_cast<unsigned char *>(ws_body) + off_info(N));
    a.blobs = static_cast<unsigned char *>(ws_body) + off_blobs(N, T_total);
    a.ybuf = reinterpret_cast<float *>(static_cast<unsigned char *>(ws_body) + off_ybuf(N, T_total));

    cudaError_t e = cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P1_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(chunk_carry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P2_SMEM);
    if (e != cudaSuccess) return e;

    CUtensorMap qkv_map;
    if (T_total > 0 && !make_bf16_plain_map(&qkv_map, qkv, T_total, CC, RAW_COLS, RAW_ROWS))
        return cudaErrorInvalidValue;
    const int n_sm = sm_count();                       // the prep grid is persistent: one CTA per SM
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    // The kernels after the schedule kernel are launched with programmatic
    // stream serialization: each may start while the one ahead finishes, and
    // waits (grid_dep_wait) before it reads that kernel's results.
    chunk_schedule_kernel<<<1, 1024, 0, s>>>(cu, N, T_total, a.max_chunks, a.chunk_off, a.chunk_info);
    e = cudaGetLastError();
    if (e == cudaSuccess && a.max_chunks > 0 && T_total > 0)
        e = launch_pdl(chunk_prep_kernel, dim3((unsigned)std::min(a.max_chunks * HK, n_sm)), dim3(P1_THREADS),
                       P1_SMEM, s, qkv_map, a);
    if (e == cudaSuccess) e = launch_pdl(chunk_carry_kernel, dim3(N, HV, NJB), dim3(P2_THREADS), P2_SMEM, s, a);
    if (e == cudaSuccess)
        e = launch_gated_norm_bf16(p->norm_w, p->norm_eps, z, a.ybuf, out, T_total, out_dt, s, true);
    if (e == cudaSuccess && cs_out) e = launch_conv_state_out_bf16(cu, N, T_total, qkv, cs_in, cs_out, s, true);
    return e;
}

cudaError_t take_chunk_error(unsigned int *word, cudaStream_t s)
{
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(word, g_chunk_error, sizeof(unsigned int), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && *word != 0)
        e = cudaMemcpyToSymbolAsync(g_chunk_error, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

}  // namespace gdn
