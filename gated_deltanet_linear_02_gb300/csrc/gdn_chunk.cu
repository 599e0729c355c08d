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
// The packed token range is processed in windows of at most W tokens (W is set
// by the workspace the caller passes), so the scratch does not grow with the
// prompt: a long prompt runs as a sequence of bounded fragments with the state
// carried between them, as the Lily page does in "Limit temporary memory by
// splitting the prompt into fragments". Per window:
//  wy_plan   the window's sequence fragments and 64-token chunks (from
//            cu_seqlens, on the device); clears the window's flags.
//  wy_act    conv + SiLU over all 8192 channels and the L2 norm of q and k per
//            head -> x^, fp16 [rows of the window][8192]; the gate records.
//  wy_fused  one cooperative grid, one CTA per SM, three roles:
//   prep     (the CTAs past the chains) one item per (chunk, K-head), for both
//            V-heads of the GQA pair, in chunk order: K K^T and Q K^T (one
//            M=128 product), P = Mask o Q K^T, the unit-lower triangular
//            inverse for T, then U^T = V^T T^T and W^T = K^T (T diag(gamma))^T.
//            It writes one operand blob per (chunk, V-head) (W^T, U^T, P, K~^T,
//            Q~) and then a flag.
//   chain    one CTA per (fragment, V-head): the chain over the fragment's
//            chunks, each taken as soon as its prep flag is set. The state
//            lives in tensor memory as S^T (lane = value column j), and its fp16
//            copy is the A operand of the next chunk's products, read from
//            tensor memory, so nothing on the chain goes through shared memory.
//            y goes out as fp16, with a flag per (chunk, V-head).
//   norm     the prep CTAs once their items are done: the gated RMSNorm .
//            silu(z) of (chunk, 4 V-heads) items whose y flags are set.
// Where a one-per-SM cooperative grid cannot be resident, the three roles run as
// the kernels wy_prep, wy_carry and wy_norm, one after the other.
// Operand precision: every product takes fp16 operands (kind::f16) with fp32
// accumulation. fp16 keeps 11 significant bits, the precision of tf32 rounded
// to nearest, at the bf16 rate. The operands are unit-norm keys and queries,
// SiLU outputs, decay-weighted combinations of them and the state, all far
// inside fp16's range (+-65504). The carried state itself stays fp32.
#include "gdn_async.cuh"
#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

#include <cuda_fp16.h>

#include <algorithm>
#include <cstddef>
#include <cstdlib>

namespace gdn {

__device__ unsigned int g_chunk_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

constexpr int CH = 64;                    // chunk length

// ---------------------------------------------------------------- tables
struct WyFrag {            // a sequence's tokens inside one window
    int seq;               // sequence index n
    int row_a, row_b;      // global rows [row_a, row_b)
    int flags;             // 1: starts the sequence, 2: ends the sequence
    int chunk0, nchunks;   // its chunks in the window's chunk table
    int pad0, pad1;
};
struct WyChunk {
    int row0;              // global row of the chunk's first token
    int nv;                // tokens in the chunk (1..64)
    int seq;               // sequence index
    int seq_start;         // the sequence's first global row
};
struct WyCount {
    int n_frag, n_chunks;
    int norm_next;         // one kernel form: the next norm item to hand out
};

// Per (chunk, V-head) operand blob, 72 KiB. The tiles are stored exactly as
// the chain's shared-memory operands, so one bulk copy moves the blob.
constexpr uint32_t BL_WT = 0;          // W^T, fp16, MN-major (N = token t, K = key i),       16 KiB
constexpr uint32_t BL_UT = 16384;      // U^T, fp16, same layout (t, value j),                 16 KiB
constexpr uint32_t BL_P = 32768;       // P = Mask o Q K^T, fp16 K-major [t][s] (Kd 64),       8 KiB
constexpr uint32_t BL_KT = 40960;      // K~ = diag(exp(G_n - G_t)) k^, fp16, two 64-column boxes
                                       // [t][i] in the 128-byte swizzle (as TMA writes x^)  16 KiB
constexpr uint32_t BL_QT = 57344;      // Q~ = diag(gamma_t) q^, fp16, same layout             16 KiB
constexpr uint32_t BLOB_BYTES = 73728;
static_assert(BLOB_BYTES % 1024 == 0, "blobs stay 1 KiB aligned");

// Gate record of one (chunk, V-head), fp32: the chunk-local cumulative
// log-decay G_t, beta_t, gamma_t = exp(G_t), and exp(G_n - G_t) (0 past the
// chunk's tokens); gamma_n = exp(G_n) is gamma_63 (g is 0 past the tokens).
constexpr int GR_G = 0, GR_B = CH, GR_GAM = 2 * CH, GR_KTF = 3 * CH, GATE_FLOATS = 4 * CH;

// (t, c) of a [t][c] fp16 tile stored MN-major with t as the contiguous (N)
// index and c as K: 8-token groups 2 KiB apart, 8-row c groups 128 B apart.
__host__ __device__ __forceinline__ uint32_t mn_off(int t, int c) { return tc::mnmajor_offset_bf16(t, c, 128); }
// (r, s) of a K-major fp16 tile with 64 columns
__host__ __device__ __forceinline__ uint32_t km64(int r, int s) { return tc::kmajor_offset<2>(r, s, 64); }

// silu(z) = z sigmoid(z) = z (1 + tanh(z / 2)) / 2, for the conv outputs and the
// output gate, with the hardware tanh approximation (one special-function
// operation instead of an exponential and a reciprocal; absolute error about
// 5e-4 on tanh, so about 2.5e-4 |z| on silu(z), below the fp16 rounding of x^
// and far below the output tolerance).
__device__ __forceinline__ float silu_gate(float z)
{
    float th;
    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * z));
    const float hz = 0.5f * z;
    return fmaf(hz, th, hz);
}

struct WyArgs {
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    float norm_eps, l2_eps;
    const bf16 *qkv, *z, *alpha, *beta;
    const int32_t *cu;
    int N, T_total;
    const bf16 *cs_in;
    const float *S_in;
    float *S_out;
    void *out;
    // the window
    int w0, wlen, f_cap, c_cap;
    WyCount *count;
    WyFrag *frags;
    WyChunk *chunks;
    __half *xhat;                // [wlen][8192]
    int gates_only;              // x^ comes from the caller (gdn_in_proj_conv): act writes the gates only
    int *flags;                  // [c_cap][16]: item (chunk, K-head) of prep done (one kernel: prep + carry), or NULL
    int *yflags;                 // [c_cap][32]: y of (chunk, V-head) written (one kernel form), or NULL
    int out_f32;                 // out is fp32 (else bf16)
    __half *ybuf;                // [wlen][4096]: y (scale applied) before the gated norm
    float *gates;                // [c_cap][32][4][64]: per (chunk, V-head) G, beta, gamma_t, exp(G_n - G_t)
    unsigned char *blobs;        // [c_cap][32] x BLOB_BYTES
    float *slot_in, *slot_out;   // [32][128][128]: the state of a sequence that crosses a window edge
};

__device__ __forceinline__ int cu_clamp(const int32_t *cu, int i, int lo, int hi)
{
    return min(max(__ldg(cu + i), lo), hi);
}

// ------------------------------------------------------------------ plan
// Fragments of the sequences that have tokens in [w0, w0 + wlen) and their
// 64-token chunks, by a block-wide exclusive scan of both counts. Counts past
// the capacities (possible only for a malformed cu_seqlens) are dropped.
__global__ void __launch_bounds__(1024) wy_plan_kernel(const WyArgs a)
{
    __shared__ int part[2][32];
    grid_dep_wait();                                   // the previous window's carry reads these tables
    grid_dep_launch();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (a.N + 1023) / 1024;
    const int lo = min(tid * per, a.N), hi = min(lo + per, a.N);
    const int e0 = a.w0, e1 = a.w0 + a.wlen;
    int nf = 0, nc = 0;
    for (int n = lo; n < hi; ++n) {
        const int s0 = cu_clamp(a.cu, n, 0, a.T_total), s1 = cu_clamp(a.cu, n + 1, s0, a.T_total);
        const int fa = max(s0, e0), fb = min(s1, e1);
        if (fa < fb) { ++nf; nc += (fb - fa + CH - 1) / CH; }
    }
    int inf = nf, inc = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int vf = __shfl_up_sync(0xffffffffu, inf, o), vc = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) { inf += vf; inc += vc; }
    }
    if (lane == 31) { part[0][warp] = inf; part[1][warp] = inc; }
    __syncthreads();
    if (warp == 0) {
        int wf = part[0][lane], wc = part[1][lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vf = __shfl_up_sync(0xffffffffu, wf, o), vc = __shfl_up_sync(0xffffffffu, wc, o);
            if (lane >= o) { wf += vf; wc += vc; }
        }
        part[0][lane] = wf;
        part[1][lane] = wc;
    }
    __syncthreads();
    int f = (warp ? part[0][warp - 1] : 0) + inf - nf;
    int g = (warp ? part[1][warp - 1] : 0) + inc - nc;
    if (tid == 0) {
        a.count->n_frag = min(part[0][31], a.f_cap);
        a.count->n_chunks = min(part[1][31], a.c_cap);
        a.count->norm_next = 0;
    }
    if (a.flags)                                       // no item of this window is done yet
        for (int i = tid; i < a.c_cap * HK; i += blockDim.x) a.flags[i] = 0;
    if (a.yflags)
        for (int i = tid; i < a.c_cap * HV; i += blockDim.x) a.yflags[i] = 0;
    for (int n = lo; n < hi; ++n) {
        const int s0 = cu_clamp(a.cu, n, 0, a.T_total), s1 = cu_clamp(a.cu, n + 1, s0, a.T_total);
        const int fa = max(s0, e0), fb = min(s1, e1);
        if (fa >= fb) continue;
        const int nch = (fb - fa + CH - 1) / CH;
        if (f < a.f_cap) {
            WyFrag fr;
            fr.seq = n;
            fr.row_a = fa;
            fr.row_b = fb;
            fr.flags = (fa == s0 ? 1 : 0) | (fb == s1 ? 2 : 0);
            fr.chunk0 = min(g, a.c_cap);
            fr.nchunks = max(0, min(nch, a.c_cap - g));
            fr.pad0 = fr.pad1 = 0;
            a.frags[f] = fr;
        }
        for (int c = 0; c < nch && g + c < a.c_cap; ++c) {
            WyChunk ck;
            ck.row0 = fa + CH * c;
            ck.nv = min(CH, fb - ck.row0);
            ck.seq = n;
            ck.seq_start = s0;
            a.chunks[g + c] = ck;
        }
        ++f;
        g += nch;
    }
}

// ------------------------------------------------------------------- act
// x^ = SiLU(conv) over all 8192 channels of a chunk's tokens, with q and k
// L2-normalised per 128-channel head, rounded to fp16. One CTA per (chunk,
// 128-channel head); thread (4 channels, 8 tokens), so a warp holds one head of
// 8 tokens and the head's norm is a warp sum. Each thread issues the loads of
// its 11 rows (3 before its first token) before it computes anything. Rows
// before the sequence start come from conv_state_in (zeros without one).
constexpr int ACT_THREADS = 256;
__global__ void __launch_bounds__(ACT_THREADS) wy_act_kernel(const WyArgs a)
{
    __shared__ float gs[2][2][CH];                     // g (then G) and beta of V-heads y, y + 16
    grid_dep_wait();
    grid_dep_launch();
    const int g = blockIdx.x;
    if (g >= a.count->n_chunks) return;
    const WyChunk ck = a.chunks[g];
    const int tid = threadIdx.x, lane = tid & 31, tg = tid >> 5;
    if (blockIdx.y < HK) {
        // the gates of V-heads y and y + 16 over this chunk (section "Decay gate"):
        // g = -exp(A_log) softplus(alpha + dt_bias), beta = sigmoid(beta); tokens
        // past the chunk get g = 0, beta = 0. Then G = the chunk-local prefix sum.
        const int h = tid >> 6, p = tid & 63, vh = blockIdx.y + HK * h;
        if (tid < 2 * CH) {
            float gg = 0.0f, bb = 0.0f;
            if (p < ck.nv) {
                const size_t r = (size_t)(ck.row0 + p) * HV + vh;
                gg = -expf(__ldg(a.A_log + vh)) * softplus_f(to_f(a.alpha[r]) + __ldg(a.dt_bias + vh));
                bb = 1.0f / (1.0f + expf(-to_f(a.beta[r])));
            }
            gs[h][0][p] = gg;
            gs[h][1][p] = bb;
        }
        __syncthreads();
        if (tg < 2) {                                  // warp h: inclusive scan of head h's log-decays
            const float g0 = gs[tg][0][2 * lane], g1 = gs[tg][0][2 * lane + 1];
            float run = g0 + g1;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float up = __shfl_up_sync(0xffffffffu, run, o);
                if (lane >= o) run += up;
            }
            gs[tg][0][2 * lane] = run - g1;
            gs[tg][0][2 * lane + 1] = run;
        }
        __syncthreads();
        if (tid < 2 * CH) {
            const float Gp = gs[h][0][p], Gn = gs[h][0][CH - 1];
            float *rec = a.gates + ((size_t)g * HV + vh) * GATE_FLOATS;
            rec[GR_G + p] = Gp;
            rec[GR_B + p] = gs[h][1][p];
            rec[GR_GAM + p] = expf(Gp);
            rec[GR_KTF + p] = p < ck.nv ? __expf(Gn - Gp) : 0.0f;
        }
    }
    if (a.gates_only) return;
    const int c0 = blockIdx.y * DK + 4 * lane;
    const int tb = 8 * tg;                             // first token (uniform over the warp)
    if (tb >= ck.nv) return;
    uint2 raw[KC - 1 + 8];
#pragma unroll
    for (int m = 0; m < KC - 1 + 8; ++m) {
        const int t = tb - (KC - 1) + m, pos = ck.row0 + t;
        raw[m] = make_uint2(0u, 0u);
        if (t < ck.nv) {
            if (pos >= ck.seq_start)
                raw[m] = __ldg(reinterpret_cast<const uint2 *>(a.qkv + (size_t)pos * CC + c0));
            else if (a.cs_in)
                raw[m] = __ldg(reinterpret_cast<const uint2 *>(
                    a.cs_in + ((size_t)ck.seq * (KC - 1) + (pos - ck.seq_start + KC - 1)) * CC + c0));
        }
    }
    float w[4][4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float4 t4 = __ldg(reinterpret_cast<const float4 *>(a.conv_w) + c0 + e);
        w[e][0] = t4.x; w[e][1] = t4.y; w[e][2] = t4.z; w[e][3] = t4.w;
    }
    const bool norm = c0 < V_OFF;                      // q and k channels
    auto chan = [&](int m, int e) {                    // channel c0 + e of row m, bf16 -> fp32
        const uint32_t u = e < 2 ? raw[m].x : raw[m].y;
        return __uint_as_float((e & 1) ? (u & 0xFFFF0000u) : (u << 16));
    };
    __half *dst = a.xhat + (size_t)(ck.row0 - a.w0 + tb) * CC + c0;
    const int tn = min(8, ck.nv - tb);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        if (t >= tn) break;                            // uniform over the warp
        float o[4];
        float s2 = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float u = w[e][0] * chan(t, e) + w[e][1] * chan(t + 1, e) + w[e][2] * chan(t + 2, e) +
                            w[e][3] * chan(t + 3, e);
            o[e] = silu_gate(u);                       // one special-function operation (tanh)
            s2 += o[e] * o[e];
        }
        if (norm) {
            const float inv = rsqrtf(warp_sum(s2) + a.l2_eps);
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] *= inv;
        }
        *reinterpret_cast<uint2 *>(dst + (size_t)t * CC) = make_uint2(tc::pack_half2(o[0], o[1]), tc::pack_half2(o[2], o[3]));
    }
}

// ------------------------------------------------------------------- prep
// One item per (chunk, K-head kh), with both V-heads vh = kh + 16 h (h = 0, 1).
// One CTA of 16 warps per SM, persistent over the items; the x^ tiles of the
// next item are loaded into the other of two buffers while the current item
// runs.
constexpr int PR_THREADS = 512;
// x^ tiles, fp16, 64 rows x 64 columns each, 128-byte swizzle (as TMA writes
// them): q^ and k^ of the K-head interleaved so that [q^; k^] is one 128-row
// K-major operand (rows 0-63 q^, rows 64-127 k^), then v^ of the two V-heads.
constexpr uint32_t PR_Q0 = 0, PR_K0 = 8192, PR_Q1 = 16384, PR_K1 = 24576;
constexpr uint32_t PR_V0 = 32768, PR_V1 = 49152;   // columns 0-63 at +0, 64-127 at +8 KiB
constexpr uint32_t PR_X_BYTES = 65536;             // one buffer; two at 0 and 64 KiB
constexpr uint32_t PR_LT = 131072;     // per head, 16 KiB: beta_t L[t][s] fp32 (lb_at), later T | T' fp16
constexpr int XLD = 68;                // row stride (floats) of the inverse X
constexpr uint32_t PR_XI = 163840;     // per head: X = (I + A)^-1, fp32 [64][68]    (17 KiB)
constexpr uint32_t PR_M = 198656;      // per head: block products, fp32 [32][36]     (4.5 KiB)
constexpr int MLD = 36;
constexpr uint32_t PR_SMALL = 207872;
struct PrSmall {
    float gr[2][2][GATE_FLOATS];       // gate records [buffer][V-head of the pair], loaded with the tiles
    uint64_t bar_x[2];                 // the x^ tiles and gate records, per buffer
    uint64_t bar_qk, bar_uw;           // tensor-core completions
    uint32_t tmem;
    int abort;
};
constexpr size_t PR_SMEM = PR_SMALL + sizeof(PrSmall) + 1024;
static_assert(PR_SMEM <= 232448, "prep shared memory");
// tensor-memory columns: [Q K^T; K K^T] (M=128, N=64); U^T and W^T of both heads (M=128, N=64)
constexpr uint32_t TP_QK = 0, TP_UW = 64, TP_COLS = 512;   // U0 W0 U1 W1 at 64, 128, 192, 256

// Float index of L[t][s] in a [64][64] tile whose 16-byte groups are XOR-swizzled
// by the row: rows written one per lane spread over the banks, and a row still
// reads as float4 groups of 4 consecutive s.
__device__ __forceinline__ int lb_at(int t, int s) { return t * CH + (((s >> 2) ^ (t & 15)) << 2) + (s & 3); }

// The dynamic shared-memory block rounded up to a 1024-byte boundary (the
// 128-byte swizzle of TMA boxes repeats every 1 KiB).
__device__ __forceinline__ unsigned char *smem_aligned1024(unsigned char *raw)
{
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// The prep work of CTA `cta` of `n_ctas` (items cta, cta + n_ctas, ..).
__device__ __forceinline__ void wy_prep_body(const CUtensorMap &xmap, const WyArgs &a, int cta, int n_ctas)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = smem_aligned1024(smem_raw);
    PrSmall &ss = *reinterpret_cast<PrSmall *>(sm + PR_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sb = smem_u32(sm);
    auto Lf = [&](int h) { return reinterpret_cast<float *>(sm + PR_LT + h * 16384); };
    auto Xi = [&](int h) { return reinterpret_cast<float *>(sm + PR_XI + h * (CH * XLD * 4)); };
    auto Mm = [&](int h) { return reinterpret_cast<float *>(sm + PR_M + h * (32 * MLD * 4)); };

    grid_dep_wait();                                   // x^ and the chunk table come from the kernels ahead
    grid_dep_launch();
    const int n_items = a.count->n_chunks * HK;
    auto stage = [&](int it, int buf) {                // caller: thread 0
        const WyChunk ck = a.chunks[it / HK];
        const int kh = it % HK, y = ck.row0 - a.w0;
        const uint32_t xb = sb + (uint32_t)buf * PR_X_BYTES;
        const uint32_t bx = smem_u32(&ss.bar_x[buf]);
        mbar_arrive_expect_tx(bx, PR_X_BYTES + 2 * GATE_FLOATS * 4);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            bulk_g2s(smem_u32(&ss.gr[buf][h][0]), a.gates + ((size_t)(it / HK) * HV + kh + HK * h) * GATE_FLOATS,
                     GATE_FLOATS * 4, bx);
        tma_load_2d(xb + PR_Q0, &xmap, Q_OFF + kh * DK, y, bx);
        tma_load_2d(xb + PR_Q1, &xmap, Q_OFF + kh * DK + 64, y, bx);
        tma_load_2d(xb + PR_K0, &xmap, K_OFF + kh * DK, y, bx);
        tma_load_2d(xb + PR_K1, &xmap, K_OFF + kh * DK + 64, y, bx);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v0 = V_OFF + (kh + HK * h) * DV;
            tma_load_2d(xb + (h ? PR_V1 : PR_V0), &xmap, v0, y, bx);
            tma_load_2d(xb + (h ? PR_V1 : PR_V0) + 8192, &xmap, v0 + 64, y, bx);
        }
    };
    if (warp == 0) {
        tc::tmem_alloc(smem_u32(&ss.tmem), TP_COLS);
        tc::tmem_relinquish();
    }
    const int stride = n_ctas;
    int item = cta;
    if (tid == 0) {
        mbar_init(smem_u32(&ss.bar_x[0]), 1);
        mbar_init(smem_u32(&ss.bar_x[1]), 1);
        mbar_init(smem_u32(&ss.bar_qk), 1);
        mbar_init(smem_u32(&ss.bar_uw), 2);            // one commit per head's issuer
        ss.abort = 0;
        fence_mbar_init();
        if (item < n_items) stage(item, 0);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = ss.tmem;
    const int q = warp & 3;                            // TMEM lane quarter
    int n = 0;                                         // items done by this CTA
    int pend_buf = -1;                                 // thread 0: buffer of a copy not yet waited for
    uint32_t pend_par = 0;
    if (tid == 0 && item < n_items) pend_buf = 0;

    for (; item < n_items; item += stride, ++n) {
        const int g = item / HK, kh = item % HK;
        const WyChunk ck = a.chunks[g];
        const int nv = ck.nv;
        const int buf = n & 1;
        const uint32_t xb = sb + (uint32_t)buf * PR_X_BYTES;
        unsigned char *blob0 = a.blobs + ((size_t)g * HV + kh) * BLOB_BYTES;
        auto blob = [&](int h) { return blob0 + (size_t)h * HK * BLOB_BYTES; };

        // ---- [q^; k^] k^T once this item's tiles have landed; the next item's tiles
        //      go to the other buffer, whose last reader (the previous item's U/W
        //      products) has completed
        if (tid == 0) {
            if (!mbar_wait_sleep(smem_u32(&ss.bar_x[buf]), (uint32_t)((n >> 1) & 1))) ss.abort = 1;
            pend_buf = -1;
            tc::fence_after_sync();
            const uint32_t id = tc::instr_desc(tc::FMT_F16, 128, CH);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32);
                tc::mma_f16(tm + TP_QK, tc::sw128_desc(xb + PR_Q0 + off), tc::sw128_desc(xb + PR_K0 + off), id,
                            kk > 0 ? 1u : 0u);
            }
            tc::mma_commit(smem_u32(&ss.bar_qk));
            if (item + stride < n_items && !ss.abort) {
                stage(item + stride, buf ^ 1);
                pend_buf = buf ^ 1;
                pend_par = (uint32_t)(((n + 1) >> 1) & 1);
            }
        }
        // the gate records of both V-heads (loaded with the tiles; thread 0 waited)
        const float (*gr)[GATE_FLOATS] = ss.gr[buf];
        auto Gof = [&](int h, int t) { return gr[h][GR_G + t]; };
        if (!mbar_wait_sleep(smem_u32(&ss.bar_qk), (uint32_t)(n & 1))) ss.abort = 1;
        tc::fence_after_sync();
        __syncthreads();                               // the records are visible to every thread
        // ---- P (rows 0-63 of the product) to the blobs; beta L (rows 64-127) to shared
        //      memory. Thread: one row, 16 columns [16 cq, 16 cq + 16), both heads.
        {
            const int cq = warp >> 2;
            float qk[16];
            tc::tmem_ld16(tc::tmem_addr(tm, 32 * q, TP_QK + 16 * cq), qk);
            tc::wait_ld();
            const int t = 32 * (q & 1) + lane;         // token row within its half of the product
            const int s0 = 16 * cq;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float Gt = Gof(h, t);
                if (q < 2) {
                    uint32_t wd[8];
#pragma unroll
                    for (int e2 = 0; e2 < 8; ++e2) {
                        float pv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int s = s0 + 2 * e2 + e;
                            pv[e] = (s <= t && t < nv) ? __expf(Gt - Gof(h, s)) * qk[2 * e2 + e] : 0.0f;
                        }
                        wd[e2] = tc::pack_half2(pv[0], pv[1]);
                    }
                    unsigned char *P = blob(h) + BL_P;
                    *reinterpret_cast<uint4 *>(P + km64(t, s0)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                    *reinterpret_cast<uint4 *>(P + km64(t, s0 + 8)) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
                } else {
                    const float bt = gr[h][GR_B + t];
                    float *L = Lf(h);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        float lv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int s = s0 + 4 * c4 + e;
                            lv[e] = (s < t && t < nv) ? bt * __expf(Gt - Gof(h, s)) * qk[4 * c4 + e] : 0.0f;
                        }
                        *reinterpret_cast<float4 *>(L + lb_at(t, s0 + 4 * c4)) = make_float4(lv[0], lv[1], lv[2], lv[3]);
                    }
                }
            }
        }
        __syncthreads();
        // ---- X = (I + A)^-1, A = diag(beta) L strictly lower, for both heads, by
        //      blocks: forward substitution inside the four 16-row diagonal blocks,
        //      then two doubling levels, each X_BA = -X_BB (A_BA X_AA) (block row B
        //      of (I + A) X = I), for 16-row and then 32-row blocks.
        if (tid < 128) {                               // level 1: thread (head, block, column)
            const int h = tid >> 6, I = (tid >> 4) & 3, c = tid & 15;
            const float *L = Lf(h);
            float *X = Xi(h);
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = 0.0f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc[4] = {(r == c) ? 1.0f : 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int s4 = 0; s4 < (r + 3) / 4; ++s4) {
                    const float4 l4 = *reinterpret_cast<const float4 *>(L + lb_at(16 * I + r, 16 * I + 4 * s4));
                    acc[0] = fmaf(-l4.x, x[4 * s4], acc[0]);
                    acc[1] = fmaf(-l4.y, x[4 * s4 + 1], acc[1]);
                    acc[2] = fmaf(-l4.z, x[4 * s4 + 2], acc[2]);
                    acc[3] = fmaf(-l4.w, x[4 * s4 + 3], acc[3]);
                }
                x[r] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) X[(16 * I + r) * XLD + 16 * I + c] = x[r];
        } else {
            // meanwhile: K~ = diag(exp(G_n - G_t)) k^ and Q~ = diag(gamma_t) q^ of both
            // heads to the blobs, in the swizzled layout of the x^ tiles (16-byte
            // unit w of a box holds row w / 8)
            for (int u = tid - 128; u < 4096; u += PR_THREADS - 128) {
                const int isq = u >> 11, h = (u >> 10) & 1, b = (u >> 9) & 1, w = u & 511, t = w >> 3;
                const uint32_t src = isq ? (b ? PR_Q1 : PR_Q0) : (b ? PR_K1 : PR_K0);
                const uint4 kv = *reinterpret_cast<const uint4 *>(sm + (uint32_t)buf * PR_X_BYTES + src + 16 * w);
                const float fsc = gr[h][(isq ? GR_GAM : GR_KTF) + t];
                const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 x2 = __half22float2(*reinterpret_cast<const __half2 *>(&kk[i]));
                    o[i] = tc::pack_half2(x2.x * fsc, x2.y * fsc);
                }
                *reinterpret_cast<uint4 *>(blob(h) + (isq ? BL_QT : BL_KT) + 8192 * b + 16 * w) =
                    make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncthreads();
        {                                              // level 2a: M = A_BA X_AA for 16-row pairs
            const int h = tid >> 8, P = (tid >> 7) & 1, r = (tid >> 3) & 15, c = 2 * (tid & 7);
            const int rA = 32 * P, rB = 32 * P + 16;  // block A rows/cols, block B rows
            const float *L = Lf(h), *X = Xi(h);
            float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
                const float4 l4 = *reinterpret_cast<const float4 *>(L + lb_at(rB + r, rA + 4 * k4));
                const float lk[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 x2 = *reinterpret_cast<const float2 *>(X + (rA + 4 * k4 + e) * XLD + rA + c);
                    m0 = fmaf(lk[e], x2.x, m0);
                    m1 = fmaf(lk[e], x2.y, m1);
                }
            }
            *reinterpret_cast<float2 *>(Mm(h) + (16 * P + r) * MLD + c) = make_float2(m0, m1);
        }
        __syncthreads();
        {                                              // level 2b: X_BA = -X_BB M
            const int h = tid >> 8, P = (tid >> 7) & 1, r = (tid >> 3) & 15, c = 2 * (tid & 7);
            const int rA = 32 * P, rB = 32 * P + 16;
            float *X = Xi(h);
            const float *M = Mm(h);
            float x0 = 0.0f, x1 = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float xb = X[(rB + r) * XLD + rB + k];
                const float2 m2 = *reinterpret_cast<const float2 *>(M + (16 * P + k) * MLD + c);
                x0 = fmaf(xb, m2.x, x0);
                x1 = fmaf(xb, m2.y, x1);
            }
            *reinterpret_cast<float2 *>(X + (rB + r) * XLD + rA + c) = make_float2(-x0, -x1);
            // the block above the diagonal is zero; the 32-row level reads it
            *reinterpret_cast<float2 *>(X + (rA + r) * XLD + rB + c) = make_float2(0.0f, 0.0f);
        }
        __syncthreads();
        // level 3 (32-row halves) on 128 threads, each a 4 x 4 block of its head's
        // 32 x 32 product: 8 vector loads per 64 multiply-adds
        if (tid < 128) {                               // level 3a: M = A_BA X_AA
            const int h = tid >> 6, r0 = 4 * ((tid >> 3) & 7), c0 = 4 * (tid & 7);
            const float *L = Lf(h), *X = Xi(h);
            float m[4][4] = {};
#pragma unroll 2
            for (int k4 = 0; k4 < 8; ++k4) {
                float av[4][4], xv[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 l4 = *reinterpret_cast<const float4 *>(L + lb_at(32 + r0 + i, 4 * k4));
                    av[i][0] = l4.x; av[i][1] = l4.y; av[i][2] = l4.z; av[i][3] = l4.w;
                    const float4 x4 = *reinterpret_cast<const float4 *>(X + (4 * k4 + i) * XLD + c0);
                    xv[i][0] = x4.x; xv[i][1] = x4.y; xv[i][2] = x4.z; xv[i][3] = x4.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) m[i][jj] = fmaf(av[i][e], xv[e][jj], m[i][jj]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4 *>(Mm(h) + (r0 + i) * MLD + c0) = make_float4(m[i][0], m[i][1], m[i][2], m[i][3]);
        }
        __syncthreads();
        if (tid < 128) {                               // level 3b: X_BA = -X_BB M
            const int h = tid >> 6, r0 = 4 * ((tid >> 3) & 7), c0 = 4 * (tid & 7);
            float *X = Xi(h);
            const float *M = Mm(h);
            float x[4][4] = {};
#pragma unroll 2
            for (int k4 = 0; k4 < 8; ++k4) {
                float bv[4][4], mv[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 b4 = *reinterpret_cast<const float4 *>(X + (32 + r0 + i) * XLD + 32 + 4 * k4);
                    bv[i][0] = b4.x; bv[i][1] = b4.y; bv[i][2] = b4.z; bv[i][3] = b4.w;
                    const float4 m4 = *reinterpret_cast<const float4 *>(M + (4 * k4 + i) * MLD + c0);
                    mv[i][0] = m4.x; mv[i][1] = m4.y; mv[i][2] = m4.z; mv[i][3] = m4.w;
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) x[i][jj] = fmaf(bv[i][e], mv[e][jj], x[i][jj]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4 *>(X + (32 + r0 + i) * XLD + c0) = make_float4(-x[i][0], -x[i][1], -x[i][2], -x[i][3]);
        }
        __syncthreads();
        {                                              // T = X diag(beta), T' = T diag(gamma): fp16, K-major
            // thread (head, 16-column group, token row t); lanes walk t, so each quarter
            // warp's 16-byte stores fill one core matrix
            const int h = tid >> 8, g2 = 2 * ((tid >> 6) & 3), t = tid & 63;
            const float *X = Xi(h);
            unsigned char *Ts = sm + PR_LT + h * 16384;   // L is no longer needed: T at +0, T' at +8 KiB
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
                const int s0 = 8 * (g2 + gg);
                float xv[8], bv[8], gv[8];
#pragma unroll
                for (int e4 = 0; e4 < 2; ++e4) {
                    const float4 x4 = *reinterpret_cast<const float4 *>(X + t * XLD + s0 + 4 * e4);
                    const float4 b4 = *reinterpret_cast<const float4 *>(&gr[h][GR_B + s0 + 4 * e4]);
                    const float4 m4 = *reinterpret_cast<const float4 *>(&gr[h][GR_GAM + s0 + 4 * e4]);
                    xv[4 * e4] = x4.x; xv[4 * e4 + 1] = x4.y; xv[4 * e4 + 2] = x4.z; xv[4 * e4 + 3] = x4.w;
                    bv[4 * e4] = b4.x; bv[4 * e4 + 1] = b4.y; bv[4 * e4 + 2] = b4.z; bv[4 * e4 + 3] = b4.w;
                    gv[4 * e4] = m4.x; gv[4 * e4 + 1] = m4.y; gv[4 * e4 + 2] = m4.z; gv[4 * e4 + 3] = m4.w;
                }
                uint32_t wt[4], wp[4];
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    float tv[2], pv[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int k = 2 * e2 + e;
                        tv[e] = s0 + k <= t ? xv[k] * bv[k] : 0.0f;
                        pv[e] = tv[e] * gv[k];
                    }
                    wt[e2] = tc::pack_half2(tv[0], tv[1]);
                    wp[e2] = tc::pack_half2(pv[0], pv[1]);
                }
                *reinterpret_cast<uint4 *>(Ts + km64(t, s0)) = make_uint4(wt[0], wt[1], wt[2], wt[3]);
                *reinterpret_cast<uint4 *>(Ts + 8192 + km64(t, s0)) = make_uint4(wp[0], wp[1], wp[2], wp[3]);
            }
        }
        fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        // ---- U^T = V^T T^T and W^T = K^T T'^T per head (M=128, N=64, K=64), A read
        //      MN-major from the swizzled x^ tiles; head h issued by thread 32 h
        if ((tid == 0 || tid == 32) && !ss.abort) {
            tc::fence_after_sync();
            const int h = tid >> 5;
            const uint32_t id = tc::instr_desc(tc::FMT_F16, 128, CH) | tc::IDESC_A_MN;
            const uint32_t vb = xb + (h ? PR_V1 : PR_V0);
            const uint32_t tb = sb + PR_LT + h * 16384;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                tc::mma_f16(tm + TP_UW + 128 * h, tc::sw128_mn_desc(vb + 2048u * kk, 8192u),
                            tc::kmajor_desc<2>(tb, 16 * kk, CH), id, kk > 0 ? 1u : 0u);
                tc::mma_f16(tm + TP_UW + 128 * h + 64, tc::sw128_mn_desc(xb + PR_K0 + 2048u * kk, PR_K1 - PR_K0),
                            tc::kmajor_desc<2>(tb + 8192, 16 * kk, CH), id, kk > 0 ? 1u : 0u);
            }
            tc::mma_commit(smem_u32(&ss.bar_uw));
        }
        if (!ss.abort && !mbar_wait_sleep(smem_u32(&ss.bar_uw), (uint32_t)(n & 1))) ss.abort = 1;
        tc::fence_after_sync();
        // ---- U^T and W^T of both heads to the blobs: warp w drains accumulator w / 4
        //      (U0, W0, U1, W1), lanes 32 (w % 4)..+31 (value j or key i); fp16, 8
        //      tokens per 16-byte store
        {
            const int acc = warp >> 2, h = acc >> 1, isw = acc & 1;
            const int row = 32 * q + lane;
            unsigned char *dstt = blob(h) + (isw ? BL_WT : BL_UT);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                float v[32];
                tc::tmem_ld32(tc::tmem_addr(tm, 32 * q, TP_UW + 64 * acc + 32 * half), v);
                tc::wait_ld();
                if (!ss.abort) {
#pragma unroll
                    for (int g8 = 0; g8 < 4; ++g8)
                        *reinterpret_cast<uint4 *>(dstt + mn_off(32 * half + 8 * g8, row)) =
                            make_uint4(tc::pack_half2(v[8 * g8], v[8 * g8 + 1]), tc::pack_half2(v[8 * g8 + 2], v[8 * g8 + 3]),
                                       tc::pack_half2(v[8 * g8 + 4], v[8 * g8 + 5]),
                                       tc::pack_half2(v[8 * g8 + 6], v[8 * g8 + 7]));
                }
            }
        }
        tc::fence_before_sync();
        if (a.flags) __threadfence();                  // the item's blob writes, before its flag
        __syncthreads();                               // TMEM, the gates and the T tiles are reused
        if (a.flags && tid == 0 && !ss.abort)          // the carry CTAs of the one-kernel form may go on
            asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(a.flags + item), "r"(1) : "memory");
        if (ss.abort) break;
    }
    // after an abort: a copy still in flight lands before the CTA exits
    if (tid == 0 && pend_buf >= 0) mbar_wait_sleep(smem_u32(&ss.bar_x[pend_buf]), pend_par);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tm, TP_COLS);
    if (tid == 0 && ss.abort) atomicExch(&g_chunk_error, (unsigned int)GDN_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(PR_THREADS, 1) wy_prep_kernel(const __grid_constant__ CUtensorMap xmap,
                                                               const WyArgs a)
{
    wy_prep_body(xmap, a, (int)blockIdx.x, (int)gridDim.x);
}

// ------------------------------------------------------------------ carry
// The chain of one (fragment, V-head vh): a CTA of the one-kernel form, or of
// wy_carry. The state is kept transposed, S^T[j][i] (lane = value column j,
// column = key i): then every product has the 128 value columns as its M
// dimension, and the fp16 state and the fp16 Vnew are A operands read straight
// from tensor memory. Per chunk, with K~ = diag(exp(G_n - G_t)) k^ and
// Q~ = diag(gamma_t) q^ from prep:
//   (1) (W S)^T[j][t] = sum_i S^T[j][i] W[t][i]   K = 128, split over two issuers
//       Y1^T[j][t]    = sum_i S^T[j][i] Q~[t][i]  (a third issuer)
//   (E1) Vnew^T = U^T - (W S)^T, zero past the chunk's tokens (their rows of U
//       and W are zero), stored once as fp16 in tensor memory: the A operand of
//       both products of (2)
//   (2) S^T[j][i] += sum_t Vnew^T[j][t] K~[t][i]   (tensor memory holds gamma_n S^T
//       beforehand)
//       Y2^T[j][t]  = sum_s Vnew^T[j][s] P[t][s]
//   (E2) S^T -> fp16 copy for the next chunk's products; gamma_n(next) S^T back.
//   (O)  y = scale (Y1 + Y2) as fp16 to the window's y buffer, off the chain. The
//        gated RMSNorm . silu(z) runs on other SMs: the norm items of the one-kernel
//        form, or wy_norm.
// Warps 0-7 run E1/E2 (lane quarter w % 4, half w / 4); warps 8-11 the output;
// warp 12 loads operands; warps 13-15 issue MMAs. The issuers and the producer
// take no part in CTA-wide barriers; every handoff is an mbarrier.
constexpr int CA_THREADS = 32 * 16;
constexpr int CA_PRODUCER = 12, CA_ISSUER0 = 13;       // warp 12: the blob copies; 13-15: the MMA issuers
constexpr uint32_t ST_BLOB = 0;                         // the blob (W^T | U^T | P | K~ | Q~ | gamma_n)
constexpr uint32_t STAGE_BYTES = BLOB_BYTES;
constexpr uint32_t CA_SMALL = 2 * STAGE_BYTES;
struct CaSmall {
    // the mbarriers first: CA_NBAR words
    uint64_t full[2], free_[2];        // operand stages
    uint64_t m1a, m1b, m2, y;          // tensor-core completions
    uint64_t vn, s16, dec, yfree;      // epilogue handoffs
    uint64_t done[3];                  // each issuer's MMAs have all completed
    uint32_t tmem;
    int abort;
};
constexpr int CA_NBAR = 15;
static_assert(offsetof(CaSmall, tmem) == CA_NBAR * sizeof(uint64_t), "the mbarriers lead CaSmall");
constexpr size_t CA_SMEM = CA_SMALL + sizeof(CaSmall) + 1024;
static_assert(CA_SMEM <= 232448, "carry shared memory");
constexpr int CA_FREE_ARRIVALS = 3 + 8;                 // three issuer commits, E1 warps
// tensor-memory columns
constexpr uint32_t TC_S = 0;       // S^T fp32 [j][i]                                      128
constexpr uint32_t TC_S16 = 128;   // S^T fp16 pairs (A operand, K = i), two buffers at +64k  128
constexpr uint32_t TC_WSA = 256;   // (W S)^T, keys 0-63                                    64
constexpr uint32_t TC_WSB = 320;   // (W S)^T, keys 64-127                                  64
constexpr uint32_t TC_AVP = 384;   // Vnew^T, fp16 pairs (A operand, K = t)                   32
constexpr uint32_t TC_Y = 448;     // Y^T = (Q~ S + P Vnew)^T                               64
constexpr uint32_t TC_COLS = 512;

// OR of a flag over the threads of a named barrier (the barrier itself included).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t count, bool p)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
                 "bar.red.or.pred b, %2, %3, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
                 : "=r"(r) : "r"((uint32_t)p), "r"(id), "r"(count) : "memory");
    return r != 0;
}
__device__ __forceinline__ void bar_named(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <typename TO> __device__ __forceinline__ void store_out4(TO *p, float a, float b, float c, float d);
template <> __device__ __forceinline__ void store_out4<float>(float *p, float a, float b, float c, float d)
{
    *reinterpret_cast<float4 *>(p) = make_float4(a, b, c, d);
}
template <> __device__ __forceinline__ void store_out4<bf16>(bf16 *p, float a, float b, float c, float d)
{
    store4(p, make_float4(a, b, c, d));
}

// The chain of fragment f, V-head vh. Returns true when it gave up on a wait.
// `again`: the CTA runs further chains after this one, so it keeps its right to
// allocate tensor memory and ends its mbarriers' life on the way out.
__device__ __forceinline__ bool wy_carry_body(const WyArgs &a, int f, int vh, bool again)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = smem_aligned1024(smem_raw);
    CaSmall &ss = *reinterpret_cast<CaSmall *>(sm + CA_SMALL);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    grid_dep_wait();                                   // blobs and tables come from the kernels ahead
    grid_dep_launch();
    if (f >= a.count->n_frag) return false;
    const WyFrag fr = a.frags[f];
    const int nc = fr.nchunks;
    if (nc <= 0) return false;
    const uint32_t sb = smem_u32(sm);
    const float *S_src = (fr.flags & 1) ? (a.S_in ? a.S_in + ((size_t)fr.seq * HV + vh) * (DV * DK) : nullptr)
                                        : a.slot_in + (size_t)vh * (DV * DK);
    float *S_dst = (fr.flags & 2) ? (a.S_out ? a.S_out + ((size_t)fr.seq * HV + vh) * (DV * DK) : nullptr)
                                  : a.slot_out + (size_t)vh * (DV * DK);
    auto blob_of = [&](int c) { return a.blobs + ((size_t)(fr.chunk0 + c) * HV + vh) * BLOB_BYTES; };
    // gamma_n of chunk c: gamma_t of its last row (g is 0 past the chunk's tokens)
    auto gamma_n = [&](int c) { return __ldg(a.gates + ((size_t)(fr.chunk0 + c) * HV + vh) * GATE_FLOATS + GR_GAM + CH - 1); };
    auto nv_of = [&](int c) { return min(CH, fr.row_b - fr.row_a - CH * c); };
    auto s16_of = [&](int c) { return TC_S16 + 64u * (uint32_t)(c & 1); };   // fp16 state the chunk's products read

    if (warp == 0) {
        tc::tmem_alloc(smem_u32(&ss.tmem), TC_COLS);
        if (!again) tc::tmem_relinquish();
    }
    if (tid == 0) {
        for (int k = 0; k < 2; ++k) {
            mbar_init(smem_u32(&ss.full[k]), 1);
            mbar_init(smem_u32(&ss.free_[k]), CA_FREE_ARRIVALS);
        }
        mbar_init(smem_u32(&ss.m1a), 1);
        mbar_init(smem_u32(&ss.m1b), 1);
        mbar_init(smem_u32(&ss.m2), 1);
        mbar_init(smem_u32(&ss.y), 1);
        mbar_init(smem_u32(&ss.vn), 8);
        mbar_init(smem_u32(&ss.s16), 8);
        mbar_init(smem_u32(&ss.dec), 8);
        mbar_init(smem_u32(&ss.yfree), 4);
        for (int k = 0; k < 3; ++k) mbar_init(smem_u32(&ss.done[k]), 1);
        ss.abort = 0;
        fence_mbar_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tm = ss.tmem;
    const volatile int &aborted = ss.abort;
    auto wait = [&](uint64_t &bar, uint32_t parity) {
        if (!mbar_wait_sleep(smem_u32(&bar), parity)) ss.abort = 1;
        return !aborted;
    };

    if (warp == CA_PRODUCER) {
        // ---------------------------------------------------------- producer: one bulk copy per chunk
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nc; ++c) {
                const int st = c & 1, u = c >> 1;
                if (u >= 1 && !wait(ss.free_[st], (uint32_t)((u - 1) & 1))) break;
                if (a.flags) {
                    // one-kernel form: the chunk's blob is written by a prep CTA of this
                    // grid; wait for its flag (bounded), then let the copy (async
                    // proxy) see those writes
                    const int *fl = a.flags + (size_t)(fr.chunk0 + c) * HK + (vh % HK);
                    uint64_t t0 = 0;
                    bool ready = false;
                    for (uint32_t it = 0;; ++it) {
                        int v;
                        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(fl) : "memory");
                        if (v) { ready = true; break; }
                        if (it == 0) t0 = global_timer_ns();
                        else if (global_timer_ns() - t0 > WAIT_LIMIT_NS) break;
                        __nanosleep(128);
                    }
                    if (!ready) { ss.abort = 1; break; }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                const uint32_t bar = smem_u32(&ss.full[st]);
                mbar_arrive_expect_tx(bar, STAGE_BYTES);
                bulk_g2s(sb + (uint32_t)st * STAGE_BYTES + ST_BLOB, blob_of(c), BLOB_BYTES, bar);
                issued = c + 1;
            }
            for (int c = max(0, issued - 2); c < issued; ++c)   // copies in flight land before the CTA exits
                mbar_wait_sleep(smem_u32(&ss.full[c & 1]), (uint32_t)((c >> 1) & 1));
        }
    } else if (warp >= CA_ISSUER0) {
        // ---------------------------------------------------------- MMA issuers
        // 13: (W S)^T keys 0-63, then the state update (the chain);
        // 14: (W S)^T keys 64-127;  15: Y = Q~ S + P Vnew.
        if (lane == 0) {
            const int role = warp - CA_ISSUER0;
            const uint32_t id_ws = tc::instr_desc(tc::FMT_F16, 128, CH) | tc::IDESC_B_MN;
            const uint32_t id_s = tc::instr_desc(tc::FMT_F16, 128, DK) | tc::IDESC_B_MN;
            const uint32_t id_y = tc::instr_desc(tc::FMT_F16, 128, CH);
            for (int c = 0; c < nc; ++c) {
                const int st = c & 1;
                const uint32_t par = (uint32_t)(c & 1), spar = (uint32_t)((c >> 1) & 1);
                const uint32_t base = sb + (uint32_t)st * STAGE_BYTES + ST_BLOB;
                const uint32_t s16 = tm + s16_of(c);
                if (!wait(ss.s16, par) || !wait(ss.full[st], spar)) break;
                if (role == 2 && c > 0 && !wait(ss.yfree, (uint32_t)((c - 1) & 1))) break;
                tc::fence_after_sync();
                if (role < 2) {
                    // (1) this issuer's K half of (W S)^T
                    const int k0 = 4 * role;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_f16_tmem_a(tm + (role ? TC_WSB : TC_WSA), s16 + 8 * (k0 + kk),
                                           tc::mn_desc(base + BL_WT + 256u * (k0 + kk), 2048u), id_ws, kk > 0 ? 1u : 0u);
                    tc::mma_commit(smem_u32(role ? &ss.m1b : &ss.m1a));
                }
                if (role == 0) {
                    // (2) the state update, once Vnew and the decayed state are in
                    if (!wait(ss.vn, par) || !wait(ss.dec, par)) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_f16_tmem_a(tm + TC_S, tm + TC_AVP + 8 * kk,
                                           tc::sw128_mn_desc(base + BL_KT + 2048u * kk, 8192u), id_s, 1u);
                    tc::mma_commit(smem_u32(&ss.m2));
                } else if (role == 2) {
                    // Y = Q~ S, then Y += P Vnew once Vnew is in
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        tc::mma_f16_tmem_a(tm + TC_Y, s16 + 8 * kk,
                                           tc::sw128_desc(base + BL_QT + (kk >> 2) * 8192 + (kk & 3) * 32), id_y,
                                           kk > 0 ? 1u : 0u);
                    if (!wait(ss.vn, par)) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc::mma_f16_tmem_a(tm + TC_Y, tm + TC_AVP + 8 * kk,
                                           tc::kmajor_desc<2>(base + BL_P, 16 * kk, CH), id_y, 1u);
                    tc::mma_commit(smem_u32(&ss.y));
                }
                tc::mma_commit(smem_u32(&ss.free_[st]));
            }
            // every MMA this issuer started has finished before the tensor memory is freed
            tc::mma_commit(smem_u32(&ss.done[role]));
        }
    } else if (warp < 8) {
        // ---------------------------------------------------------- chain epilogues
        const int q = warp & 3, hh = warp >> 2;
        const int j = 32 * q + lane;
        const uint32_t lq = (uint32_t)(32 * q) << 16;
        // initial state block: row j, keys [64 hh, 64 hh + 64)
        {
            float s[2][32];
#pragma unroll
            for (int p = 0; p < 2; ++p)
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const float4 v = S_src ? *reinterpret_cast<const float4 *>(S_src + (size_t)j * DK + 64 * hh + 32 * p + e)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    s[p][e] = v.x; s[p][e + 1] = v.y; s[p][e + 2] = v.z; s[p][e + 3] = v.w;
                }
            const float g0 = gamma_n(0);
#pragma unroll
            for (int p = 0; p < 2; ++p) {
                uint32_t wd[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) wd[e] = tc::pack_half2(s[p][2 * e], s[p][2 * e + 1]);
                tc::tmem_st16_u32(tm + lq + s16_of(0) + 32 * hh + 16 * p, wd);
#pragma unroll
                for (int e = 0; e < 32; ++e) s[p][e] *= g0;
                tc::tmem_st32(tm + lq + TC_S + 64 * hh + 32 * p, s[p]);
            }
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) { mbar_arrive(smem_u32(&ss.s16)); mbar_arrive(smem_u32(&ss.dec)); }
        }
        for (int c = 0; c < nc; ++c) {
            const int st = c & 1;
            const uint32_t par = (uint32_t)(c & 1), spar = (uint32_t)((c >> 1) & 1);
            const unsigned char *stg = sm + st * STAGE_BYTES + ST_BLOB;
            const float g_next = c + 1 < nc ? gamma_n(c + 1) : 0.0f;
            // ---- E1: Vnew^T for tokens [32 hh, 32 hh + 32). Tokens past the chunk need
            //      no mask: their rows of U and W are zero, so Vnew is zero there.
            if (!wait(ss.full[st], spar) || !wait(ss.m1a, par) || !wait(ss.m1b, par)) break;
            tc::fence_after_sync();
            {
                uint32_t wp[16];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int tq = 32 * hh + 16 * hf;  // first token of this half
                    float va[16], vb[16];
                    tc::tmem_ld16(tm + lq + TC_WSA + tq, va);
                    tc::tmem_ld16(tm + lq + TC_WSB + tq, vb);
                    uint4 u4[2];
#pragma unroll
                    for (int g8 = 0; g8 < 2; ++g8)
                        u4[g8] = *reinterpret_cast<const uint4 *>(stg + BL_UT + mn_off(tq + 8 * g8, j));
                    tc::wait_ld();
#pragma unroll
                    for (int g8 = 0; g8 < 2; ++g8) {
                        const uint32_t uu[4] = {u4[g8].x, u4[g8].y, u4[g8].z, u4[g8].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 u2 = __half22float2(*reinterpret_cast<const __half2 *>(&uu[e]));
                            const int t = 8 * g8 + 2 * e;
                            wp[8 * hf + 4 * g8 + e] = tc::pack_half2(u2.x - (va[t] + vb[t]), u2.y - (va[t + 1] + vb[t + 1]));
                        }
                    }
                }
                // the previous chunk's Y has read the copy this overwrites (its state
                // update too: the previous E2 waited for it)
                if (c > 0 && !wait(ss.y, (uint32_t)((c - 1) & 1))) break;
                tc::fence_after_sync();
                tc::tmem_st16_u32(tm + lq + TC_AVP + 16 * hh, wp);
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) { mbar_arrive(smem_u32(&ss.vn)); mbar_arrive(smem_u32(&ss.free_[st])); }
            }
            // ---- E2: the updated state block (keys [64 hh, 64 hh + 64)), 32 keys at a
            //      time, into the other fp16 buffer (whose last reader, the previous
            //      chunk's Y, completed before E1 above), then the decay
            if (!wait(ss.m2, par)) break;
            tc::fence_after_sync();
            if (c + 1 < nc) {
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    float sv[32];
                    tc::tmem_ld32(tm + lq + TC_S + 64 * hh + 32 * p, sv);
                    tc::wait_ld();
                    uint32_t wd[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) wd[e] = tc::pack_half2(sv[2 * e], sv[2 * e + 1]);
                    tc::tmem_st16_u32(tm + lq + s16_of(c + 1) + 32 * hh + 16 * p, wd);
                }
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ss.s16));
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    float sv[32];
                    tc::tmem_ld32(tm + lq + TC_S + 64 * hh + 32 * p, sv);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) sv[e] *= g_next;
                    tc::tmem_st32(tm + lq + TC_S + 64 * hh + 32 * p, sv);
                }
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&ss.dec));
            } else if (S_dst) {
                float *d = S_dst + (size_t)j * DK + 64 * hh;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    float sv[32];
                    tc::tmem_ld32(tm + lq + TC_S + 64 * hh + 32 * p, sv);
                    tc::wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4 *>(d + 32 * p + e) = make_float4(sv[e], sv[e + 1], sv[e + 2], sv[e + 3]);
                }
            }
        }
    } else {
        // ---------------------------------------------------------- output: y to the buffer
        // Warps 8-11 (lane quarter w % 4): y = scale Y of column j for the
        // chunk's 64 tokens, stored as fp16; a warp's store for one token covers
        // 32 consecutive columns (64 bytes). The gated RMSNorm . silu(z) across
        // each head's 128 columns runs on other SMs: in the one-kernel form on the
        // CTAs past their prep items, which wait for a flag per (chunk, V-head),
        // else as its own kernel.
        const int q = warp & 3;
        const int j = 32 * q + lane;
        const uint32_t lq = (uint32_t)(32 * q) << 16;
        const float scale = rsqrtf((float)DK);
        for (int c = 0; c < nc; ++c) {
            const uint32_t par = (uint32_t)(c & 1);
            const int nv = nv_of(c);
            const bool ok = wait(ss.y, par);
            if (bar_red_or(1, 128, !ok)) break;        // the four warps leave together
            tc::fence_after_sync();
            float y[2][32];
            tc::tmem_ld32(tm + lq + TC_Y, y[0]);
            tc::tmem_ld32(tm + lq + TC_Y + 32, y[1]);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ss.yfree));
            // one kernel form: the previous chunk's y of this head is complete (the
            // barrier above follows the four warps' stores of it). One thread
            // releases its flag, after Y is handed back, so that the release's
            // fence stays off the chain; a chunk late, so that it finds those
            // stores long done.
            if (a.yflags && c > 0 && warp == 8 && lane == 0)
                asm volatile("st.release.gpu.global.s32 [%0], %1;"
                             ::"l"(a.yflags + (size_t)(fr.chunk0 + c - 1) * HV + vh), "r"(1) : "memory");
            __half *yr = a.ybuf + (size_t)(fr.row_a + CH * c - a.w0) * DI + (size_t)vh * DV + j;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int t = 0; t < 32; ++t)
                    if (32 * hh + t < nv) yr[(size_t)(32 * hh + t) * DI] = __float2half_rn(scale * y[hh][t]);
            if (a.yflags && c == nc - 1) {             // the last chunk's y
                bar_named(2, 128);
                if (warp == 8 && lane == 0)
                    asm volatile("st.release.gpu.global.s32 [%0], %1;"
                                 ::"l"(a.yflags + (size_t)(fr.chunk0 + c) * HV + vh), "r"(1) : "memory");
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp >= CA_ISSUER0 && lane == 0) mbar_wait_sleep(smem_u32(&ss.done[warp - CA_ISSUER0]), 0u);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tm, TC_COLS);
    const bool gave_up = aborted;
    if (tid == 0 && gave_up) atomicExch(&g_chunk_error, (unsigned int)GDN_ERR_TIMEOUT);
    if (again && !gave_up && tid == 0)                 // every wait on them has ended (the barrier above)
        for (int k = 0; k < CA_NBAR; ++k) mbar_inval(smem_u32(reinterpret_cast<uint64_t *>(&ss) + k));
    return gave_up;
}

__global__ void __launch_bounds__(CA_THREADS, 1) wy_carry_kernel(const WyArgs a)
{
    wy_carry_body(a, (int)blockIdx.x, (int)blockIdx.y, false);
}

// Norm items of the one-kernel form: the gated RMSNorm . silu(z) of section
// "Output path", out = y (mean_j y^2 + eps)^-1/2 w_j silu(z) per token and
// V-head, over items (chunk, 2 V-heads) handed out in chunk order from a
// counter, so that a CTA past its prep items takes the next item whose y is
// (about to be) written. Warp 0 runs an item ahead: it takes a ticket, waits
// (bounded, with a back-off that keeps the polling off the chains' way) for the
// item's two y flags, and brings the item's y and z rows (64 x 256 columns each)
// into one of two shared-memory buffers by TMA; plain loads would have to stage
// through the little L1 that the kernel's shared memory leaves. Warps 1-15
// normalise the item in the other buffer meanwhile, one (row, head) unit at a
// time with the unit's loads issued first; lane l holds columns 4l..4l+3 of the
// head, so the head's sum of squares is a warp sum. The two sides meet only
// through mbarriers (bounded waits), never a CTA-wide barrier.
constexpr int NI_HEADS = 2;
constexpr uint32_t NI_TILE = CH * NI_HEADS * DV * 2;        // 32 KiB: 64 rows x 256 columns
constexpr uint32_t NI_BUF = 2 * NI_TILE;                    // y, then z
constexpr uint32_t NI_BAR = 2 * NI_BUF;                     // full[2], used[2], the items of the buffers
static_assert(NI_BAR + 64 <= PR_SMALL, "the norm buffers fit below the prep block's mbarriers");
constexpr int NI_WORKERS = PR_THREADS / 32 - 1;             // warps 1-15
constexpr int NI_UNITS = CH * NI_HEADS;                     // (row, head) units of an item
constexpr int NI_PER_WARP = (NI_UNITS + NI_WORKERS - 1) / NI_WORKERS;
template <typename TO>
__device__ void wy_norm_items(const CUtensorMap &ymap, const CUtensorMap &zmap, const WyArgs &a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = smem_aligned1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + NI_BAR);     // [2]: the buffer's copies landed
    uint64_t *used = full + 2;                                       // [2]: the workers are done with it
    int *item_of = reinterpret_cast<int *>(full + 4);                // [2]: its item, -1 to end
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_items = a.count->n_chunks * (HV / NI_HEADS);
    if (tid == 0) {
        for (int k = 0; k < 2; ++k) {
            mbar_init(smem_u32(&full[k]), 1);
            mbar_init(smem_u32(&used[k]), NI_WORKERS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 0) {
        // ---------------------------------------------------------- the item ahead
        for (int n = 0;; ++n) {
            const int buf = n & 1;
            bool ok = true;
            if (n >= 2 && lane == 0)                  // the workers are done with item n - 2
                ok = mbar_wait_sleep(smem_u32(&used[buf]), (uint32_t)(((n >> 1) - 1) & 1));
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            int item = -1;
            if (ok) {
                int t = 0;
                if (lane == 0) t = atomicAdd(&a.count->norm_next, 1);
                item = __shfl_sync(0xffffffffu, t, 0);
                if (item >= n_items) item = -1;
            }
            if (item >= 0) {
                const int g = item / (HV / NI_HEADS), h0 = NI_HEADS * (item % (HV / NI_HEADS));
                bool ready = true;
                if (lane < NI_HEADS) {                // one y flag per lane
                    const int *fl = a.yflags + (size_t)g * HV + h0 + lane;
                    const uint64_t t0 = global_timer_ns();
                    for (;;) {
                        int v;
                        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(fl) : "memory");
                        if (v) break;
                        if (global_timer_ns() - t0 > WAIT_LIMIT_NS) { ready = false; break; }
                        __nanosleep(500);
                    }
                }
                if (!__all_sync(0xffffffffu, ready)) {
                    ok = false;
                    item = -1;
                } else if (lane == 0) {
                    // the copies (async proxy) after the flags and after this CTA's
                    // earlier generic accesses of the same shared memory
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    const WyChunk ck = a.chunks[g];
                    item_of[buf] = item;
                    const uint32_t bar = smem_u32(&full[buf]);
                    mbar_arrive_expect_tx(bar, NI_BUF);
                    tma_load_2d(sb + buf * NI_BUF, &ymap, h0 * DV, ck.row0 - a.w0, bar);
                    tma_load_2d(sb + buf * NI_BUF + NI_TILE, &zmap, h0 * DV, ck.row0, bar);
                }
            }
            if (item < 0) {                           // the end (or a wait that gave up)
                if (lane == 0) {
                    if (!ok) atomicExch(&g_chunk_error, (unsigned int)GDN_ERR_TIMEOUT);
                    item_of[buf] = -1;
                    mbar_arrive(smem_u32(&full[buf]));
                }
                break;
            }
        }
    } else {
        // ---------------------------------------------------------- the workers
        const bool has_w = a.norm_w != nullptr;
        const float4 w = has_w ? __ldg(reinterpret_cast<const float4 *>(a.norm_w) + lane) : make_float4(1.f, 1.f, 1.f, 1.f);
        for (int n = 0;; ++n) {
            const int buf = n & 1;
            if (!mbar_wait_sleep(smem_u32(&full[buf]), (uint32_t)((n >> 1) & 1))) {
                if (lane == 0) atomicExch(&g_chunk_error, (unsigned int)GDN_ERR_TIMEOUT);
                break;
            }
            const int item = item_of[buf];
            if (item < 0) break;
            const int g = item / (HV / NI_HEADS), h0 = NI_HEADS * (item % (HV / NI_HEADS));
            const WyChunk ck = a.chunks[g];
            const unsigned char *yt = sm + buf * NI_BUF, *zt = yt + NI_TILE;
            uint2 yv[NI_PER_WARP], zv[NI_PER_WARP];
#pragma unroll
            for (int k = 0; k < NI_PER_WARP; ++k) {
                const int u = (warp - 1) + NI_WORKERS * k;
                const uint32_t off = (uint32_t)(u >> 1) * (NI_HEADS * DV * 2) + (uint32_t)((u & 1) * DV + 4 * lane) * 2u;
                if (u < NI_UNITS) {
                    yv[k] = *reinterpret_cast<const uint2 *>(yt + off);
                    zv[k] = *reinterpret_cast<const uint2 *>(zt + off);
                }
            }
#pragma unroll
            for (int k = 0; k < NI_PER_WARP; ++k) {
                const int u = (warp - 1) + NI_WORKERS * k, r = u >> 1, hh = u & 1;
                if (u >= NI_UNITS || r >= ck.nv) continue;   // uniform over the warp
                const float2 y01 = __half22float2(*reinterpret_cast<const __half2 *>(&yv[k].x));
                const float2 y23 = __half22float2(*reinterpret_cast<const __half2 *>(&yv[k].y));
                float o0 = y01.x, o1 = y01.y, o2 = y23.x, o3 = y23.y;
                if (has_w) {
                    const float ms = warp_sum(o0 * o0 + o1 * o1 + o2 * o2 + o3 * o3) * (1.0f / DV);
                    const float rs = rsqrtf(ms + a.norm_eps);
                    o0 *= rs * w.x * silu_gate(__uint_as_float(zv[k].x << 16));
                    o1 *= rs * w.y * silu_gate(__uint_as_float(zv[k].x & 0xFFFF0000u));
                    o2 *= rs * w.z * silu_gate(__uint_as_float(zv[k].y << 16));
                    o3 *= rs * w.w * silu_gate(__uint_as_float(zv[k].y & 0xFFFF0000u));
                }
                store_out4<TO>(static_cast<TO *>(a.out) + (size_t)(ck.row0 + r) * DI + (size_t)(h0 + hh) * DV + 4 * lane,
                               o0, o1, o2, o3);
            }
            __syncwarp();                             // the warp's reads of the buffer are done
            if (lane == 0) mbar_arrive(smem_u32(&used[buf]));
        }
    }
}

// One kernel for prep and the chains of a window. The first 32 G CTAs run the
// chains, G = min(fragments, FU_GROUPS): CTA b takes V-head b % 32 of fragments
// b / 32, b / 32 + G, .. one after the other; the other CTAs run the prep items
// in chunk order. A chain takes a chunk's operands as soon as the prep CTA of
// that (chunk, K-head) has flagged it, so prep and chains run side by side on
// separate SMs. Launched cooperatively (every CTA resident at once): the chain
// CTAs wait on flags the prep CTAs set, never the other way round.
constexpr int FU_GROUPS = 2;
static_assert(PR_THREADS == CA_THREADS, "one block size for both roles");
__global__ void __launch_bounds__(PR_THREADS, 1) wy_fused_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                const __grid_constant__ CUtensorMap ymap,
                                                                const __grid_constant__ CUtensorMap zmap,
                                                                const WyArgs a)
{
    const int n_frag = a.count->n_frag;                // the plan kernel ahead has completed
    const int groups = max(1, min(n_frag, FU_GROUPS));
    const int nca = groups * HV, b = (int)blockIdx.x;
    if (b < nca) {
        for (int f = b / HV; f < n_frag; f += groups)
            if (wy_carry_body(a, f, b % HV, true)) break;
    } else {
        wy_prep_body(xmap, a, b - nca, (int)gridDim.x - nca);
        // then the gated norm of the chunks whose y the chains have written
        __syncthreads();                               // every prep access of the shared memory is done
        if (a.out_f32) wy_norm_items<float>(ymap, zmap, a);
        else wy_norm_items<bf16>(ymap, zmap, a);
    }
}

// The gated RMSNorm . silu(z) of section "Output path" over the window's rows:
// out = y (mean_j y^2 + eps)^-1/2 w_j silu(z), per token and V-head over the
// head's 128 columns. One warp per (token, four V-heads); lane l holds columns
// 4l..4l+3 of a head, so the head's sum of squares is a warp sum and every
// access is a vector of 4.
template <typename TO>
__global__ void __launch_bounds__(256) wy_norm_kernel(const WyArgs a)
{
    grid_dep_wait();                                   // y comes from the carry kernel
    grid_dep_launch();
    const int row = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (row >= a.wlen) return;
    const size_t g = (size_t)(a.w0 + row);
    if (a.norm_w == nullptr) {                         // no norm weights: out is y itself
#pragma unroll
        for (int hh = 0; hh < HV / 8; ++hh) {
            const int vh = warp * (HV / 8) + hh;
            const uint2 yv = *reinterpret_cast<const uint2 *>(a.ybuf + (size_t)row * DI + (size_t)vh * DV + 4 * lane);
            const float2 y01 = __half22float2(*reinterpret_cast<const __half2 *>(&yv.x));
            const float2 y23 = __half22float2(*reinterpret_cast<const __half2 *>(&yv.y));
            store_out4<TO>(static_cast<TO *>(a.out) + g * DI + (size_t)vh * DV + 4 * lane, y01.x, y01.y, y23.x, y23.y);
        }
        return;
    }
    const float4 w = __ldg(reinterpret_cast<const float4 *>(a.norm_w) + lane);
#pragma unroll
    for (int hh = 0; hh < HV / 8; ++hh) {
        const int vh = warp * (HV / 8) + hh;
        const uint2 yv = *reinterpret_cast<const uint2 *>(a.ybuf + (size_t)row * DI + (size_t)vh * DV + 4 * lane);
        const float2 y01 = __half22float2(*reinterpret_cast<const __half2 *>(&yv.x));
        const float2 y23 = __half22float2(*reinterpret_cast<const __half2 *>(&yv.y));
        const float4 zz = load4(a.z + g * DI + (size_t)vh * DV + 4 * lane);
        const float ms = warp_sum(y01.x * y01.x + y01.y * y01.y + y23.x * y23.x + y23.y * y23.y) * (1.0f / DV);
        const float r = rsqrtf(ms + a.norm_eps);
        store_out4<TO>(static_cast<TO *>(a.out) + g * DI + (size_t)vh * DV + 4 * lane, y01.x * r * w.x * silu_gate(zz.x),
                       y01.y * r * w.y * silu_gate(zz.y), y23.x * r * w.z * silu_gate(zz.z),
                       y23.y * r * w.w * silu_gate(zz.w));
    }
}

// Sequences with no tokens: their SSM state passes through (zeros without an
// input state). One CTA per (sequence, V-head).
__global__ void __launch_bounds__(256) wy_passthrough_kernel(const int32_t *__restrict__ cu, int T_total,
                                                            const float *S_in, float *S_out)
{
    const int n = blockIdx.x, vh = blockIdx.y;
    grid_dep_wait();
    const int s0 = cu_clamp(cu, n, 0, T_total), s1 = cu_clamp(cu, n + 1, s0, T_total);
    if (s1 > s0 || S_out == nullptr || S_out == S_in) return;
    const size_t base = ((size_t)n * HV + vh) * (DV * DK) / 4;
    for (int e = threadIdx.x; e < DV * DK / 4; e += blockDim.x)
        reinterpret_cast<float4 *>(S_out)[base + e] =
            S_in ? reinterpret_cast<const float4 *>(S_in)[base + e] : make_float4(0.f, 0.f, 0.f, 0.f);
}

// ---------------------------------------------------------------- launcher

cudaError_t launch_conv_state_out_bf16(const int32_t *cu, int N, int T_total, const void *qkv, const void *cs_in,
                                       void *cs_out, cudaStream_t s, bool pdl);
int sm_count();

static size_t rnd256(size_t x) { return (x + 255) & ~(size_t)255; }
static size_t rnd1024(size_t x) { return (x + 1023) & ~(size_t)1023; }

struct WyLayout {
    size_t count, frags, chunks, flags, yflags, gates, xhat, ybuf, blobs, slots, total;
    int W, f_cap, c_cap;
};

// Workspace of the chunked path for windows of W tokens (W a multiple of 64):
// counts | fragments | chunks | prep flags [c_cap][16] | y flags [c_cap][32] | gate records [c_cap][32] |
// x^ [W][8192] fp16 | y [W][4096] fp16 |
// blobs [c_cap][32] | two state slots.
static WyLayout wy_layout(int N, int W)
{
    WyLayout L;
    L.W = W;
    L.f_cap = std::max(1, std::min(N, W));
    L.c_cap = W / CH + L.f_cap;
    size_t o = 0;
    L.count = o;  o = rnd256(o + sizeof(WyCount));
    L.frags = o;  o = rnd256(o + (size_t)L.f_cap * sizeof(WyFrag));
    L.chunks = o; o = rnd256(o + (size_t)L.c_cap * sizeof(WyChunk));
    L.flags = o;  o = rnd256(o + (size_t)L.c_cap * HK * sizeof(int));
    L.yflags = o; o = rnd1024(o + (size_t)L.c_cap * HV * sizeof(int));
    L.gates = o;  o = rnd1024(o + (size_t)L.c_cap * HV * GATE_FLOATS * sizeof(float));
    L.xhat = o;   o = rnd1024(o + (size_t)W * CC * sizeof(__half));
    L.ybuf = o;   o = rnd1024(o + (size_t)W * DI * sizeof(__half));
    L.blobs = o;  o = rnd1024(o + (size_t)L.c_cap * HV * BLOB_BYTES);
    L.slots = o;  o += 2 * (size_t)HV * DV * DK * sizeof(float);
    L.total = o;
    return L;
}

// The window the library sizes its workspace for by default: one window up to
// this many tokens; a longer prompt runs as several.
constexpr int WY_DEFAULT_WINDOW = 4096;

size_t chunk_workspace_bytes(int N, int T_total)
{
    const int W = std::max(CH, std::min(WY_DEFAULT_WINDOW, (T_total + CH - 1) / CH * CH));
    return wy_layout(N, W).total;
}

// The smallest workspace the chunked path runs in: windows of one chunk.
size_t chunk_min_workspace_bytes(int N) { return wy_layout(N, CH).total; }

// The largest window (a multiple of 64 tokens, at most the prompt rounded up)
// whose layout fits in ws_bytes; 0 if not even one chunk fits.
static int wy_window(int N, int T_total, size_t ws_bytes)
{
    if (wy_layout(N, CH).total > ws_bytes) return 0;
    int lo = 1, hi = std::max(1, (T_total + CH - 1) / CH);   // in chunks
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (wy_layout(N, mid * CH).total <= ws_bytes) lo = mid;
        else hi = mid - 1;
    }
    return lo * CH;
}

// GDN_PREFILL_SPLIT=1 in the environment keeps prep and the chains in two
// kernels (for a device share too small for a one-per-SM cooperative grid).
static bool prefill_split_forced()
{
    static const bool forced = [] {
        const char *v = std::getenv("GDN_PREFILL_SPLIT");
        return v != nullptr && v[0] == '1';
    }();
    return forced;
}

static cudaError_t wy_setup()
{
    cudaError_t e = cudaFuncSetAttribute(wy_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PR_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(wy_carry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CA_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(wy_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)std::max(PR_SMEM, CA_SMEM));
    return e;
}

cudaError_t launch_prefill_chunked(const gdn_params *p, const void *qkv, const void *z, const void *alpha,
                                   const void *beta, const int32_t *cu, int N, int T_total, const void *cs_in,
                                   void *cs_out, const float *S_in, float *S_out, void *out, gdn_dtype out_dt,
                                   void *ws_body, size_t ws_bytes, cudaStream_t s, const void *xhat_ext)
{
    cudaError_t e = wy_setup();
    if (e != cudaSuccess) return e;
    const int n_sm = sm_count();
    if (n_sm <= 0) return cudaErrorInvalidDevice;
    if (T_total > 0) {
        const int W = wy_window(N, T_total, ws_bytes);
        if (W <= 0) return cudaErrorInvalidValue;      // the caller checked the minimum
        const WyLayout L = wy_layout(N, W);
        unsigned char *ws = static_cast<unsigned char *>(ws_body);
        WyArgs a;
        a.conv_w = p->conv_w; a.A_log = p->A_log; a.dt_bias = p->dt_bias; a.norm_w = p->norm_w;
        a.norm_eps = p->norm_eps; a.l2_eps = p->l2_eps;
        a.qkv = (const bf16 *)qkv; a.z = (const bf16 *)z; a.alpha = (const bf16 *)alpha; a.beta = (const bf16 *)beta;
        a.cu = cu; a.N = N; a.T_total = T_total;
        a.cs_in = (const bf16 *)cs_in; a.S_in = S_in; a.S_out = S_out; a.out = out;
        a.f_cap = L.f_cap; a.c_cap = L.c_cap;
        a.count = reinterpret_cast<WyCount *>(ws + L.count);
        a.frags = reinterpret_cast<WyFrag *>(ws + L.frags);
        a.chunks = reinterpret_cast<WyChunk *>(ws + L.chunks);
        // the one-kernel form when every CTA of a one-per-SM grid can be resident
        // at once (a cooperative launch), else the prep and carry kernels apart
        int coop = 0, per_sm = 0, dev = 0;
        bool fused = n_sm > FU_GROUPS * HV && !prefill_split_forced();
        if (fused)
            fused = cudaGetDevice(&dev) == cudaSuccess &&
                    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, wy_fused_kernel, PR_THREADS,
                                                                  std::max(PR_SMEM, CA_SMEM)) == cudaSuccess &&
                    per_sm >= 1;
        cudaGetLastError();                            // a refused query only means: separate kernels
        a.flags = fused ? reinterpret_cast<int *>(ws + L.flags) : nullptr;
        a.yflags = fused ? reinterpret_cast<int *>(ws + L.yflags) : nullptr;
        a.out_f32 = out_dt == GDN_F32;
        a.gates = reinterpret_cast<float *>(ws + L.gates);
        a.xhat = reinterpret_cast<__half *>(ws + L.xhat);
        a.gates_only = xhat_ext != nullptr;
        a.ybuf = reinterpret_cast<__half *>(ws + L.ybuf);
        a.blobs = ws + L.blobs;
        float *slots = reinterpret_cast<float *>(ws + L.slots);
        CUtensorMap ymap, zmap;                        // y of the window and z, in boxes of 64 rows x 256 columns
        if (fused && (!make_bf16_plain_map(&ymap, a.ybuf, W, DI, 256, CH) ||
                      !make_bf16_plain_map(&zmap, z, T_total, DI, 256, CH)))
            return cudaErrorInvalidValue;
        int wi = 0;
        for (int w0 = 0; w0 < T_total && e == cudaSuccess; w0 += W, ++wi) {
            a.w0 = w0;
            a.wlen = std::min(W, T_total - w0);
            a.slot_in = slots + (size_t)((wi + 1) & 1) * HV * DV * DK;
            a.slot_out = slots + (size_t)(wi & 1) * HV * DV * DK;
            CUtensorMap xmap;                          // x^ rows of this window; rows past it read as zero
            const void *xrows = xhat_ext ? static_cast<const void *>(static_cast<const __half *>(xhat_ext) +
                                                                     (size_t)w0 * CC)
                                         : static_cast<const void *>(a.xhat);
            if (!make_bf16_sw128_map(&xmap, xrows, a.wlen, CC, CH)) return cudaErrorInvalidValue;
            // Each kernel is launched with programmatic stream serialization and waits
            // (grid_dep_wait) before it touches what the kernel ahead writes.
            e = launch_pdl(wy_plan_kernel, dim3(1), dim3(1024), 0, s, a);
            if (e == cudaSuccess)
                e = launch_pdl(wy_act_kernel, dim3((unsigned)L.c_cap, xhat_ext ? HK : CC / DK), dim3(ACT_THREADS), 0,
                               s, a);
            if (fused) {
                // prep and the chains in one cooperative grid, one CTA per SM
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3((unsigned)n_sm);
                cfg.blockDim = dim3(PR_THREADS);
                cfg.dynamicSmemBytes = std::max(PR_SMEM, CA_SMEM);
                cfg.stream = s;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeCooperative;
                attr[0].val.cooperative = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, wy_fused_kernel, xmap, ymap, zmap, a);
            } else {
                if (e == cudaSuccess)
                    e = launch_pdl(wy_prep_kernel, dim3((unsigned)std::min(L.c_cap * HK, n_sm)), dim3(PR_THREADS),
                                   PR_SMEM, s, xmap, a);
                if (e == cudaSuccess)
                    e = launch_pdl(wy_carry_kernel, dim3((unsigned)L.f_cap, HV), dim3(CA_THREADS), CA_SMEM, s, a);
            }
            if (e == cudaSuccess && !fused) {
                if (out_dt == GDN_F32)
                    e = launch_pdl(wy_norm_kernel<float>, dim3((unsigned)a.wlen), dim3(256), 0, s, a);
                else
                    e = launch_pdl(wy_norm_kernel<bf16>, dim3((unsigned)a.wlen), dim3(256), 0, s, a);
            }
        }
    }
    if (e == cudaSuccess && N > 0)
        e = launch_pdl(wy_passthrough_kernel, dim3((unsigned)N, HV), dim3(256), 0, s, cu, T_total, S_in, S_out);
    if (e == cudaSuccess && cs_out) e = launch_conv_state_out_bf16(cu, N, T_total, qkv, cs_in, cs_out, s, true);
    return e;
}

// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *chunk_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_chunk_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
