// gdn_attn.cu -- decode attention of the full-attention layers on 5th-generation
// tensor cores: one new token per sequence attends over its bf16 KV cache, and
// the output gate follows. These are steps 5-6 of section "Full-attention
// block" of "qwen35moe -- Forward-Pass Design (Pantheon port)": GQA attention
// with 16 query heads and 2 KV heads of head_dim 256, scale 1/sqrt(head_dim),
// then cur = attn_out * sigmoid(z). The query arrives after its RMSNorm and
// partial RoPE (steps 2-4), and the cache holds keys after theirs.
//
// Decode attention is bound by reading the cache: 1 KiB of keys and values per
// cached position and KV head. Two ideas from the pages' attention section
// ("Read the attention cache efficiently") carry over:
//  - GQA packing: the 8 query heads that share a KV head are served by one CTA,
//    which reads each key and value row once for all 8;
//  - fixed blocks: the context is cut into blocks of 128 * tps positions that
//    CTAs process in parallel, and the blocks' partial softmax sums are merged
//    at the end. Long contexts and small batches still fill the GPU.
//
// Per CTA = (sequence b, KV head g, block s), tiles of 128 positions:
//  - warp 0, lane 0, TMA producer: per tile, four 32 KiB copies (keys dims
//    0-127, keys 128-255, values 0-127, values 128-255), each two boxes of 64
//    dims x 128 positions in the 128-byte swizzle, through a ring of 3 slots;
//  - warp 1, lane 0, MMA issuer:
//      S^T[pos][head] = K Q^T   (M = 128 positions, N = 16, K = 256 dims),
//      O^T[dim][head] = V^T P^T (M = 128 dims x 2, N = 16, K = 128 positions),
//    with Q^T and P^T as 16-row B operands whose rows 8..15 are don't-care:
//    their accumulator columns are never read. V^T is the cache tile read
//    MN-major, so no transpose is ever stored;
//  - warps 2..5 (128 threads): the online softmax. For scores, thread r holds
//    position r's 8 scores (its TMEM lane); the tile maximum per head crosses
//    the 4 warps through shared memory; p = 2^(s log2 e - m) is rounded to bf16
//    and stored as the P^T operand. For outputs, thread r holds dims r and
//    128 + r of all 8 heads and rescales its running sums by the factor
//    2^(m_old - m_new) before adding the tile's O^T.
// A context that fits one block is finished in place: o = acc / sum, times
// sigmoid(z). Otherwise each block stores its unnormalised output, maximum and
// sum in the workspace, and a combine kernel (one warp per sequence and query
// head) merges them. Merging inside the last block to
// finish was measured slower: its dependent L2 round trips hold an SM slot that
// streaming blocks need. Positions at or past the context
// length are masked (their scores), and their value rows in shared memory are
// zeroed, so nothing stored past ctx_len can reach the output. An empty context
// gives zeros. The TMA producer starts as soon as the barriers exist; the Q
// operand and the TMEM allocation are ready before the first MMA.
//
// Every mbarrier wait is bounded; a wait that gives up records GDN_ERR_TIMEOUT.
#include <cuda.h>

#include <mutex>

#include "gdn_async.cuh"
#include "gdn_common.cuh"
#include "gdn_tc.cuh"
#include "gdn_tma.cuh"

namespace gdn {

__device__ unsigned int g_attn_error;   // GDN_ERR_TIMEOUT if a bounded wait gave up

constexpr int AT_HQ = GDN_ATTN_Q_HEADS;           // 16
constexpr int AT_HKV = GDN_ATTN_KV_HEADS;         // 2
constexpr int AT_D = GDN_ATTN_HEAD_DIM;           // 256
constexpr int AT_G = AT_HQ / AT_HKV;              // 8 query heads per KV head
constexpr int AT_TILE = 128;                      // positions per tile (the first product's M)
constexpr int AT_SLOTS = 3;
constexpr uint32_t AT_BOX = AT_TILE * 128;        // one TMA box: 128 rows x 128 bytes = 16 KiB
constexpr uint32_t AT_SLOT_BYTES = 2 * AT_BOX;    // 128 dims of one tile = 32 KiB
constexpr int AT_THREADS = 192;                   // TMA warp, MMA warp, 4 softmax warps
constexpr int AT_TPS_MAX = 8;                     // tiles per block, at most
constexpr uint32_t AT_TMEM_COLS = 128;
constexpr uint32_t TC_D2 = 0;                     // O^T: 2 buffers x (2 halves x 16 columns)
constexpr uint32_t TC_D1 = 64;                    // S^T: 16 columns
static_assert(AT_D == 256 && AT_G == 8, "one CTA serves the 8 query heads of a KV head");

// Shared-memory layout from a 1024-byte aligned base. The 16-row B operands are
// stored as 8-row atoms 1 KiB apart; the descriptors' 8-row-group stride (SBO)
// of 1 KiB makes rows 8..15 of each atom read the next KiB, which only feeds
// accumulator columns 8..15. The overhang of the last atom lands inside the ring.
constexpr uint32_t SA_Q = 0;                      // Q^T: 4 atoms (64 dims each) x 8 heads x 128 B
constexpr uint32_t SA_P = 4096;                   // P^T: 2 buffers x 2 atoms (64 positions each)
constexpr uint32_t SA_RING = 8192;                // 3 slots x 32 KiB
constexpr uint32_t SA_SMALL = SA_RING + AT_SLOTS * AT_SLOT_BYTES;

struct AttnSmall {
    uint64_t full[AT_SLOTS], empty[AT_SLOTS];
    uint64_t d1_full, p_full[2], d2_full[2], done;
    uint32_t tmem;
    int abort;
    float red[2][4][AT_G];                        // per-warp tile maxima, double-buffered by tile
    float lred[4][AT_G];                          // per-warp softmax sums
};
constexpr size_t AT_SMEM = SA_SMALL + sizeof(AttnSmall) + 1024;   // + slack to align the block

template <typename TO>
struct AttnArgs {
    const bf16 *q;            // [B][16][256]
    const bf16 *z;            // [B][16][256]
    const int32_t *ctx_len;   // [B]
    TO *out;                  // [B][16][256]
    float *part_o;            // [items][8][256]: unnormalised block outputs
    float *part_ml;           // [items][8][2]: block maximum (log2 units), block sum
    int Lmax, S, tps;         // cache rows per (sequence, KV head), blocks per (b, g), tiles per block
};

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// Barrier over the 128 softmax threads (named barrier 1) that also returns the
// AND of `p` over them, so that every thread takes the same branch after it.
__device__ __forceinline__ bool softmax_bar_and(bool p)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred a, b;\n\tsetp.ne.u32 a, %1, 0;\n\t"
                 "bar.red.and.pred b, 1, 128, a;\n\tselp.u32 %0, 1, 0, b;\n\t}"
                 : "=r"(r) : "r"((uint32_t)p) : "memory");
    return r != 0;
}
__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// MN-major operand in the 128-byte swizzle: atoms of 64 elements along M x 8
// rows along K, as a TMA box 64 elements wide writes them. LBO = distance of the
// next 64 elements along M (the next box), SBO = distance of the next 8 rows
// along K (1 KiB).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo)
{
    return tc::smem_desc(saddr, lbo, 1024u) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }

template <typename TO>
__global__ void __launch_bounds__(AT_THREADS, 2) attn_block_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                   const __grid_constant__ CUtensorMap vmap,
                                                                   const AttnArgs<TO> a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *blk = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    AttnSmall &ss = *reinterpret_cast<AttnSmall *>(blk + SA_SMALL);
    const uint32_t sb = smem_u32(blk);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int item = blockIdx.x;
    const int sp = item % a.S, bg = item / a.S, b = bg / AT_HKV, g = bg % AT_HKV;
    grid_dep_wait();                                   // q, the cache and ctx_len may come from the kernel ahead
    grid_dep_launch();
    const int L = min(max(__ldg(a.ctx_len + b), 0), a.Lmax);
    const int p0 = sp * a.tps * AT_TILE;               // this block's positions [p0, p1)
    const int p1 = min(L, p0 + a.tps * AT_TILE);
    const int nt = p1 > p0 ? (p1 - p0 + AT_TILE - 1) / AT_TILE : 0;
    const int nb = (L + a.tps * AT_TILE - 1) / (a.tps * AT_TILE);   // non-empty blocks of (b, g)
    const size_t hout = ((size_t)b * AT_HQ + (size_t)AT_G * g) * AT_D;   // the group's first output
    if (nt == 0) {                                     // nothing cached here
        if (L == 0 && sp == 0)                         // an empty context: zeros
            for (int i = tid; i < AT_G * AT_D; i += AT_THREADS) a.out[hout + i] = from_f<TO>(0.0f);
        return;
    }
    const volatile int &aborted = ss.abort;

    if (tid == 0) {
        for (int s = 0; s < AT_SLOTS; ++s) {
            mbar_init(smem_u32(&ss.full[s]), 1);
            mbar_init(smem_u32(&ss.empty[s]), 1);
        }
        mbar_init(smem_u32(&ss.d1_full), 1);
        mbar_init(smem_u32(&ss.done), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&ss.p_full[i]), 128);
            mbar_init(smem_u32(&ss.d2_full[i]), 1);
        }
        ss.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();                                   // barriers exist: the producer may start
    if (warp == 1) {
        tc::tmem_alloc(smem_u32(&ss.tmem), AT_TMEM_COLS);
        tc::tmem_relinquish();
    }
    if (warp >= 2) {
        // Q^T operand: the group's 8 query heads, scaled by 1/sqrt(256) = 1/16
        // (a power of two: exact in bf16), 16-byte chunk c of head h's atom row
        // stored at chunk c ^ h (the 128-byte swizzle).
        const int t = tid - 64;
        const bf16 *qg = a.q + ((size_t)b * AT_HQ + (size_t)AT_G * g) * AT_D;
        for (int c = t; c < AT_G * AT_D / 8; c += 128) {
            const int h = c >> 5, cc = c & 31;
            uint4 u = __ldg(reinterpret_cast<const uint4 *>(qg + (size_t)h * AT_D) + cc);
            bf16 *e = reinterpret_cast<bf16 *>(&u);
#pragma unroll
            for (int i = 0; i < 8; ++i) e[i] = __float2bfloat16_rn(to_f(e[i]) * 0.0625f);
            *reinterpret_cast<uint4 *>(blk + SA_Q + (cc >> 3) * 1024 + h * 128 + (((cc & 7) ^ h) << 4)) = u;
        }
        fence_proxy_async_smem();
    }
    if (warp >= 1) {                                   // Q^T and TMEM ready for the issuer and softmax
        tc::fence_before_sync();
        asm volatile("bar.sync 2, 160;" ::: "memory");
        tc::fence_after_sync();
    }
    const uint32_t tm = warp >= 1 ? ss.tmem : 0u;
    auto slot_addr = [&](int i) { return sb + SA_RING + (uint32_t)(i % AT_SLOTS) * AT_SLOT_BYTES; };
    auto wait_full = [&](int i) {
        return mbar_wait_bounded(smem_u32(&ss.full[i % AT_SLOTS]), (uint32_t)((i / AT_SLOTS) & 1));
    };

    if (warp == 0) {
        // ---- TMA producer: copy i is tile i / 4, part i % 4 (K lo, K hi, V lo, V hi)
        if (lane == 0) {
            const int row0 = bg * a.Lmax + p0;
            int i = 0;
            for (; i < 4 * nt && !aborted; ++i) {
                const int s = i % AT_SLOTS;
                if (i >= AT_SLOTS &&
                    !mbar_wait_bounded(smem_u32(&ss.empty[s]), (uint32_t)((i / AT_SLOTS - 1) & 1))) {
                    ss.abort = 1;
                    break;
                }
                const CUtensorMap *m = (i & 2) ? &vmap : &kmap;
                const int x0 = (i & 1) * 128, y = row0 + (i >> 2) * AT_TILE;
                const uint32_t bar = smem_u32(&ss.full[s]);
                mbar_arrive_expect_tx(bar, AT_SLOT_BYTES);
                tma_load_2d(slot_addr(i), m, x0, y, bar);
                tma_load_2d(slot_addr(i) + AT_BOX, m, x0 + 64, y, bar);
            }
            for (int k = max(0, i - AT_SLOTS); k < i; ++k)   // copies in flight land before the CTA exits
                wait_full(k);
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            const uint32_t id1 = tc::instr_desc(tc::FMT_BF16, AT_TILE, 16);
            const uint32_t id2 = id1 | (1u << 15);     // A = V^T, read MN-major
            bool ok = true;
            for (int t = 0; t < nt && ok && !aborted; ++t) {
                const int i0 = 4 * t;
                ok = wait_full(i0) && wait_full(i0 + 1);
                if (!ok) break;
                tc::fence_after_sync();
                for (int kk = 0; kk < 16; ++kk) {          // S^T = K Q^T, 16 dims per step
                    const uint64_t ad =
                        tc::sw128_desc(slot_addr(i0 + (kk >> 3)) + ((kk >> 2) & 1) * AT_BOX + (kk & 3) * 32);
                    const uint64_t bd = tc::sw128_desc(sb + SA_Q + (kk >> 2) * 1024 + (kk & 3) * 32);
                    tc::mma_f16(tm + TC_D1, ad, bd, id1, kk > 0 ? 1u : 0u);
                }
                tc::mma_commit(smem_u32(&ss.empty[i0 % AT_SLOTS]));
                tc::mma_commit(smem_u32(&ss.empty[(i0 + 1) % AT_SLOTS]));
                tc::mma_commit(smem_u32(&ss.d1_full));
                ok = mbar_wait_bounded(smem_u32(&ss.p_full[t & 1]), (uint32_t)((t >> 1) & 1)) && wait_full(i0 + 2) &&
                     wait_full(i0 + 3);
                if (!ok || aborted) break;
                tc::fence_after_sync();
                const uint32_t pb = sb + SA_P + (uint32_t)(t & 1) * 2048;
                for (int hh = 0; hh < 2; ++hh) {           // O^T = V^T P^T, dims [128 hh, 128 hh + 128)
                    for (int kk = 0; kk < 8; ++kk) {       // 16 positions per step
                        const uint64_t ad = sw128_mn_desc(slot_addr(i0 + 2 + hh) + kk * 2048, AT_BOX);
                        const uint64_t bd = tc::sw128_desc(pb + (kk >> 2) * 1024 + (kk & 3) * 32);
                        tc::mma_f16(tm + TC_D2 + (t & 1) * 32 + hh * 16, ad, bd, id2, kk > 0 ? 1u : 0u);
                    }
                }
                tc::mma_commit(smem_u32(&ss.empty[(i0 + 2) % AT_SLOTS]));
                tc::mma_commit(smem_u32(&ss.empty[(i0 + 3) % AT_SLOTS]));
                tc::mma_commit(smem_u32(&ss.d2_full[t & 1]));
            }
            if (!ok) ss.abort = 1;
            tc::mma_commit(smem_u32(&ss.done));        // every MMA completes before TMEM is freed
            mbar_wait_bounded(smem_u32(&ss.done), 0u);
        }
    } else {
        // ---- online softmax (warps 2..5)
        const int q4 = warp & 3;                       // this warp's TMEM lane quarter
        const int r = 32 * q4 + lane;                  // position in a tile / dim in a half
        const uint32_t lbase = tm + ((uint32_t)(32 * q4) << 16);
        constexpr float LOG2E = 1.4426950408889634f;
        float m[AT_G], lsum[AT_G], acc0[AT_G], acc1[AT_G], corr_prev[AT_G];
#pragma unroll
        for (int h = 0; h < AT_G; ++h) {
            m[h] = -INFINITY;
            lsum[h] = acc0[h] = acc1[h] = corr_prev[h] = 0.0f;
        }
        bool ok = true;
        for (int t = 0; t <= nt; ++t) {
            float corr[AT_G];
            if (t < nt) {
                // scores of tile t
                const bool w = mbar_wait_bounded(smem_u32(&ss.d1_full), (uint32_t)(t & 1));
                if (!softmax_bar_and(w && !aborted)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                float s[AT_G];
                tmem_ld8(lbase + TC_D1, s);
                tc::wait_ld();
                const int nvalid = p1 - p0 - t * AT_TILE;  // valid positions in this tile (> 0)
                const bool valid = r < nvalid;
                float x[AT_G], mx[AT_G];
#pragma unroll
                for (int h = 0; h < AT_G; ++h) {
                    x[h] = valid ? s[h] * LOG2E : -INFINITY;
                    mx[h] = x[h];
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
                    for (int h = 0; h < AT_G; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
                if (lane == 0)
#pragma unroll
                    for (int h = 0; h < AT_G; ++h) ss.red[t & 1][q4][h] = mx[h];
                softmax_bar();
                unsigned char *pbuf = blk + SA_P + (t & 1) * 2048 + (r >> 6) * 1024;
#pragma unroll
                for (int h = 0; h < AT_G; ++h) {
                    const float tmx = fmaxf(fmaxf(ss.red[t & 1][0][h], ss.red[t & 1][1][h]),
                                            fmaxf(ss.red[t & 1][2][h], ss.red[t & 1][3][h]));
                    const float mn = fmaxf(m[h], tmx);     // finite: the tile has a valid position
                    corr[h] = exp2f(m[h] - mn);            // 0 on the first tile
                    m[h] = mn;
                    const bf16 pq = __float2bfloat16_rn(exp2f(x[h] - mn));
                    lsum[h] = lsum[h] * corr[h] + to_f(pq);   // the sum of the weights the MMA uses
                    *reinterpret_cast<bf16 *>(pbuf + h * 128 + ((((r & 63) >> 3) ^ h) << 4) + (r & 7) * 2) = pq;
                }
                if (nvalid < AT_TILE) {
                    // the tail tile: zero the value rows of the masked positions,
                    // whatever the cache holds there (0 * NaN would poison O)
                    const bool w2 = wait_full(4 * t + 2) && wait_full(4 * t + 3);
                    if (!softmax_bar_and(w2 && !aborted)) {
                        ok = false;
                        break;
                    }
                    if (!valid) {
                        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                        for (int part = 0; part < 2; ++part)
#pragma unroll
                            for (int box = 0; box < 2; ++box) {
                                uint4 *row = reinterpret_cast<uint4 *>(
                                    blk + (slot_addr(4 * t + 2 + part) - sb) + box * AT_BOX + r * 128);
#pragma unroll
                                for (int c = 0; c < 8; ++c) row[c] = zero;
                            }
                    }
                }
                fence_proxy_async_smem();                  // P^T (and zeroed rows) -> tensor core
                tc::fence_before_sync();                   // S^T read before it is overwritten
                mbar_arrive(smem_u32(&ss.p_full[t & 1]));
            }
            if (t > 0) {
                // outputs of tile t - 1
                const int u = t - 1;
                const bool w = mbar_wait_bounded(smem_u32(&ss.d2_full[u & 1]), (uint32_t)((u >> 1) & 1));
                if (!softmax_bar_and(w && !aborted)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                float o0[AT_G], o1[AT_G];
                tmem_ld8(lbase + TC_D2 + (u & 1) * 32, o0);
                tmem_ld8(lbase + TC_D2 + (u & 1) * 32 + 16, o1);
                tc::wait_ld();
#pragma unroll
                for (int h = 0; h < AT_G; ++h) {
                    acc0[h] = acc0[h] * corr_prev[h] + o0[h];
                    acc1[h] = acc1[h] * corr_prev[h] + o1[h];
                }
            }
            if (t < nt)
#pragma unroll
                for (int h = 0; h < AT_G; ++h) corr_prev[h] = corr[h];
        }
        if (ok) {
#pragma unroll
            for (int h = 0; h < AT_G; ++h) {
                float l = lsum[h];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                if (lane == 0) ss.lred[q4][h] = l;
            }
            softmax_bar();
            if (nb == 1) {
                // the whole context in this block: normalise and gate in place
#pragma unroll
                for (int h = 0; h < AT_G; ++h) {
                    const float inv = 1.0f / (ss.lred[0][h] + ss.lred[1][h] + ss.lred[2][h] + ss.lred[3][h]);
                    const size_t o = hout + (size_t)h * AT_D + r;
                    a.out[o] = from_f<TO>(acc0[h] * inv * sigmoid_f(to_f(a.z[o])));
                    a.out[o + 128] = from_f<TO>(acc1[h] * inv * sigmoid_f(to_f(a.z[o + 128])));
                }
            } else {
                float *po = a.part_o + (size_t)item * AT_G * AT_D;
                float *pml = a.part_ml + (size_t)item * AT_G * 2;
#pragma unroll
                for (int h = 0; h < AT_G; ++h) {
                    po[h * AT_D + r] = acc0[h];
                    po[h * AT_D + 128 + r] = acc1[h];
                }
                if (r < AT_G) {
                    float mr = m[0];                   // m[r], picked with static indices
#pragma unroll
                    for (int h = 1; h < AT_G; ++h) mr = r == h ? m[h] : mr;
                    pml[2 * r] = mr;
                    pml[2 * r + 1] = ss.lred[0][r] + ss.lred[1][r] + ss.lred[2][r] + ss.lred[3][r];
                }
            }
        } else if (r == 0) {
            ss.abort = 1;
        }
        tc::fence_before_sync();
    }
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tm, AT_TMEM_COLS);
    }
    if (tid == 0 && ss.abort) atomicExch(&g_attn_error, (unsigned int)GDN_ERR_TIMEOUT);
}

// Merges the blocks of each (sequence, query head) whose context spans nb > 1
// blocks: with block maxima m_s (log2 units), sums l_s and unnormalised outputs
// o_s, M = max m_s, w_s = 2^(m_s - M) and
//   out = (sum_s w_s o_s) / (sum_s w_s l_s) * sigmoid(z).
// One warp per (sequence, head), 8 dims per lane. Blocks are taken 8 at a time
// with all their loads issued before any is used (one memory round trip per 8
// blocks), and merged online with a running maximum.
template <typename TO>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float *__restrict__ part_o,
                                                           const float *__restrict__ part_ml,
                                                           const int32_t *__restrict__ ctx_len,
                                                           const bf16 *__restrict__ z, TO *__restrict__ out, int B,
                                                           int Lmax, int S, int tps)
{
    const int bh = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (bh >= B * AT_HQ) return;
    const int b = bh / AT_HQ, h = bh % AT_HQ, g = h / AT_G, hl = h % AT_G;
    grid_dep_wait();                                   // the partials come from the block kernel
    const int L = min(max(__ldg(ctx_len + b), 0), Lmax);
    const int nb = (L + tps * AT_TILE - 1) / (tps * AT_TILE);
    if (nb <= 1) return;                               // finished in place (or an empty context)
    const size_t it0 = ((size_t)b * AT_HKV + g) * S * AT_G + hl;   // (block 0, head hl) of this (b, g)
    float M = -INFINITY, l = 0.0f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int s0 = 0; s0 < nb; s0 += 8) {
        float mv[8], lv[8];
        float4 va[8], vb[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (s0 + j < nb) {
                const size_t it = it0 + (size_t)(s0 + j) * AT_G;
                mv[j] = __ldg(part_ml + it * 2);
                lv[j] = __ldg(part_ml + it * 2 + 1);
                const float4 *src = reinterpret_cast<const float4 *>(part_o + it * AT_D) + 2 * lane;
                va[j] = __ldg(src);
                vb[j] = __ldg(src + 1);
            } else {
                mv[j] = -INFINITY;
                lv[j] = 0.0f;
                va[j] = vb[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float Mc = M;
#pragma unroll
        for (int j = 0; j < 8; ++j) Mc = fmaxf(Mc, mv[j]);
        const float sc = exp2f(M - Mc);                // 0 for the first 8 blocks
        l *= sc;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] *= sc;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float w = exp2f(mv[j] - Mc);         // 0 for the padding entries
            l += w * lv[j];
            o[0] += w * va[j].x; o[1] += w * va[j].y; o[2] += w * va[j].z; o[3] += w * va[j].w;
            o[4] += w * vb[j].x; o[5] += w * vb[j].y; o[6] += w * vb[j].z; o[7] += w * vb[j].w;
        }
        M = Mc;
    }
    const float inv = 1.0f / l;
    const size_t o0 = (size_t)bh * AT_D + 8 * lane;
    const uint4 zr = __ldg(reinterpret_cast<const uint4 *>(z + o0));
    const uint32_t zw[4] = {zr.x, zr.y, zr.z, zr.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float zz = __uint_as_float((e & 1) ? (zw[e >> 1] & 0xFFFF0000u) : (zw[e >> 1] << 16));
        out[o0 + e] = from_f<TO>(o[e] * inv * sigmoid_f(zz));
    }
}

// ------------------------------------------------------------------ launcher

// Tiles per block: enough blocks for about six waves of two CTAs on each of
// 152 SMs, with blocks of at most 8 tiles (1024 positions). Measured at B=256
// and a 4K context: 8 tiles per block 312 us per call, 4 tiles 329, 16 tiles
// 322, whole contexts (no merge) 318. A pure function of (B, Lmax), so that
// the workspace size is too.
int attn_tiles_per_block(int B, int Lmax)
{
    const long long tiles = (Lmax + AT_TILE - 1) / AT_TILE;
    const long long t = (long long)B * AT_HKV * tiles / (6 * 2 * 152);
    return (int)(t < 1 ? 1 : (t > AT_TPS_MAX ? AT_TPS_MAX : t));
}

static int attn_blocks(int B, int Lmax)
{
    const int tiles = (Lmax + AT_TILE - 1) / AT_TILE, tps = attn_tiles_per_block(B, Lmax);
    return (tiles + tps - 1) / tps;
}

// Workspace: the partials of every block.
size_t attn_workspace_bytes(int B, int Lmax)
{
    const size_t items = (size_t)B * AT_HKV * attn_blocks(B, Lmax);
    return items * (AT_G * AT_D + 2 * AT_G) * sizeof(float);
}

template <typename TO>
static cudaError_t launch_attn_typed(const CUtensorMap &km, const CUtensorMap &vm, AttnArgs<TO> a, int B,
                                     cudaStream_t s)
{
    static std::mutex mu;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            e = cudaFuncSetAttribute(attn_block_kernel<TO>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)AT_SMEM);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
    }
    const size_t items = (size_t)B * AT_HKV * a.S;
    // both kernels use programmatic stream serialization (see grid_dep_wait)
    e = launch_pdl(attn_block_kernel<TO>, dim3((unsigned)items), dim3(AT_THREADS), AT_SMEM, s, km, vm, a);
    if (e != cudaSuccess || a.S == 1) return e;        // one block per context: nothing to merge
    return launch_pdl(attn_combine_kernel<TO>, dim3((unsigned)((B * AT_HQ + 7) / 8)), dim3(256), 0, s,
                      (const float *)a.part_o, (const float *)a.part_ml, a.ctx_len, a.z, a.out, B, a.Lmax, a.S,
                      a.tps);
}

cudaError_t launch_attn_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *ctx_len,
                               const void *z, void *out, int B, int Lmax, void *ws, gdn_dtype out_dt,
                               cudaStream_t s)
{
    if (B <= 0) return cudaSuccess;
    CUtensorMap km, vm;
    const long long rows = (long long)B * AT_HKV * Lmax;
    if (!make_bf16_sw128_map(&km, k_cache, rows, AT_D, AT_TILE) ||
        !make_bf16_sw128_map(&vm, v_cache, rows, AT_D, AT_TILE))
        return cudaErrorInvalidValue;
    const int tps = attn_tiles_per_block(B, Lmax), S = attn_blocks(B, Lmax);
    const size_t items = (size_t)B * AT_HKV * S;
    float *part_o = (float *)ws;
    float *part_ml = part_o + items * AT_G * AT_D;
    if (out_dt == GDN_F32) {
        AttnArgs<float> a{(const bf16 *)q, (const bf16 *)z, ctx_len, (float *)out, part_o, part_ml, Lmax, S, tps};
        return launch_attn_typed(km, vm, a, B, s);
    }
    AttnArgs<bf16> a{(const bf16 *)q, (const bf16 *)z, ctx_len, (bf16 *)out, part_o, part_ml, Lmax, S, tps};
    return launch_attn_typed(km, vm, a, B, s);
}

// Reads and clears this file's device error word (synchronous on `s`).
// Device address of this file's error word, for gdn_device_error, which reads
// and clears every word of the library in one kernel (NULL if the lookup fails).
void *attn_error_word()
{
    void *p = nullptr;
    return cudaGetSymbolAddress(&p, g_attn_error) == cudaSuccess ? p : nullptr;
}

}  // namespace gdn
