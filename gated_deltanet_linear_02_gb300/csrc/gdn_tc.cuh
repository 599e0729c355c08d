// gdn_tc.cuh -- 5th-generation tensor core (tcgen05) primitives as inline PTX
// for sm_103a: tensor-memory allocation, shared-memory matrix descriptors, the
// instruction descriptor, MMA issue and commit, TMEM loads and stores, and the
// fences that order them against ordinary thread synchronisation.
//
// Operand layout used throughout libgdn: K-major, no swizzle. A tile of R rows
// (the M or N extent) by Kd elements along K is stored as 8-row x 16-byte
// "core matrices" (8 rows of 16 contiguous bytes, 128 bytes in all).
// Consecutive core matrices along K are 128 bytes apart (the leading-dimension
// byte offset, LBO). Consecutive 8-row groups are Kd * elem_size * 8 bytes
// apart (the stride-dimension byte offset, SBO). Element (r, k) lives at
//   (r / 8) * SBO + (k / kc) * 128 + (r % 8) * 16 + (k % kc) * elem_size,
// with kc = 16 / elem_size (8 for bf16, 4 for tf32).
#pragma once

#include <stdint.h>

#include "gdn_async.cuh"

namespace gdn {
namespace tc {

// byte offset of element (r, k) in a K-major no-swizzle tile with Kd columns
template <int ES>
__host__ __device__ __forceinline__ uint32_t kmajor_offset(int r, int k, int Kd)
{
    constexpr int kc = 16 / ES;
    return (uint32_t)((r >> 3) * (Kd * ES * 8) + (k / kc) * 128 + (r & 7) * 16 + (k % kc) * ES);
}

// Shared-memory matrix descriptor (sm_100 family): start address, LBO and SBO
// in 16-byte units, version 1 at bits 46-47, no swizzle (layout type 0).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Descriptor of the K-slice starting at element k0 of a K-major tile with Kd
// columns and element size ES, based at shared address `base`.
template <int ES>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int k0, int Kd)
{
    return smem_desc(base + (uint32_t)((k0 / (16 / ES)) * 128), 128u, (uint32_t)(Kd * ES * 8));
}

// Descriptor of a K-major tile in the 128-byte-swizzle layout that a TMA copy
// with CU_TENSOR_MAP_SWIZZLE_128B writes for a box 128 bytes wide: rows of 128
// bytes (64 bf16), the 16-byte chunks of row r permuted by XOR with r % 8, and
// 8-row groups 1024 bytes apart (SBO). Layout type 2 (bits 61-63) selects the
// 128-byte swizzle; the leading-dimension offset is unused for this layout. The
// tile base must be 1024-byte aligned. A K offset of b bytes inside the row is
// added to the start address (b >> 4 in the descriptor's low field).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    return smem_desc(saddr, 16u, 1024u) | ((uint64_t)2 << 61);
}

enum : uint32_t { FMT_F16 = 0, FMT_BF16 = 1, FMT_TF32 = 2 };

// An fp32 value rounded to the nearest tf32 (10-bit mantissa). The tensor core
// only reads the top 19 bits of a tf32 operand, which truncates it toward zero.
// Over long sums that truncation bias grows about 3x larger than the
// round-to-nearest error, so every tf32 operand is rounded when stored.
__device__ __forceinline__ float tf32_rn(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
__device__ __forceinline__ float4 tf32_rn(float4 v)
{
    return make_float4(tf32_rn(v.x), tf32_rn(v.y), tf32_rn(v.z), tf32_rn(v.w));
}

// Instruction descriptor: fp32 accumulator, A/B formats, both K-major, N and M.
__host__ __device__ constexpr uint32_t instr_desc(uint32_t ab_fmt, int M, int N)
{
    return (1u << 4) | (ab_fmt << 7) | (ab_fmt << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---- tensor memory
// Allocates `ncols` columns (power of two >= 32); the base address is written
// to *smem_dst. Must be executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_dst), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- MMA: D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrives once on `bar` when every MMA issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// D (+)= A * B^T over the K extent `kd`, A and B K-major tiles with `kd`
// columns, in steps of the instruction K (16 for bf16, 8 for tf32).
template <bool TF32>
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_base, int a_kd, uint32_t b_base, int b_kd,
                                         int kd, uint32_t idesc, bool accumulate)
{
    constexpr int ES = TF32 ? 4 : 2;
    constexpr int KI = TF32 ? 8 : 16;
    for (int k0 = 0; k0 < kd; k0 += KI) {
        const uint64_t a = kmajor_desc<ES>(a_base, k0, a_kd);
        const uint64_t b = kmajor_desc<ES>(b_base, k0, b_kd);
        if (TF32) mma_tf32(d_tmem, a, b, idesc, (accumulate || k0 > 0) ? 1u : 0u);
        else mma_f16(d_tmem, a, b, idesc, (accumulate || k0 > 0) ? 1u : 0u);
    }
}

// Same product with both descriptors given for the first K step: every MMA
// instruction covers 32 bytes of K, i.e. two 128-byte core matrices along K, so
// the next step's descriptors are the previous ones plus 256 B >> 4 = 16 in the
// start-address field. This holds for K-major tiles (LBO 128) and for MN-major
// bf16 tiles with 128-byte K-group stride.
template <bool TF32>
__device__ __forceinline__ void mma_steps(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, int steps, uint32_t idesc,
                                          bool accumulate)
{
    for (int s = 0; s < steps; ++s) {
        if (TF32) mma_tf32(d_tmem, a_desc + 16u * s, b_desc + 16u * s, idesc, (accumulate || s > 0) ? 1u : 0u);
        else mma_f16(d_tmem, a_desc + 16u * s, b_desc + 16u * s, idesc, (accumulate || s > 0) ? 1u : 0u);
    }
}

// Byte offset of element (n, k) in an MN-major, no-swizzle bf16 tile with Kd
// columns along K: 16-byte MN groups (8 elements) are SBO = Kd * 16 bytes apart,
// groups of 8 K rows are 128 bytes apart, and each K row is 16 bytes.
__host__ __device__ __forceinline__ uint32_t mnmajor_offset_bf16(int n, int k, int Kd)
{
    return (uint32_t)((n >> 3) * (Kd * 16) + (k >> 3) * 128 + (k & 7) * 16 + (n & 7) * 2);
}

// ---- fences around thread synchronisation
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- TMEM <-> registers: 32 lanes (this warp's quarter) x 16 consecutive
// 32-bit columns; thread t gets lane (32 * (warp % 4) + t). `taddr` carries
// the lane base in bits 31..16 and the column in bits 15..0.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                   "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                   "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                   "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                   "r"(__float_as_uint(v[15]))
                 : "memory");
}

__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int lane, int col)
{
    return base + ((uint32_t)lane << 16) + (uint32_t)col;
}

// ---- fp16 forms used by the chunked prefill

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16: the A operand (M rows x 16 K
// elements) is read from tensor memory, row m in lane m, two 16-bit elements per
// 32-bit column (the even K index in the low half), so one K step of 16 is 8
// columns. Issued by one thread.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Descriptor of an MN-major no-swizzle 16-bit tile laid out as
// mnmajor_offset_bf16: 8-element MN groups SBO bytes apart, 8-row K groups 128
// bytes apart. A K step of 16 adds 256 bytes to the start address.
__device__ __forceinline__ uint64_t mn_desc(uint32_t saddr, uint32_t sbo_bytes)
{
    return smem_desc(saddr, 128u, sbo_bytes);
}

// Descriptor of an MN-major 16-bit operand in the 128-byte swizzle, as a TMA box
// 64 elements wide writes it: atoms of 64 MN elements x 8 K rows (1 KiB), LBO =
// distance to the next 64 MN elements (the next box), SBO = 1 KiB to the next 8
// K rows. A K step of 16 rows adds 2 KiB to the start address. Box bases are
// 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t lbo_bytes)
{
    return smem_desc(saddr, lbo_bytes, 1024u) | ((uint64_t)2 << 61);
}

// Instruction-descriptor bits selecting MN-major (transposed) A and B operands.
constexpr uint32_t IDESC_A_MN = 1u << 15;
constexpr uint32_t IDESC_B_MN = 1u << 16;

// Two fp32 values rounded to fp16 and packed in one word, the first in the low half.
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 32 lanes x 32 consecutive 32-bit columns (see tmem_ld16).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive 32-bit columns of raw words (packed fp16 pairs).
__device__ __forceinline__ void tmem_st16_u32(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                   "r"(r[15])
                 : "memory");
}

// 32 lanes x 8 consecutive 32-bit columns of raw words (packed fp16 pairs).
__device__ __forceinline__ void tmem_st8_u32(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                   "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                   "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                   "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                   "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                   "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                   "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
                   "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                   "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
                   "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                   "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
}

}  // namespace tc
}  // namespace gdn
