// gdn_tma.cuh -- tiled TMA (tensor-map) copies shared by the tensor-core
// kernels: the 2-D box load, and the host-side encoding of a row-major bf16
// matrix as a tensor map read in boxes 64 elements (128 bytes) wide with the
// 128-byte swizzle that tcgen05 shared-memory descriptors describe.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace gdn {

// 2-D tiled TMA load of the box at element coordinates (x = column, y = row),
// completion counted in bytes on the mbarrier `bar`. x * 2 bytes must be a
// multiple of 16 (every caller passes multiples of 64 columns).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                 "[%0], [%1, {%2, %3}], [%4];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

// Row-major bf16 matrix [rows][cols] (row stride cols * 2 bytes, a multiple of
// 16; base 16-byte aligned) as a tensor map read in boxes of 64 columns x
// box_rows rows, 128-byte swizzle; elements past either end read as zero.
// False if the driver's encoder is unavailable or rejects the arguments.
bool make_bf16_sw128_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_rows);

// The same matrix read in boxes of box_cols x box_rows elements without
// swizzle: a box lands in shared memory as box_rows dense rows of box_cols * 2
// bytes (box_cols a multiple of 8, at most 256; box_rows at most 256).
bool make_bf16_plain_map(CUtensorMap *map, const void *base, long long rows, int cols, int box_cols, int box_rows);

}  // namespace gdn
