// tile_layout.cuh -- shared-memory layout of the 128-row operand tiles.
//
// Every tile (Q, K, V and the rotary "lo" side buffers) holds 128 rows of bf16 and is
// stored as column blocks of 32 elements: block cb covers columns [32cb, 32cb+32) and is
// a dense [128][32] array (64-byte rows, 8 KB) with the 64-byte TMA/UMMA swizzle, i.e.
// the 16-byte chunk index (byte bits 4-5) is XORed with byte bits 7-8 (= (row >> 1) & 3).
// TMA writes exactly this layout for a {32 x 128} box with CU_TENSOR_MAP_SWIZZLE_64B, and
// the tensor cores read it through the descriptors below.  Blocks are 1 KB aligned.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace neox {

constexpr int kRows = 128;                  // rows per tile (BM = BN = 128)
constexpr int kBlkCols = 32;                // bf16 columns per column block
constexpr int kBlkBytes = kRows * kBlkCols * 2;  // 8 KB

__host__ __device__ constexpr int tile_bytes(int cols) { return (cols / kBlkCols) * kBlkBytes; }

// Byte offset of element (row, col) inside a tile.
__device__ __forceinline__ uint32_t sw64_off(int row, int col) {
  const int cb = col >> 5, chunk = (col >> 3) & 3;
  return static_cast<uint32_t>(cb * kBlkBytes + row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4) + (col & 7) * 2);
}

// K-major operand descriptor for the 16-column chunk kc of a tile whose rows are the
// MMA's M (or N) dimension and whose columns are the contraction dimension.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_saddr, int kc) {
  const uint32_t a = tile_saddr + static_cast<uint32_t>((kc >> 1) * kBlkBytes + (kc & 1) * 32);
  return sdesc_sw64(a, 16, 8 * 64);
}

// MN-major operand descriptor for a V tile (rows = keys = contraction, columns = head
// dims = N): 16 keys starting at key 16*kk; N blocks of 32 dims are kBlkBytes apart.
__device__ __forceinline__ uint64_t vmajor_desc(uint32_t tile_saddr, int kk) {
  const uint32_t a = tile_saddr + static_cast<uint32_t>(kk * 16 * 64);
  return sdesc_sw64(a, kBlkBytes, 8 * 64);
}

}  // namespace neox
