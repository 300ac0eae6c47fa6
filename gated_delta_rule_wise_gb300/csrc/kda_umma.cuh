// kda_umma.cuh -- operand layouts and descriptors for tcgen05.mma (kind::f16,
// bf16 inputs, f32 accumulate) as used by the tensor-core chunked prefill.
//
// Every shared-memory operand is K-major with the 128-byte swizzle: the K
// axis is cut into atoms of 64 bf16 (128 bytes); an atom column of a tile
// with R rows is an [R x 128 B] block of 8-row groups (1024 B each), and the
// 16-byte chunk c of row r sits at chunk position c ^ (r & 7).  The blocks of
// successive K atoms follow each other.  A tile built this way in registers,
// written to global memory as-is and copied back with a bulk copy is again a
// valid operand, which is how the prep kernel hands its per-chunk matrices
// to the scan kernel.
#pragma once

#include <stdint.h>

namespace kda {
namespace umma {

// Byte offset of element (row, k) of a K-major SW128 bf16 tile with `rows` rows.
__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int k, int rows) {
  const int katom = k >> 6, kk = k & 63;
  const uint32_t base = (uint32_t)katom * rows * 128u + (uint32_t)(row >> 3) * 1024u +
                        (uint32_t)(row & 7) * 128u;
  return base + ((uint32_t)((kk >> 3) ^ (row & 7)) << 4) + (uint32_t)(kk & 7) * 2u;
}
// Byte offset of the 16-byte chunk holding k = 8*c8 .. 8*c8+7 of `row`.
__host__ __device__ __forceinline__ uint32_t sw128_chunk(int row, int c8, int rows) {
  const int katom = c8 >> 3, cc = c8 & 7;
  return (uint32_t)katom * rows * 128u + (uint32_t)(row >> 3) * 1024u +
         (uint32_t)(row & 7) * 128u + ((uint32_t)(cc ^ (row & 7)) << 4);
}
// Bytes of a [rows x K] tile.
__host__ __device__ constexpr uint32_t tile_bytes(int rows, int K) { return (uint32_t)rows * K * 2u; }

// Shared-memory matrix descriptor for a SW128 K-major operand whose 8-row
// groups are 1024 B apart (the tile's atom column must be 1024-B aligned).
__device__ __forceinline__ uint64_t sdesc(uint32_t smem_addr) {
  uint64_t d = (uint64_t)((smem_addr & 0x3FFFFu) >> 4);  // start address / 16
  d |= (uint64_t)1u << 16;                                 // leading offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;                       // stride offset: 8-row groups
  d |= (uint64_t)1u << 46;                                 // descriptor version
  d |= (uint64_t)2u << 61;                                 // 128-byte swizzle
  return d;
}

// Descriptor of the K-slice [16*ks, 16*ks + 16) of a [rows x K] tile at `tile`.
__device__ __forceinline__ uint64_t sdesc_k(uint32_t tile, int rows, int ks) {
  return sdesc(tile + (uint32_t)(ks >> 2) * rows * 128u + (uint32_t)(ks & 3) * 32u);
}

// Descriptor of the K-slice [16*ks, 16*ks + 16) of an MN-major operand stored
// as a K-major SW128 tile whose ROWS run along K (the operand's K index) and
// whose columns run along MN: the same bytes as the tile of the transposed
// matrix.  `tile_rows` is the row count of the containing tile (its 64-column
// blocks are tile_rows * 128 B apart); `tile` may point at a row that is a
// multiple of 8 inside it.
__device__ __forceinline__ uint64_t sdesc_mn(uint32_t tile, int tile_rows, int ks) {
  uint64_t d = (uint64_t)(((tile + (uint32_t)ks * 2048u) & 0x3FFFFu) >> 4);
  d |= (uint64_t)(((uint32_t)tile_rows * 128u) >> 4) << 16;  // between 64-wide MN blocks
  d |= (uint64_t)(1024u >> 4) << 32;                         // between 8-row K groups
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)2u << 61;
  return d;
}

// Instruction descriptor: D f32, A and B bf16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// Same with the A operand MN-major, the B operand MN-major, or both.
__host__ __device__ constexpr uint32_t idesc_bf16_amn(int M, int N) { return idesc_bf16(M, N) | (1u << 15); }
__host__ __device__ constexpr uint32_t idesc_bf16_bmn(int M, int N) { return idesc_bf16(M, N) | (1u << 16); }
__host__ __device__ constexpr uint32_t idesc_bf16_abmn(int M, int N) {
  return idesc_bf16(M, N) | (1u << 15) | (1u << 16);
}

}  // namespace umma
}  // namespace kda
