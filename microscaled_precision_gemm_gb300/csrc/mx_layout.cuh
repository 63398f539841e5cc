// MXFP6 storage layout shared by the quantizer, the GEMM and the host API.
//
// Codes: 6-bit E2M3 codes packed densely per row, little-endian -- code j of a
// row occupies bits [6j, 6j + 6) of the row's bit string -- so a row of K
// elements is 3K/4 bytes and every 16 codes are the 12-byte group that the
// tensor-memory-access unit's 16 x U6 type moves into a 16-byte shared-memory
// slot (12 data bytes + 4 padding bytes), the operand form tcgen05.mma reads.
//
// Scales: one E8M0 byte per (row, 32-element K-block), in the tiled order the
// tensor cores' scale-factor copy (tcgen05.cp 32x128b.warpx4) consumes: 512-byte
// atoms, one per (128-row group, 4 consecutive K-blocks), atoms of a row group
// consecutive along K. Inside an atom, row r = 32*r1 + r0 and K-block j sit at
// byte 16*r0 + 4*r1 + j, i.e. one 16-byte tensor-memory lane row per r0 holding
// four 32-bit columns (r1), one byte per K-block (the MMA's scale-factor id).
// Rows are padded to a multiple of 128; padding scales are written as 0.
#pragma once

#include <cstdint>

namespace mxk {

constexpr int kBlock = 32;           // elements per scale
constexpr int kAtomRows = 128;       // rows per scale atom
constexpr int kAtomK = 128;          // K elements per scale atom (4 blocks)
constexpr int kAtomBytes = 512;

__host__ __device__ __forceinline__ int64_t pad_rows(int64_t rows) { return (rows + 127) / 128 * 128; }

__host__ __device__ __forceinline__ int64_t codes_bytes(int64_t rows, int64_t k) { return rows * k / 4 * 3; }

__host__ __device__ __forceinline__ int64_t scales_bytes(int64_t rows, int64_t k) {
  return pad_rows(rows) * (k / kBlock);
}

// Byte offset of the 4-byte scale word of (row, K-blocks 4*kc .. 4*kc+3).
__host__ __device__ __forceinline__ int64_t scale_word_offset(int64_t row, int64_t kc, int64_t k) {
  return ((row / kAtomRows) * (k / kAtomK) + kc) * kAtomBytes + (row % 32) * 16 + ((row % 128) / 32) * 4;
}

}  // namespace mxk
