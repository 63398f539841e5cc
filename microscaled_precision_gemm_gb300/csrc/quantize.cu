// K1: BF16 -> MXFP6 (E2M3 codes + E8M0 scales per 32 consecutive K-elements).
//
// "Optimizing Krea 3 on AMD Instinct MI355X", section "Fusion cut intermediate
// memory traffic": activations are quantized once and read once by the GEMM.
// The rule (OCP MX v1.0 conversion): amax over the block; scale exponent
// s = floor(log2 amax) - 2, clamped to [-127, 127]; each element rounds
// v * 2^-s to the nearest E2M3 value, ties to even, saturating at +-7.5.
//
// HBM-bound: 2 bytes in, 0.75 + 1/32 bytes out per element. Each lane owns 8
// consecutive elements (one 16-byte load, fully coalesced across the warp), four
// lanes share a block and reduce its amax with two shuffles, lane pairs merge
// their 6 code bytes into one 12-byte store, and 16 lanes merge four scale
// bytes into one 32-bit store in the tiled scale layout.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "mx_layout.cuh"
#include "ptx.cuh"

namespace mxk {

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;   // 16-byte loads in flight per lane

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Quantize 8 BF16 values (one 16-byte chunk) whose block shares `fac` = 2^-s.
// Returns the 8 codes packed into 48 bits (code i at bits 6i).
__device__ __forceinline__ uint64_t encode8(const uint4 raw, float fac) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint64_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = __uint_as_float(w[i] << 16) * fac;         // element 2i
    const float hi = __uint_as_float(w[i] & 0xFFFF0000u) * fac;  // element 2i+1
    const uint32_t p = cvt_e2m3x2(hi, lo);
    const uint64_t pair = (p & 0x3Fu) | (((p >> 8) & 0x3Fu) << 6);
    out |= pair << (12 * i);
  }
  return out;
}

__global__ void __launch_bounds__(kQuantThreads) quantize_bf16_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t k, int64_t ld_x, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t chunks_per_row = k / 8;
  const int64_t total_chunks = rows * chunks_per_row;
  const int64_t total_units = (total_chunks + 31) / 32;  // one unit = 32 chunks = 256 elements
  const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x) / 32;
  const int64_t warps_total = static_cast<int64_t>(gridDim.x) * kQuantThreads / 32;

  for (int64_t base = warp_global * kQuantUnroll; base < total_units; base += warps_total * kQuantUnroll) {
    uint4 raw[kQuantUnroll];
    int64_t chunk[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      chunk[u] = (base + u) * 32 + lane;
      raw[u] = make_uint4(0, 0, 0, 0);
      if (chunk[u] < total_chunks) {
        const int64_t r = chunk[u] / chunks_per_row;
        const int64_t c = (chunk[u] - r * chunks_per_row) * 8;
        raw[u] = ld_stream(x + r * ld_x + c);
      }
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      // |v| ordering of BF16 equals unsigned ordering of (bits & 0x7FFF); NaN/Inf sort last.
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
      uint32_t amax = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = max(amax, w[i] & 0x7FFFu);
        amax = max(amax, (w[i] >> 16) & 0x7FFFu);
      }
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
      amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
      uint32_t scale;
      uint64_t bits48;
      if (amax >= 0x7F80u) {  // Inf or NaN in the block: E8M0 NaN, zero codes
        scale = 0xFFu;
        bits48 = 0;
      } else {
        const int e = static_cast<int>(amax >> 7);         // biased exponent of amax (0 if subnormal)
        const int sc = e > 2 ? e - 2 : 0;                   // E8M0 code = max(floor(log2 amax) - 2, -127) + 127
        const float fac = __uint_as_float(static_cast<uint32_t>(254 - sc) << 23);  // 2^-s, exact
        scale = static_cast<uint32_t>(sc);
        bits48 = encode8(raw[u], fac);
      }
      // lane pairs: the even lane stores 16 codes = 12 bytes
      const uint64_t other = __shfl_xor_sync(0xffffffffu, bits48, 1);
      // four blocks (16 lanes) -> one 32-bit scale word
      const uint32_t s1 = __shfl_down_sync(0xffffffffu, scale, 4);
      const uint32_t s2 = __shfl_down_sync(0xffffffffu, scale, 8);
      const uint32_t s3 = __shfl_down_sync(0xffffffffu, scale, 12);
      if (chunk[u] < total_chunks) {
        if ((lane & 1) == 0) {
          uint32_t* dst = reinterpret_cast<uint32_t*>(codes + chunk[u] * 6);
          dst[0] = static_cast<uint32_t>(bits48);
          dst[1] = static_cast<uint32_t>(bits48 >> 32) | static_cast<uint32_t>(other << 16);
          dst[2] = static_cast<uint32_t>(other >> 16);
        }
        if ((lane & 15) == 0) {
          const int64_t elem = chunk[u] * 8;
          const int64_t r = elem / k;
          const int64_t kc = (elem - r * k) / kAtomK;
          const uint32_t word = scale | (s1 << 8) | (s2 << 16) | (s3 << 24);
          *reinterpret_cast<uint32_t*>(scales + scale_word_offset(r, kc, k)) = word;
        }
      }
    }
  }

  // Zero the scale words of the padding rows (rows .. rows rounded up to 128).
  const int64_t kcs = k / kAtomK;
  const int64_t pad_words = (pad_rows(rows) - rows) * kcs;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x; i < pad_words;
       i += static_cast<int64_t>(gridDim.x) * kQuantThreads) {
    const int64_t r = rows + i / kcs;
    const int64_t kc = i % kcs;
    *reinterpret_cast<uint32_t*>(scales + scale_word_offset(r, kc, k)) = 0u;
  }
}

cudaError_t launch_quantize_bf16(const void* x, int64_t rows, int64_t k, int64_t ld_x, void* codes, void* scales,
                                 int num_sms, cudaStream_t stream) {
  const int64_t units = (rows * (k / 8) + 31) / 32;
  const int64_t warps_needed = (units + kQuantUnroll - 1) / kQuantUnroll;
  int64_t blocks = (warps_needed * 32 + kQuantThreads - 1) / kQuantThreads;
  const int64_t pad_blocks = ((pad_rows(rows) - rows) * (k / kAtomK) + kQuantThreads - 1) / kQuantThreads;
  if (blocks < pad_blocks) blocks = pad_blocks;
  const int64_t cap = static_cast<int64_t>(num_sms) * (2048 / kQuantThreads);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  quantize_bf16_kernel<<<static_cast<unsigned>(blocks), kQuantThreads, 0, stream>>>(
      static_cast<const uint16_t*>(x), rows, k, ld_x, static_cast<uint8_t*>(codes),
      static_cast<uint8_t*>(scales));
  return cudaGetLastError();
}

}  // namespace mxk
