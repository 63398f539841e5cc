// K1: BF16 -> MXFP6 (E2M3 codes + E8M0 scales per 32 consecutive K-elements).
//
// "Optimizing Krea 3 on AMD Instinct MI355X", section "Fusion cut intermediate
// memory traffic": activations are quantized once and read once by the GEMM.
// The rule (OCP MX v1.0 conversion): amax over the block; scale exponent
// s = floor(log2 amax) - 2, clamped to [-127, 127]; each element rounds
// v * 2^-s to the nearest E2M3 value, ties to even, saturating at +-7.5.
//
// HBM-bound: 2 bytes in, 0.75 + 1/32 bytes out per element. One lane owns one
// 32-element block, so the amax is thread-local; the lane widens its BF16 values to
// fp32 (exact) and runs the block encoder the GEMM epilogues use.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "mx_layout.cuh"
#include "mx_quant.cuh"
#include "ptx.cuh"

namespace mxk {

constexpr int kQuantThreads = 256;

// Quotient of n by an invariant divisor d with a precomputed magic number
// (division by invariant integers using multiplication, round-up variant):
// m = floor(2^32 (2^l - d) / d) + 1 with l = ceil(log2 d); q = (mulhi(n, m) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
};

__host__ __device__ __forceinline__ uint32_t fast_div(uint32_t n, FastDiv f) {
#ifdef __CUDA_ARCH__
  return static_cast<uint32_t>((static_cast<uint64_t>(__umulhi(n, f.m)) + n) >> f.l);
#else
  return n / f.d;
#endif
}

static FastDiv make_fast_div(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t{1} << l) < d) ++l;
  const uint64_t m = ((uint64_t{1} << 32) * ((uint64_t{1} << l) - d)) / d + 1;
  return FastDiv{d, static_cast<uint32_t>(m), l};
}

// One lane quantizes one 32-element block: 64 contiguous input bytes (four
// 16-byte loads), a thread-local amax, the E2M3 conversions, 24 packed code bytes.
// A warp owns 32 consecutive blocks of the flattened [rows][K/32] block grid, so
// its 768 code bytes are contiguous in the packed output; they are staged in
// shared memory and written as 16-byte stores. Four consecutive lanes (4 K-blocks
// of one row) form one 32-bit tiled scale word. The loads of the lane's next block
// are issued before the current one is encoded.
__global__ void __launch_bounds__(kQuantThreads, 4) quantize_bf16_kernel(
    const uint16_t* __restrict__ x, int rows, int k, int64_t ld_x, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, FastDiv blocks_per_row, uint32_t total_blocks, unsigned* __restrict__ zero_words,
    int zero_count) {
  const int lane = threadIdx.x & 31;
  const uint32_t warp_global = (blockIdx.x * kQuantThreads + threadIdx.x) / 32;
  const uint32_t stride = gridDim.x * kQuantThreads;   // blocks per grid-wide step
  __shared__ __align__(16) uint32_t stage[kQuantThreads / 32][192];
  uint32_t* st = stage[threadIdx.x / 32];

  // programmatic dependent launch: let the next kernel be scheduled, and read x /
  // write the outputs only once the previous kernel has completed
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < zero_count; i += kQuantThreads) zero_words[i] = 0u;

  auto load_block = [&](uint32_t b, uint4 (&v)[4]) {
    const uint32_t r = fast_div(b, blocks_per_row);
    const uint16_t* src = x + static_cast<int64_t>(r) * ld_x + (b - r * blocks_per_row.d) * 32;
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = b < total_blocks ? ld_nc(src + 8 * j) : make_uint4(0, 0, 0, 0);
  };
  uint4 next[4];
  load_block(warp_global * 32 + lane, next);
  for (uint32_t base = warp_global * 32; base < total_blocks; base += stride) {
    const uint32_t b = base + lane;
    const bool valid = b < total_blocks;
    const uint32_t row = fast_div(b, blocks_per_row);
    const uint32_t kb = b - row * blocks_per_row.d;
    uint4 raw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) raw[j] = next[j];
    load_block(b + stride, next);
    // BF16 -> fp32 is exact, so the fp32 block encoder gives the BF16 rule's result
    // (amax, scale, codes; NaN/Inf blocks included)
    float f[32];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t v[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        f[8 * j + 2 * i] = __uint_as_float(v[i] << 16);
        f[8 * j + 2 * i + 1] = __uint_as_float(v[i] & 0xFFFF0000u);
      }
    }
    uint32_t w[6];
    const uint32_t sc = quant_block32(f, w);
    uint2* s2 = reinterpret_cast<uint2*>(&st[6 * lane]);
    s2[0] = make_uint2(w[0], w[1]);
    s2[1] = make_uint2(w[2], w[3]);
    s2[2] = make_uint2(w[4], w[5]);
    // four consecutive blocks (K-blocks 4c..4c+3 of one row) -> one tiled scale word
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, sc, 1);
    const uint32_t s2b = __shfl_down_sync(0xffffffffu, sc, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, sc, 3);
    if (valid && (lane & 3) == 0)
      *reinterpret_cast<uint32_t*>(scales + scale_word_offset(row, kb / 4, k)) =
          sc | (s1 << 8) | (s2b << 16) | (s3 << 24);
    __syncwarp();
    // the warp's blocks are consecutive: their codes are 24 * 32 contiguous bytes
    const uint32_t nblk = min(32u, total_blocks - base);  // a multiple of 4
    const uint32_t chunks = nblk * 24 / 16;
    uint4* dst = reinterpret_cast<uint4*>(codes + static_cast<int64_t>(base) * 24);
    const uint4* src = reinterpret_cast<const uint4*>(st);
    for (uint32_t c = lane; c < chunks; c += 32) dst[c] = src[c];
    __syncwarp();
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
                                 int num_sms, cudaStream_t stream, unsigned* zero_words, int zero_count) {
  const int64_t total_blocks = rows * (k / kBlock);
  if (total_blocks > (int64_t{1} << 32) - (int64_t{1} << 28)) return cudaErrorInvalidValue;  // host checks first
  const int64_t warps_needed = (total_blocks + 31) / 32;
  int64_t blocks = (warps_needed * 32 + kQuantThreads - 1) / kQuantThreads;
  const int64_t pad_blocks = ((pad_rows(rows) - rows) * (k / kAtomK) + kQuantThreads - 1) / kQuantThreads;
  if (blocks < pad_blocks) blocks = pad_blocks;
  // every block resident at once (grid-stride), so no second partial wave
  static std::atomic<int> resident_per_sm[64];   // per-device occupancy, any thread may fill it
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  int per_sm = (dev >= 0 && dev < 64) ? resident_per_sm[dev].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_bf16_kernel, kQuantThreads, 0);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    if (dev >= 0 && dev < 64) resident_per_sm[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t cap = static_cast<int64_t>(num_sms) * per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kQuantThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, quantize_bf16_kernel, static_cast<const uint16_t*>(x), static_cast<int>(rows),
                                     static_cast<int>(k), ld_x, static_cast<uint8_t*>(codes),
                                     static_cast<uint8_t*>(scales), make_fast_div(static_cast<uint32_t>(k / kBlock)),
                                     static_cast<uint32_t>(total_blocks), zero_words, zero_words ? zero_count : 0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mxk
