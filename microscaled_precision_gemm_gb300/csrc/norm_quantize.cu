// K1 with the step before it fused in: row-wise RMS normalisation, modulation and
// the MXFP6 quantization of the result, one pass over the BF16 activations.
//
//   y[m][k] = x[m][k] / sqrt(mean_k' x[m][k']^2 + eps) * (1 + scale[k]) + shift[k]
//   (codes, scales) = MXFP6(y)        (the quantizer's rule, on fp32 y)
//
// "Optimizing Krea 3 on AMD Instinct MI355X", section "Fusion cut intermediate
// memory traffic": modulation merges with RMSNorm before the projections, so the
// normalised activations never travel through HBM in BF16. "Creating Custom
// Kernels for the AMD MI300", section "Fused RMS Norm Kernel": one block per row,
// the row's sum of squares reduced across the block, vectorised 16-byte loads.
//
// HBM-bound like K1: 2 bytes in, 0.75 + 1/32 bytes out per element. A CTA owns
// whole rows (one warp per 1024 columns, K <= 8192); lane l of warp w owns K-block
// 32 w + l for every row, so its 32 modulation pairs (1 + scale, shift) stay in
// registers for the whole kernel. Per row: each lane's sum of squares, a warp
// tree, one barrier to combine the warps' partials (double-buffered slots), then
// y, its amax and the paired E2M3 conversions; the next row is already in flight,
// loaded into the other of two register buffers that alternate from row to row.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "mx_layout.cuh"
#include "mx_quant.cuh"
#include "ptx.cuh"

namespace mxk {

constexpr int kNormMaxWarps = 8;   // K <= 8192

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <bool DBG>
__global__ void __launch_bounds__(kNormMaxWarps * 32, 2) norm_modulate_quantize_kernel(
    const uint16_t* __restrict__ x, int rows, int k, int64_t ld_x, const uint16_t* __restrict__ shift,
    const uint16_t* __restrict__ scale, float eps, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
    float* __restrict__ dbg, unsigned* __restrict__ zero_words, int zero_count) {
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int nwarps = blockDim.x / 32;
  const int blocks_per_row = k / kBlock;
  const int kb = warp * 32 + lane;            // this lane's K-block
  const bool active = kb < blocks_per_row;
  const float inv_k = 1.0f / static_cast<float>(k);
  __shared__ float partial[2][kNormMaxWarps];
  __shared__ __align__(16) uint32_t stage[kNormMaxWarps][192];

  // programmatic dependent launch: let the next kernel be scheduled, and read the
  // inputs / write the outputs only once the previous kernel has completed
  if (threadIdx.x == 0) griddep_launch_dependents();
  griddep_wait();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < zero_count; i += blockDim.x) zero_words[i] = 0u;

  // this lane's 32 columns of the modulation: (1 + scale) in fp32, shift as BF16 pairs
  float opp[32];
  uint32_t sh[16];
#pragma unroll
  for (int i = 0; i < 32; ++i) opp[i] = 1.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) sh[i] = 0u;
  if (active) {
    if (scale != nullptr) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(scale + kb * kBlock) + j);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          opp[8 * j + 2 * t] = 1.0f + bf16_lo(w[t]);
          opp[8 * j + 2 * t + 1] = 1.0f + bf16_hi(w[t]);
        }
      }
    }
    if (shift != nullptr) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(shift + kb * kBlock) + j);
        sh[4 * j] = v.x;
        sh[4 * j + 1] = v.y;
        sh[4 * j + 2] = v.z;
        sh[4 * j + 3] = v.w;
      }
    }
  }

  int parity = 0;
  auto process_row = [&](int row, const uint4 (&cur)[4]) {
    const uint32_t xw[16] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w, cur[1].x, cur[1].y, cur[1].z, cur[1].w,
                             cur[2].x, cur[2].y, cur[2].z, cur[2].w, cur[3].x, cur[3].y, cur[3].z, cur[3].w};
    // four interleaved partial sums (two packed pairs) keep the dependent chain 8 deep
    uint64_t s2[2] = {0ull, 0ull};
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint64_t xp = f2_pack(bf16_lo(xw[i]), bf16_hi(xw[i]));
      s2[i & 1] = f2_fma(xp, xp, s2[i & 1]);
    }
    float s4[4];
    f2_unpack(s2[0], s4[0], s4[1]);
    f2_unpack(s2[1], s4[2], s4[3]);
    float ss = (s4[0] + s4[1]) + (s4[2] + s4[3]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) partial[parity][warp] = ss;
    __syncthreads();
    float tot = partial[parity][0];
    for (int w = 1; w < nwarps; ++w) tot += partial[parity][w];   // same order in every thread
    const float rstd = rsqrtf(fmaf(tot, inv_k, eps));   // CUDA's rsqrtf: within 2 ulp

    uint32_t sc = 0;
    if (active) {
      float y[32];
      const uint64_t rstd2 = f2_pack(rstd, rstd);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint64_t xr = f2_mul(f2_pack(bf16_lo(xw[i]), bf16_hi(xw[i])), rstd2);
        f2_unpack(f2_fma(xr, f2_pack(opp[2 * i], opp[2 * i + 1]), f2_pack(bf16_lo(sh[i]), bf16_hi(sh[i]))),
                  y[2 * i], y[2 * i + 1]);
      }
      if constexpr (DBG) {
        float4* d = reinterpret_cast<float4*>(dbg + static_cast<int64_t>(row) * k + kb * kBlock);
#pragma unroll
        for (int v = 0; v < 8; ++v) d[v] = make_float4(y[4 * v], y[4 * v + 1], y[4 * v + 2], y[4 * v + 3]);
      }
      uint32_t w[6];
      sc = quant_block32(y, w);
      uint2* s2 = reinterpret_cast<uint2*>(&stage[warp][6 * lane]);
      s2[0] = make_uint2(w[0], w[1]);
      s2[1] = make_uint2(w[2], w[3]);
      s2[2] = make_uint2(w[4], w[5]);
    }
    // four consecutive K-blocks of the row -> one tiled scale word
    const uint32_t s1 = __shfl_down_sync(0xffffffffu, sc, 1);
    const uint32_t s2b = __shfl_down_sync(0xffffffffu, sc, 2);
    const uint32_t s3 = __shfl_down_sync(0xffffffffu, sc, 3);
    if (active && (lane & 3) == 0)
      *reinterpret_cast<uint32_t*>(scales + scale_word_offset(row, kb / 4, k)) =
          sc | (s1 << 8) | (s2b << 16) | (s3 << 24);
    __syncwarp();
    // the warp's blocks are consecutive in the row: their codes are contiguous
    const int nblk = min(32, blocks_per_row - warp * 32);   // a multiple of 4 (K % 128 == 0)
    if (nblk > 0) {
      const int chunks = nblk * 24 / 16;
      uint4* dst = reinterpret_cast<uint4*>(codes + static_cast<int64_t>(row) * (k / 4 * 3) + warp * 768);
      const uint4* src = reinterpret_cast<const uint4*>(stage[warp]);
      for (int c = lane; c < chunks; c += 32) dst[c] = src[c];
    }
    __syncwarp();
    parity ^= 1;
  };
  auto load_row = [&](int r, uint4 (&v)[4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = make_uint4(0, 0, 0, 0);
    if (r < rows && active) {
      const uint16_t* src = x + static_cast<int64_t>(r) * ld_x + kb * kBlock;
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = ld_nc_v4(src + 8 * j);
    }
  };
  // two row buffers in turn: the next row's block is in flight while one row is
  // reduced and quantized, without copying registers between iterations
  const int step = gridDim.x;
  uint4 buf0[4], buf1[4];
  int row = blockIdx.x;
  load_row(row, buf0);
  for (; row < rows; row += 2 * step) {
    load_row(row + step, buf1);
    process_row(row, buf0);
    if (row + step >= rows) break;
    load_row(row + 2 * step, buf0);
    process_row(row + step, buf1);
  }

  // Zero the scale words of the padding rows (rows .. rows rounded up to 128).
  const int64_t kcs = k / kAtomK;
  const int64_t pad_words = (pad_rows(rows) - rows) * kcs;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < pad_words;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = rows + i / kcs;
    const int64_t kc = i % kcs;
    *reinterpret_cast<uint32_t*>(scales + scale_word_offset(r, kc, k)) = 0u;
  }
}

int norm_quantize_max_k() { return kNormMaxWarps * 1024; }

cudaError_t launch_norm_modulate_quantize(const void* x, int64_t rows, int64_t k, int64_t ld_x, const void* shift,
                                          const void* scale, float eps, void* codes, void* scales, float* dbg,
                                          int num_sms, cudaStream_t stream, unsigned* zero_words, int zero_count) {
  if (k % kAtomK != 0 || k > norm_quantize_max_k() || rows > (int64_t{1} << 31) - 1) return cudaErrorInvalidValue;
  const int warps = static_cast<int>((k / kBlock + 31) / 32);
  const int threads = 32 * warps;
  auto kern = dbg != nullptr ? norm_modulate_quantize_kernel<true> : norm_modulate_quantize_kernel<false>;
  // as many CTAs as are resident at once (each walks rows with a grid stride)
  static std::atomic<int> resident[64][2][kNormMaxWarps + 1];   // any thread may fill it
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const int di = dbg != nullptr ? 1 : 0;
  int per_sm = (dev >= 0 && dev < 64) ? resident[dev][di][warps].load(std::memory_order_relaxed) : 0;
  if (per_sm == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0);
    if (e != cudaSuccess || per_sm < 1) per_sm = 1;
    if (dev >= 0 && dev < 64) resident[dev][di][warps].store(per_sm, std::memory_order_relaxed);
  }
  int64_t blocks = static_cast<int64_t>(num_sms) * per_sm;
  const int64_t pad_blocks = ((pad_rows(rows) - rows) * (k / kAtomK) + threads - 1) / threads;
  if (blocks > rows) blocks = rows;
  if (blocks < pad_blocks) blocks = pad_blocks;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t*>(x), static_cast<int>(rows),
                                     static_cast<int>(k), ld_x, static_cast<const uint16_t*>(shift),
                                     static_cast<const uint16_t*>(scale), eps, static_cast<uint8_t*>(codes),
                                     static_cast<uint8_t*>(scales), dbg, zero_words, zero_words ? zero_count : 0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mxk
