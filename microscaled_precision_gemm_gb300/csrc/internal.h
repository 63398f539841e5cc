// Internal launchers shared between the kernel translation units and the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace mxk {

// Bits of the device-side error word (read by mx_device_error).
enum : unsigned {
  kErrWaitProducer = 1u << 0,   // TMA producer gave up waiting for a free stage
  kErrWaitMma = 1u << 1,        // MMA issuer gave up waiting for operands / accumulator
  kErrWaitEpilogue = 1u << 2,   // epilogue gave up waiting for the accumulator
  kErrDrain = 1u << 3,          // copies or MMAs still in flight after an abort
  kErrSelfTest = 1u << 4,       // the deliberate timeout of mx_selftest_wait_timeout
};

cudaError_t launch_quantize_bf16(const void* x, int64_t rows, int64_t k, int64_t ld_x, void* codes, void* scales,
                                 int num_sms, cudaStream_t stream);

// Fused RMSNorm + modulation + MXFP6 quantization (K <= norm_quantize_max_k()).
int norm_quantize_max_k();
cudaError_t launch_norm_modulate_quantize(const void* x, int64_t rows, int64_t k, int64_t ld_x, const void* shift,
                                          const void* scale, float eps, void* codes, void* scales, float* dbg,
                                          int num_sms, cudaStream_t stream);

struct GemmArgs {
  const void* a_codes;
  const void* a_scales;
  const void* b_codes;
  const void* b_scales;
  const void* bias;        // bf16 [N] or null
  const void* gate;        // bf16 [N] or null (epilogue 3 only; null = 1)
  const void* residual;    // bf16 [M][N] (epilogue 3 only; may equal out)
  void* out;               // bf16 [M][N] or packed codes [M][3F/4]
  void* out_scales;        // tiled scales of the MXFP6 output
  float* debug_prequant;   // fp32 [M][F] or null (MXFP6 epilogues only)
  int64_t m, n, k;         // n: rows of B (2F for the stacked gate/up weight)
  int epilogue;            // 0: bias + BF16, 1: bias + GELU + MXFP6, 2: bias + SwiGLU + MXFP6
                           // (F = N/2 outputs), 3: residual + gate * (C + bias), BF16
};

// Returns cudaSuccess or the first CUDA error; `encode_failed` is set when the
// tensor-map encoder rejected the operands.
cudaError_t launch_gemm(const GemmArgs& args, int num_sms, cudaStream_t stream, bool* encode_failed);

cudaError_t launch_wait_selftest(cudaStream_t stream);

// Reads (and optionally clears) the device error word of the current device.
cudaError_t read_device_error(unsigned* flags, bool clear);

}  // namespace mxk
