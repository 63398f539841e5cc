// C ABI (include/mx.h): argument validation, device checks and the three-launch
// MLP orchestration. Everything here is host code; the arithmetic lives in the
// kernels (quantize.cu, gemm.cu).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "mx.h"
#include "mx_layout.cuh"

namespace {

constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;
constexpr int kMaxDevices = 64;

std::atomic<int> g_device_ok[kMaxDevices];   // 0 unknown, 1 sm_103, -1 other
std::atomic<int> g_device_sms[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Checks the current device once per device; fills the SM count.
mx_status device_check(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MX_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MX_ERR_UNSUPPORTED_DEVICE;
  int state = g_device_ok[dev].load(std::memory_order_relaxed);
  if (state == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MX_ERR_CUDA;
    state = (major == 10 && minor == 3) ? 1 : -1;
    g_device_sms[dev].store(sms, std::memory_order_relaxed);
    g_device_ok[dev].store(state, std::memory_order_relaxed);
  }
  if (state != 1) return MX_ERR_UNSUPPORTED_DEVICE;
  *num_sms = g_device_sms[dev].load(std::memory_order_relaxed);
  return MX_OK;
}

mx_status check_quantize(const void* x, int64_t rows, int64_t K, int64_t ld_x, const void* codes,
                         const void* scales) {
  if (rows < 0 || K < 0 || ld_x < K) return MX_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || K > kMaxDim || rows > kMaxDim || ld_x > (int64_t{1} << 40))
    return MX_ERR_UNSUPPORTED_SHAPE;
  if (ld_x % 8 != 0) return MX_ERR_MISALIGNED;
  if (rows * (K / 32) > (int64_t{1} << 32) - (int64_t{1} << 28)) return MX_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MX_OK;
  if (x == nullptr || codes == nullptr || scales == nullptr) return MX_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 32) || !aligned(scales, 16)) return MX_ERR_MISALIGNED;
  return MX_OK;
}

mx_status check_norm_quantize(const void* x, int64_t rows, int64_t K, int64_t ld_x, const void* shift,
                              const void* scale, float eps, const void* codes, const void* scales, const float* dbg) {
  if (!(eps >= 0.0f) || eps > 3.0e38f) return MX_ERR_INVALID_ARG;   // negative, NaN or infinite
  mx_status st = check_quantize(x, rows, K, ld_x, codes, scales);
  if (st != MX_OK) return st;
  if (K > mxk::norm_quantize_max_k()) return MX_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return MX_OK;
  if ((shift != nullptr && !aligned(shift, 16)) || (scale != nullptr && !aligned(scale, 16)) ||
      (dbg != nullptr && !aligned(dbg, 16)))
    return MX_ERR_MISALIGNED;
  return MX_OK;
}

// epi: an mx_epilogue value; MX_EPI_GATE_RESIDUAL_BF16 only through mx_gemm_gate_residual,
// mx_quantize_gemm and the DiT block.
constexpr int kEpiGateResidual = MX_EPI_GATE_RESIDUAL_BF16;

bool mxfp6_out(int epi) { return epi == MX_EPI_BIAS_GELU_MXFP6 || epi == MX_EPI_BIAS_SWIGLU_MXFP6; }

mx_status check_gemm(const void* a_codes, const void* a_scales, const void* b_codes, const void* b_scales,
                     const void* bias, int64_t M, int64_t N, int64_t K, int epi, const void* out,
                     const void* out_scales, const float* dbg) {
  if (epi != MX_EPI_BIAS_BF16 && epi != MX_EPI_BIAS_GELU_MXFP6 && epi != MX_EPI_BIAS_SWIGLU_MXFP6 &&
      epi != kEpiGateResidual)
    return MX_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return MX_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N % 256 != 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MX_ERR_UNSUPPORTED_SHAPE;
  if (((M + 127) / 128) * (N / 256) > kMaxDim) return MX_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return MX_OK;
  if (a_codes == nullptr || a_scales == nullptr || b_codes == nullptr || b_scales == nullptr || out == nullptr)
    return MX_ERR_INVALID_ARG;
  if (mxfp6_out(epi) && out_scales == nullptr) return MX_ERR_INVALID_ARG;
  if (!aligned(a_codes, 32) || !aligned(b_codes, 32) || !aligned(a_scales, 16) || !aligned(b_scales, 16))
    return MX_ERR_MISALIGNED;
  if (bias != nullptr && !aligned(bias, 16)) return MX_ERR_MISALIGNED;
  if (!mxfp6_out(epi) && !aligned(out, 16)) return MX_ERR_MISALIGNED;
  if (mxfp6_out(epi) && (!aligned(out, 32) || !aligned(out_scales, 16))) return MX_ERR_MISALIGNED;
  if (mxfp6_out(epi) && dbg != nullptr && !aligned(dbg, 16)) return MX_ERR_MISALIGNED;
  return MX_OK;
}

// MLP workspace: xq | xs | hq | hs | the in-kernel quantizer's row-block counters,
// then the split-tail region both GEMMs use in turn (the first kernel zeroes the
// counters and the split tail's arrival counters, which are contiguous). `base` is
// the smallest workspace the MLP runs with (no split tail), `total` the one
// mx_mlp_workspace_bytes reports.
struct MlpLayout {
  size_t xq, xs, hq, hs, ready, split, base, total;
};

MlpLayout mlp_layout(int64_t M, int64_t d, int64_t ff) {
  MlpLayout l;
  l.xq = 0;
  l.xs = align256(l.xq + static_cast<size_t>(mxk::codes_bytes(M, d)));
  l.hq = align256(l.xs + static_cast<size_t>(mxk::scales_bytes(M, d)));
  l.hs = align256(l.hq + static_cast<size_t>(mxk::codes_bytes(M, ff)));
  l.ready = align256(l.hs + static_cast<size_t>(mxk::scales_bytes(M, ff)));
  l.split = align256(l.ready + 4 * static_cast<size_t>(mxk::qa_counter_words(M)));
  l.base = l.split;
  // the up-projection is at most 2 ff wide (the stacked gate/up weight)
  const size_t up = mxk::split_workspace_bytes(M, 2 * ff, d), down = mxk::split_workspace_bytes(M, d, ff);
  l.total = align256(l.split + (up > down ? up : down));
  return l;
}

// In-kernel quantizer of a GEMM launch (x null: none): A = MXFP6(x) goes to the
// A operand's buffers; rows below lead_rows are there already and the counters
// `ready` are zero.
struct QaLaunch {
  const void* x = nullptr;
  int64_t ld_x = 0;
  int64_t lead_rows = 0;
  unsigned* ready = nullptr;
};

// split_ws: split-tail workspace (arrival counters zero) or null.
mx_status gemm_launch(const void* a_codes, const void* a_scales, const void* b_codes, const void* b_scales,
                      const void* bias, int64_t M, int64_t N, int64_t K, int epi, void* out, void* out_scales,
                      float* dbg, int num_sms, cudaStream_t stream, void* split_ws, size_t split_bytes,
                      const void* gate = nullptr, const void* residual = nullptr, const QaLaunch& qa = QaLaunch()) {
  if (M == 0 || N == 0) return MX_OK;
  mxk::GemmArgs a;
  a.a_codes = a_codes;
  a.a_scales = a_scales;
  a.b_codes = b_codes;
  a.b_scales = b_scales;
  a.bias = bias;
  a.gate = gate;
  a.residual = residual;
  a.out = out;
  a.out_scales = out_scales;
  a.debug_prequant = mxfp6_out(epi) ? dbg : nullptr;
  a.m = M;
  a.n = N;
  a.k = K;
  a.epilogue = epi;
  a.workspace = split_ws;
  a.workspace_bytes = split_ws != nullptr ? split_bytes : 0;
  a.x = qa.x;
  a.ld_x = qa.ld_x;
  a.lead_rows = qa.lead_rows;
  a.ready = qa.ready;
  bool encode_failed = false;
  cudaError_t e = mxk::launch_gemm(a, num_sms, stream, &encode_failed);
  if (encode_failed) return MX_ERR_CUDA;
  return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

// The MLP's workspace cut into its parts: MXFP6 x, MXFP6 h, and the split-tail
// region when the workspace holds it (its first kernel zeroes the arrival counters).
struct MlpWorkspace {
  void* xq;
  void* xs;
  void* hq;
  void* hs;
  unsigned* ready;      // the in-kernel quantizer's row-block counters
  void* split;          // null: the GEMMs run unsplit
  size_t split_bytes;
  unsigned* zero;       // the counter words the first kernel zeroes
  int zero_count;
};

mx_status slice_mlp_workspace(int64_t M, int64_t d, int64_t ff, void* workspace, size_t workspace_bytes,
                              MlpWorkspace* w) {
  if (workspace == nullptr) return MX_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return MX_ERR_MISALIGNED;
  const MlpLayout l = mlp_layout(M, d, ff);
  if (workspace_bytes < l.base) return MX_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  w->xq = ws + l.xq;
  w->xs = ws + l.xs;
  w->hq = ws + l.hq;
  w->hs = ws + l.hs;
  // the split tail runs when the workspace holds its region (mx_mlp_workspace_bytes)
  w->ready = reinterpret_cast<unsigned*>(ws + l.ready);
  w->split = workspace_bytes >= l.total && l.total > l.base ? ws + l.split : nullptr;
  w->split_bytes = w->split != nullptr ? workspace_bytes - l.split : 0;
  // the row-block counters, and the split tail's arrival counters right after them
  w->zero = w->ready;
  w->zero_count = static_cast<int>(((w->split != nullptr ? l.split + mxk::kArrivalsBytes : l.split) - l.ready) /
                                   sizeof(unsigned));
  return MX_OK;
}

// K1 -> up-projection (GELU, or SwiGLU on the stacked gate/up weight) -> K2.
mx_status mlp_impl(const void* x, int64_t M, int64_t d, int64_t ff, int up_epi, const void* w_up_codes,
                   const void* w_up_scales, const void* b_up, const void* w2_codes, const void* w2_scales,
                   const void* b2, void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  mx_status st = mxk::mlp_check_shape(M, d, ff, up_epi == MX_EPI_BIAS_SWIGLU_MXFP6);
  if (st != MX_OK) return st;
  const int64_t n_up = up_epi == MX_EPI_BIAS_SWIGLU_MXFP6 ? 2 * ff : ff;
  if (M == 0) return MX_OK;
  if (x == nullptr || w_up_codes == nullptr || w_up_scales == nullptr || w2_codes == nullptr ||
      w2_scales == nullptr || y == nullptr)
    return MX_ERR_INVALID_ARG;
  MlpWorkspace w;
  if ((st = slice_mlp_workspace(M, d, ff, workspace, workspace_bytes, &w)) != MX_OK) return st;
  st = check_quantize(x, M, d, d, w.xq, w.xs);
  if (st != MX_OK) return st;
  st = check_gemm(w.xq, w.xs, w_up_codes, w_up_scales, b_up, M, n_up, d, up_epi, w.hq, w.hs, nullptr);
  if (st != MX_OK) return st;
  st = check_gemm(w.hq, w.hs, w2_codes, w2_scales, b2, M, d, ff, MX_EPI_BIAS_BF16, y, nullptr, nullptr);
  if (st != MX_OK) return st;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  // the up-projection quantizes x itself beyond the rows its first round of
  // tiles reads, which the quantize kernel encodes first (unless the up-projection
  // splits its tail, or those rows are all of x)
  QaLaunch qa;
  int clusters = 0;
  if (mxk::gemm_max_clusters(&clusters) != cudaSuccess) return MX_ERR_CUDA;
  const int64_t lead = mxk::qa_lead_rows(M, n_up, clusters);
  if (lead < M && mxk::plan_gemm(M, n_up, d, clusters, w.split, w.split_bytes).sk_tiles == 0) {
    qa.x = x;
    qa.ld_x = d;
    qa.lead_rows = lead;
    qa.ready = w.ready;
  }
  if (mxk::launch_quantize_bf16(x, qa.x != nullptr ? lead : M, d, d, w.xq, w.xs, sms, stream, w.zero,
                                w.zero_count) != cudaSuccess)
    return MX_ERR_CUDA;
  st = gemm_launch(w.xq, w.xs, w_up_codes, w_up_scales, b_up, M, n_up, d, up_epi, w.hq, w.hs, nullptr, sms, stream,
                   w.split, w.split_bytes, nullptr, nullptr, qa);
  if (st != MX_OK) return st;
  // the up-projection leaves the arrival counters at zero again
  return gemm_launch(w.hq, w.hs, w2_codes, w2_scales, b2, M, d, ff, MX_EPI_BIAS_BF16, y, nullptr, nullptr, sms,
                     stream, w.split, w.split_bytes);
}

// The MLP half of a DiT block: fused norm quantizer -> up-projection -> down-projection
// with gate and residual (the residual is x itself).
mx_status dit_block_impl(const void* x, int64_t M, int64_t d, int64_t ff, const void* shift, const void* scale,
                         const void* gate, float eps, int activation, const void* w_up_codes, const void* w_up_scales,
                         const void* b_up, const void* w2_codes, const void* w2_scales, const void* b2, void* y,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (M < 0 || d < 0 || ff < 0) return MX_ERR_INVALID_ARG;
  if (activation != MX_ACT_GELU_TANH && activation != MX_ACT_SWIGLU) return MX_ERR_INVALID_ARG;
  const int up_epi = activation == MX_ACT_SWIGLU ? MX_EPI_BIAS_SWIGLU_MXFP6 : MX_EPI_BIAS_GELU_MXFP6;
  const int64_t n_up = activation == MX_ACT_SWIGLU ? 2 * ff : ff;
  mx_status st = mxk::mlp_check_shape(M, d, ff, activation == MX_ACT_SWIGLU);
  if (st != MX_OK) return st;
  if (M == 0) return MX_OK;
  if (x == nullptr || w_up_codes == nullptr || w_up_scales == nullptr || w2_codes == nullptr ||
      w2_scales == nullptr || y == nullptr)
    return MX_ERR_INVALID_ARG;
  MlpWorkspace w;
  if ((st = slice_mlp_workspace(M, d, ff, workspace, workspace_bytes, &w)) != MX_OK) return st;
  st = check_norm_quantize(x, M, d, d, shift, scale, eps, w.xq, w.xs, nullptr);
  if (st != MX_OK) return st;
  st = check_gemm(w.xq, w.xs, w_up_codes, w_up_scales, b_up, M, n_up, d, up_epi, w.hq, w.hs, nullptr);
  if (st != MX_OK) return st;
  st = check_gemm(w.hq, w.hs, w2_codes, w2_scales, b2, M, d, ff, kEpiGateResidual, y, nullptr, nullptr);
  if (st != MX_OK) return st;
  if (gate != nullptr && !aligned(gate, 16)) return MX_ERR_MISALIGNED;
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), y0 = reinterpret_cast<uintptr_t>(y);
  const uintptr_t bytes = static_cast<uintptr_t>(M) * static_cast<uintptr_t>(d) * 2u;
  if (x0 != y0 && x0 < y0 + bytes && y0 < x0 + bytes) return MX_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  if (mxk::launch_norm_modulate_quantize(x, M, d, d, shift, scale, eps, w.xq, w.xs, nullptr, sms, stream, w.zero,
                                         w.zero_count) != cudaSuccess)
    return MX_ERR_CUDA;
  st = gemm_launch(w.xq, w.xs, w_up_codes, w_up_scales, b_up, M, n_up, d, up_epi, w.hq, w.hs, nullptr, sms, stream,
                   w.split, w.split_bytes);
  if (st != MX_OK) return st;
  return gemm_launch(w.hq, w.hs, w2_codes, w2_scales, b2, M, d, ff, kEpiGateResidual, y, nullptr, nullptr, sms,
                     stream, w.split, w.split_bytes, gate, x);
}

// mx_quantize_gemm's workspace: MXFP6(x) codes | tiled scales | row-block counters.
struct QgLayout {
  size_t xs, ready, total;
};

QgLayout qg_layout(int64_t M, int64_t K) {
  QgLayout l;
  l.xs = align256(static_cast<size_t>(mxk::codes_bytes(M, K)));
  l.ready = align256(l.xs + static_cast<size_t>(mxk::scales_bytes(M, K)));
  l.total = align256(l.ready + 4 * static_cast<size_t>(mxk::qa_counter_words(M)));
  return l;
}

bool overlaps(const void* a, uintptr_t a_bytes, const void* b, uintptr_t b_bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  const uintptr_t a1 = a_bytes > UINTPTR_MAX - a0 ? UINTPTR_MAX : a0 + a_bytes;
  const uintptr_t b1 = b_bytes > UINTPTR_MAX - b0 ? UINTPTR_MAX : b0 + b_bytes;
  return a0 < b1 && b0 < a1;
}

// x * y (both >= 0), saturated at UINTPTR_MAX: a byte span that cannot exist
// overlaps everything rather than wrapping around.
uintptr_t mul_sat(uint64_t x, uint64_t y) {
  if (x != 0 && y > UINTPTR_MAX / x) return UINTPTR_MAX;
  return static_cast<uintptr_t>(x * y);
}

}  // namespace

namespace mxk {
mx_status mlp_check_shape(int64_t M, int64_t d, int64_t ff, bool swiglu) {
  if (M < 0 || d < 0 || ff < 0) return MX_ERR_INVALID_ARG;
  const int64_t n_up = swiglu ? 2 * ff : ff;
  if (d == 0 || ff == 0 || d % 256 != 0 || ff % 128 != 0 || n_up % 256 != 0 || M > kMaxDim || d > kMaxDim ||
      n_up > kMaxDim)
    return MX_ERR_UNSUPPORTED_SHAPE;
  return MX_OK;
}

size_t mlp_min_workspace_bytes(int64_t M, int64_t d, int64_t ff) {
  if (M < 0 || d < 0 || ff < 0) return 0;
  return mlp_layout(M, d, ff).base;
}

bool current_context_id(unsigned long long* id) {
  typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
  typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    void* q = nullptr;
    cudaDriverEntryPointQueryResult r1, r2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &r1) == cudaSuccess &&
        r1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &q, 12000, cudaEnableDefault, &r2) == cudaSuccess &&
        r2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
      get_id = reinterpret_cast<CtxGetIdFn>(q);
    }
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}
}  // namespace mxk

extern "C" {

size_t mx_codes_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return static_cast<size_t>(mxk::codes_bytes(rows, K));
}

size_t mx_scales_bytes(int64_t rows, int64_t K) {
  if (rows < 0 || K < 0) return 0;
  return static_cast<size_t>(mxk::scales_bytes(rows, K));
}

mx_status mx_quantize(const void* x, int64_t rows, int64_t K, int64_t ld_x, void* codes, void* scales,
                      cudaStream_t stream) {
  mx_status st = check_quantize(x, rows, K, ld_x, codes, scales);
  if (st != MX_OK || rows == 0) return st;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  return mxk::launch_quantize_bf16(x, rows, K, ld_x, codes, scales, sms, stream) == cudaSuccess ? MX_OK
                                                                                                : MX_ERR_CUDA;
}

mx_status mx_quantize_stacked(const void* const* x_parts, const int64_t* part_rows, const int64_t* ld_x, int n_parts,
                              int64_t K, void* codes, void* scales, cudaStream_t stream) {
  if (x_parts == nullptr || part_rows == nullptr || n_parts < 1) return MX_ERR_INVALID_ARG;
  // every part is checked before anything is launched
  int64_t total = 0;
  for (int i = 0; i < n_parts; ++i) {
    const int64_t r = part_rows[i];
    const int64_t ld = ld_x != nullptr ? ld_x[i] : K;
    if (r < 0) return MX_ERR_INVALID_ARG;
    if (i + 1 < n_parts && r % 128 != 0) return MX_ERR_UNSUPPORTED_SHAPE;   // parts start on a scale atom
    if (total > kMaxDim - r) return MX_ERR_UNSUPPORTED_SHAPE;
    // the part's own checks, at its place in the stacked buffers (32-byte aligned
    // codes: a row offset that is a multiple of 128 keeps the stacked base's alignment)
    const mx_status st = check_quantize(x_parts[i], r, K, ld, codes, scales);
    if (st != MX_OK) return st;
    total += r;
  }
  if (total == 0) return MX_OK;
  // the stacked tensor's own size limit (the parts were each within it)
  if (total * (K / 32) > (int64_t{1} << 32) - (int64_t{1} << 28)) return MX_ERR_UNSUPPORTED_SHAPE;
  mx_status st = MX_OK;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  int64_t r0 = 0;
  for (int i = 0; i < n_parts; ++i) {
    const int64_t r = part_rows[i];
    const int64_t ld = ld_x != nullptr ? ld_x[i] : K;
    if (r > 0 && mxk::launch_quantize_bf16(x_parts[i], r, K, ld, static_cast<uint8_t*>(codes) + mxk::codes_bytes(r0, K),
                                           static_cast<uint8_t*>(scales) + mxk::scales_bytes(r0, K), sms,
                                           stream) != cudaSuccess)
      return MX_ERR_CUDA;
    r0 += r;
  }
  return MX_OK;
}

mx_status mx_quantize_rmsnorm_modulate(const void* x, int64_t rows, int64_t K, int64_t ld_x, const void* shift,
                                       const void* scale, float eps, void* codes, void* scales, float* debug_y,
                                       cudaStream_t stream) {
  mx_status st = check_norm_quantize(x, rows, K, ld_x, shift, scale, eps, codes, scales, debug_y);
  if (st != MX_OK || rows == 0) return st;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  return mxk::launch_norm_modulate_quantize(x, rows, K, ld_x, shift, scale, eps, codes, scales, debug_y, sms,
                                            stream) == cudaSuccess
             ? MX_OK
             : MX_ERR_CUDA;
}

mx_status mx_gemm(const void* a_codes, const void* a_scales, const void* b_codes, const void* b_scales,
                  const void* bias, int64_t M, int64_t N, int64_t K, mx_epilogue epi, void* out,
                  void* out_scales, float* debug_prequant, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream) {
  if (static_cast<int>(epi) == kEpiGateResidual) return MX_ERR_INVALID_ARG;  // needs mx_gemm_gate_residual
  mx_status st = check_gemm(a_codes, a_scales, b_codes, b_scales, bias, M, N, K, static_cast<int>(epi), out,
                            out_scales, debug_prequant);
  if (st != MX_OK || M == 0 || N == 0) return st;
  if (workspace != nullptr && !aligned(workspace, 256)) return MX_ERR_MISALIGNED;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  return gemm_launch(a_codes, a_scales, b_codes, b_scales, bias, M, N, K, static_cast<int>(epi), out, out_scales,
                     debug_prequant, sms, stream, workspace, workspace_bytes);
}

mx_status mx_gemm_gate_residual(const void* a_codes, const void* a_scales, const void* b_codes,
                                const void* b_scales, const void* bias, const void* gate, const void* residual,
                                int64_t M, int64_t N, int64_t K, void* out, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  mx_status st = check_gemm(a_codes, a_scales, b_codes, b_scales, bias, M, N, K, kEpiGateResidual, out, nullptr,
                            nullptr);
  if (st != MX_OK || M == 0 || N == 0) return st;
  if (residual == nullptr) return MX_ERR_INVALID_ARG;
  if (!aligned(residual, 16) || (gate != nullptr && !aligned(gate, 16))) return MX_ERR_MISALIGNED;
  // the residual may be the output itself (in-place update), but not overlap it otherwise
  const uintptr_t r0 = reinterpret_cast<uintptr_t>(residual), o0 = reinterpret_cast<uintptr_t>(out);
  const uintptr_t bytes = static_cast<uintptr_t>(M) * static_cast<uintptr_t>(N) * 2u;
  if (r0 != o0 && r0 < o0 + bytes && o0 < r0 + bytes) return MX_ERR_INVALID_ARG;
  if (workspace != nullptr && !aligned(workspace, 256)) return MX_ERR_MISALIGNED;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  return gemm_launch(a_codes, a_scales, b_codes, b_scales, bias, M, N, K, kEpiGateResidual, out, nullptr, nullptr,
                     sms, stream, workspace, workspace_bytes, gate, residual);
}

size_t mx_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || N % 256 != 0 || K % 128 != 0) return 0;
  return mxk::split_workspace_bytes(M, N, K);
}

mx_status mx_gemm_launch_plan(int64_t M, int64_t N, int64_t K, size_t workspace_bytes, int* pairs,
                              int* split_tiles) {
  if (pairs == nullptr || split_tiles == nullptr || M < 0 || N < 0 || K < 0) return MX_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N % 256 != 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return MX_ERR_UNSUPPORTED_SHAPE;
  *pairs = 0;
  *split_tiles = 0;
  if (M == 0 || N == 0) return MX_OK;
  int sms = 0;
  mx_status st = device_check(&sms);
  if (st != MX_OK) return st;
  int clusters = 0;
  if (mxk::gemm_max_clusters(&clusters) != cudaSuccess) return MX_ERR_CUDA;
  // any non-null pointer: only the size decides
  const mxk::GemmPlan p = mxk::plan_gemm(M, N, K, clusters, workspace_bytes > 0 ? &clusters : nullptr,
                                         workspace_bytes);
  *pairs = p.clusters;
  *split_tiles = p.sk_tiles;
  return MX_OK;
}

size_t mx_quantize_gemm_workspace_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  return qg_layout(M, K).total;
}

mx_status mx_quantize_gemm(const void* x, int64_t M, int64_t K, int64_t ld_x, const void* b_codes,
                           const void* b_scales, const void* bias, int64_t N, mx_epilogue epi, const void* gate,
                           const void* residual, void* out, void* out_scales, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  const int e = static_cast<int>(epi);
  if (e < MX_EPI_BIAS_BF16 || e > MX_EPI_GATE_RESIDUAL_BF16) return MX_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || ld_x < K) return MX_ERR_INVALID_ARG;
  const QgLayout l = qg_layout(M, K);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // the shape and pointer rules of mx_quantize and of the GEMM, on the workspace's parts
  const bool empty = M == 0 || N == 0;
  void* xq = empty ? nullptr : ws;
  void* xs = empty ? nullptr : ws + l.xs;
  mx_status st = check_quantize(x, empty ? 0 : M, K, ld_x, xq, xs);
  if (st != MX_OK) return st;
  st = check_gemm(xq, xs, b_codes, b_scales, bias, M, N, K, e, out, out_scales, nullptr);
  if (st != MX_OK || empty) return st;
  if (workspace == nullptr) return MX_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return MX_ERR_MISALIGNED;
  if (workspace_bytes < l.total) return MX_ERR_WORKSPACE_TOO_SMALL;
  // byte spans of x (rows of ld_x elements, the last one K) and of the output
  const uintptr_t x_rows = mul_sat(static_cast<uint64_t>(M - 1), static_cast<uint64_t>(ld_x));
  const uintptr_t x_bytes = mul_sat(x_rows > UINTPTR_MAX - static_cast<uint64_t>(K) ? UINTPTR_MAX : x_rows + K, 2);
  const uint64_t w_out = e == MX_EPI_BIAS_SWIGLU_MXFP6 ? N / 2 : N;
  const uintptr_t out_bytes = mxfp6_out(e) ? mul_sat(mul_sat(static_cast<uint64_t>(M), w_out), 3) / 4
                                           : mul_sat(mul_sat(static_cast<uint64_t>(M), static_cast<uint64_t>(N)), 2);
  if (e == MX_EPI_GATE_RESIDUAL_BF16) {
    if (residual == nullptr) return MX_ERR_INVALID_ARG;
    if (!aligned(residual, 16) || (gate != nullptr && !aligned(gate, 16))) return MX_ERR_MISALIGNED;
    // the residual may be the output itself (in-place update), but not overlap it
    // otherwise, nor the workspace the GEMM writes MXFP6(x) into
    if (residual != out && overlaps(residual, out_bytes, out, out_bytes)) return MX_ERR_INVALID_ARG;
    if (overlaps(residual, out_bytes, workspace, l.total)) return MX_ERR_INVALID_ARG;
  }
  // x is read while the output and the workspace are written
  if (overlaps(x, x_bytes, out, out_bytes) || overlaps(x, x_bytes, workspace, l.total) ||
      overlaps(out, out_bytes, workspace, l.total))
    return MX_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = device_check(&sms)) != MX_OK) return st;
  int clusters = 0;
  if (mxk::gemm_max_clusters(&clusters) != cudaSuccess) return MX_ERR_CUDA;
  // the quantize kernel encodes the rows the first round of tiles reads and
  // zeroes the counters; the GEMM encodes the rest itself
  QaLaunch qa;
  const int64_t lead = mxk::qa_lead_rows(M, N, clusters);
  unsigned* ready = reinterpret_cast<unsigned*>(ws + l.ready);
  if (lead < M) {
    qa.x = x;
    qa.ld_x = ld_x;
    qa.lead_rows = lead;
    qa.ready = ready;
  }
  if (mxk::launch_quantize_bf16(x, lead, K, ld_x, xq, xs, sms, stream, ready,
                                static_cast<int>(mxk::qa_counter_words(M))) != cudaSuccess)
    return MX_ERR_CUDA;
  const bool gr = e == MX_EPI_GATE_RESIDUAL_BF16;
  return gemm_launch(xq, xs, b_codes, b_scales, bias, M, N, K, e, out, mxfp6_out(e) ? out_scales : nullptr, nullptr,
                     sms, stream, nullptr, 0, gr ? gate : nullptr, gr ? residual : nullptr, qa);
}

size_t mx_mlp_workspace_bytes(int64_t M, int64_t d, int64_t ff) {
  if (M < 0 || d < 0 || ff < 0) return 0;
  return mlp_layout(M, d, ff).total;
}

mx_status mx_mlp(const void* x, int64_t M, int64_t d, int64_t ff, const void* w1_codes, const void* w1_scales,
                 const void* b1, const void* w2_codes, const void* w2_scales, const void* b2, void* y,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return mlp_impl(x, M, d, ff, MX_EPI_BIAS_GELU_MXFP6, w1_codes, w1_scales, b1, w2_codes, w2_scales, b2, y,
                  workspace, workspace_bytes, stream);
}

mx_status mx_gated_mlp(const void* x, int64_t M, int64_t d, int64_t ff, const void* wgu_codes,
                       const void* wgu_scales, const void* bgu, const void* w2_codes, const void* w2_scales,
                       const void* b2, void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return mlp_impl(x, M, d, ff, MX_EPI_BIAS_SWIGLU_MXFP6, wgu_codes, wgu_scales, bgu, w2_codes, w2_scales, b2, y,
                  workspace, workspace_bytes, stream);
}

mx_status mx_dit_mlp_block(const void* x, int64_t M, int64_t d, int64_t ff, const void* shift, const void* scale,
                           const void* gate, float eps, mx_activation activation, const void* w_up_codes,
                           const void* w_up_scales, const void* b_up, const void* w2_codes, const void* w2_scales,
                           const void* b2, void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return dit_block_impl(x, M, d, ff, shift, scale, gate, eps, static_cast<int>(activation), w_up_codes, w_up_scales,
                        b_up, w2_codes, w2_scales, b2, y, workspace, workspace_bytes, stream);
}

const char* mx_status_string(mx_status status) {
  switch (status) {
    case MX_OK: return "MX_OK";
    case MX_ERR_INVALID_ARG: return "MX_ERR_INVALID_ARG: null pointer, negative size or bad enum";
    case MX_ERR_UNSUPPORTED_SHAPE: return "MX_ERR_UNSUPPORTED_SHAPE: need K % 128 == 0, N % 256 == 0, sizes < 2^31";
    case MX_ERR_MISALIGNED: return "MX_ERR_MISALIGNED: codes need 32-byte, other buffers 16-byte alignment";
    case MX_ERR_WORKSPACE_TOO_SMALL: return "MX_ERR_WORKSPACE_TOO_SMALL: see mx_mlp_workspace_bytes";
    case MX_ERR_UNSUPPORTED_DEVICE: return "MX_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
    case MX_ERR_CUDA: return "MX_ERR_CUDA: a CUDA call or kernel launch failed";
  }
  return "unknown mx_status";
}

mx_status mx_scales_to_plain(const void* tiled_host, void* plain_host, int64_t rows, int64_t K) {
  if (tiled_host == nullptr || plain_host == nullptr || rows < 0 || K < 0) return MX_ERR_INVALID_ARG;
  if (K % 128 != 0) return MX_ERR_UNSUPPORTED_SHAPE;
  const uint8_t* t = static_cast<const uint8_t*>(tiled_host);
  uint8_t* p = static_cast<uint8_t*>(plain_host);
  const int64_t kb = K / 32;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < kb; ++b) p[r * kb + b] = t[mxk::scale_word_offset(r, b / 4, K) + (b % 4)];
  return MX_OK;
}

mx_status mx_scales_from_plain(const void* plain_host, void* tiled_host, int64_t rows, int64_t K) {
  if (tiled_host == nullptr || plain_host == nullptr || rows < 0 || K < 0) return MX_ERR_INVALID_ARG;
  if (K % 128 != 0) return MX_ERR_UNSUPPORTED_SHAPE;
  const uint8_t* p = static_cast<const uint8_t*>(plain_host);
  uint8_t* t = static_cast<uint8_t*>(tiled_host);
  const int64_t kb = K / 32;
  const int64_t padded = mxk::pad_rows(rows);
  for (int64_t r = 0; r < padded; ++r)
    for (int64_t b = 0; b < kb; ++b)
      t[mxk::scale_word_offset(r, b / 4, K) + (b % 4)] = r < rows ? p[r * kb + b] : 0;
  return MX_OK;
}

mx_status mx_device_error(unsigned* flags_host, int clear) {
  if (flags_host == nullptr) return MX_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return MX_ERR_CUDA;
  return mxk::read_device_error(flags_host, clear != 0) == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

mx_status mx_selftest_wait_timeout(cudaStream_t stream) {
  int sms = 0;
  mx_status st = device_check(&sms);
  if (st != MX_OK) return st;
  return mxk::launch_wait_selftest(stream) == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}

int mx_version(void) { return 100; }

}  // extern "C"
