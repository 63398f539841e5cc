// Internal launchers shared between the kernel translation units and the C ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "mx.h"

namespace mxk {

// Bits of the device-side error word (read by mx_device_error).
enum : unsigned {
  kErrWaitProducer = 1u << 0,   // TMA producer gave up waiting for a free stage
  kErrWaitMma = 1u << 1,        // MMA issuer gave up waiting for operands / accumulator
  kErrWaitEpilogue = 1u << 2,   // epilogue gave up waiting for the accumulator
  kErrDrain = 1u << 3,          // copies or MMAs still in flight after an abort
  kErrSelfTest = 1u << 4,       // the deliberate timeout of mx_selftest_wait_timeout
  kErrWaitQuant = 1u << 5,      // TMA producer gave up waiting for in-kernel quantized A rows
};

// zero_words / zero_count: a buffer the kernel also sets to zero (after the previous
// kernel in the stream has completed), e.g. the split-tail arrival counters of the
// GEMMs that follow; null / 0 for none.
cudaError_t launch_quantize_bf16(const void* x, int64_t rows, int64_t k, int64_t ld_x, void* codes, void* scales,
                                 int num_sms, cudaStream_t stream, unsigned* zero_words = nullptr,
                                 int zero_count = 0);

// Fused RMSNorm + modulation + MXFP6 quantization (K <= norm_quantize_max_k()).
int norm_quantize_max_k();
cudaError_t launch_norm_modulate_quantize(const void* x, int64_t rows, int64_t k, int64_t ld_x, const void* shift,
                                          const void* scale, float eps, void* codes, void* scales, float* dbg,
                                          int num_sms, cudaStream_t stream, unsigned* zero_words = nullptr,
                                          int zero_count = 0);

// ---------------------------------------------------------------- split tail
// The GEMM walks pair tiles of 256 x 256 outputs, 128 K-elements per step.
// When the tile count leaves only a small last round for the co-resident CTA
// pairs, most pairs would idle through it; with a workspace, the first
// pairs + (tiles mod pairs) tiles are instead divided along K so that every
// pair gets the same number of K-steps, and a tile two pairs share is summed
// through the workspace (gemm.cu). The split costs about a third of a long tile
// per pair (two more tile boundaries, the partial sums' stores and loads), so it
// is taken only where it wins on GB300 (measured): the leftover round at most a
// quarter full, and at least 32 K-steps (K >= 4096) per tile. Workspace layout
// (256-byte aligned):
//   [0, kArrivalsBytes)   arrival counters, one per (split tile, CTA, epilogue warp);
//                         zero before the launch (the caller's duty, or the MLP's
//                         first kernel), and zero again after it
//   [kArrivalsBytes, ...) partial accumulators, two 256 KB slots per pair
constexpr int kPairTileRows = 256;
constexpr int kPairTileCols = 256;
constexpr int kStepK = 128;
constexpr int kMaxSplitClusters = 80;             // pairs the workspace bound covers (GB300 runs 76)
constexpr int kMinSplitKSteps = 32;               // shorter tiles: the exchange costs more than it saves
constexpr int kMaxSplitLeftoverDiv = 4;           // split when tiles mod pairs <= pairs / 4
constexpr size_t kSplitSlotBytes = size_t{2} * 128 * 256 * 4;
constexpr int kArrivalWordsPerTile = 2 * 8;       // CTAs x epilogue warps
constexpr size_t kArrivalsBytes =
    ((size_t{2} * kMaxSplitClusters * kArrivalWordsPerTile * 4) + 255) / 256 * 256;
static_assert(kArrivalsBytes == MX_GEMM_WORKSPACE_COUNTER_BYTES, "counter bytes of the public header");

struct SplitArgs {
  int sk_tiles;          // tiles divided along K (0: none)
  float4* partial;       // partial-accumulator slots
  unsigned* arrivals;    // arrival counters
  int half_tiles;        // trailing tiles run as two 128-column halves (0: none)
};

struct GemmPlan {
  int64_t tiles;    // pair tiles
  int clusters;     // CTA pairs launched
  int sk_tiles;     // leading tiles divided along K
  int half_tiles;   // trailing tiles run as two 128-column halves
};

// ---------------------------------------------------------------- half tiles
// Without a split tail, the last round's tiles (tiles mod pairs of them, or all
// tiles when there are fewer than pairs) can run as two 128-column halves each,
// on twice as many pairs: a half moves 3/4 of a tile's operand bytes (all of its
// A rows, half of its B rows) for half the work, so a nearly empty last round
// ends sooner and its last epilogue is half as long. Taken when the halves fit in
// one round (at most pairs / 2 such tiles), for the epilogues with one output
// column per accumulator column (not the stacked SwiGLU weight).

inline int64_t gemm_pair_tiles(int64_t m, int64_t n) {
  return ((m + kPairTileRows - 1) / kPairTileRows) * (n / kPairTileCols);
}

inline size_t split_arrival_words(int sk_tiles) { return static_cast<size_t>(sk_tiles) * kArrivalWordsPerTile; }

// Workspace bytes that let a GEMM of this shape divide its tail (0: it never does;
// whether it does also depends on the device's pair count).
inline size_t split_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  const int64_t tiles = gemm_pair_tiles(m, n);
  if (k / kStepK < kMinSplitKSteps || tiles < 2) return 0;
  const int64_t pairs = tiles - 1 < kMaxSplitClusters ? tiles - 1 : kMaxSplitClusters;
  return kArrivalsBytes + static_cast<size_t>(2 * pairs) * kSplitSlotBytes;
}

// Launch plan: CTA pairs (co-resident ones, at most one per tile or half tile),
// the split tail, and the half tiles when halves_ok.
inline GemmPlan plan_gemm(int64_t m, int64_t n, int64_t k, int max_clusters, const void* workspace,
                          size_t workspace_bytes, bool halves_ok = false) {
  GemmPlan p;
  p.tiles = gemm_pair_tiles(m, n);
  p.clusters = static_cast<int>(max_clusters < p.tiles ? max_clusters : p.tiles);
  p.sk_tiles = 0;
  p.half_tiles = 0;
  const int64_t rem = p.clusters > 0 ? p.tiles % p.clusters : 0;
  if (workspace != nullptr && p.tiles > p.clusters && rem != 0 && rem * kMaxSplitLeftoverDiv <= p.clusters &&
      k / kStepK >= kMinSplitKSteps && p.clusters <= kMaxSplitClusters && (p.clusters + rem) * (k / kStepK) < (int64_t{1} << 31) &&
      workspace_bytes >= kArrivalsBytes + static_cast<size_t>(2 * p.clusters) * kSplitSlotBytes)
    p.sk_tiles = static_cast<int>(p.clusters + rem);
  if (halves_ok && p.sk_tiles == 0 && p.tiles > 0) {
    if (p.tiles > max_clusters) {
      if (rem != 0 && 2 * rem <= p.clusters) p.half_tiles = static_cast<int>(rem);
    } else if (2 * p.tiles <= max_clusters) {
      p.half_tiles = static_cast<int>(p.tiles);
      p.clusters = static_cast<int>(2 * p.tiles);
    }
  }
  return p;
}

// ---------------------------------------------------------- in-kernel quantizer
// With BF16 activations, the GEMM can quantize A itself (gemm.cu): a quantize
// kernel first encodes the rows the first round of tiles reads (and zeroes the
// row-block counters), then one extra warp per CTA of the GEMM encodes the rest,
// in row order, while the main loop runs, publishing each 128-row block on a
// counter that the TMA producers wait for before loading that block. The leading
// rows: those of the row tiles of tiles [0, pairs), the first round (the second
// round's rows are encoded in-kernel in time; two rounds up front measured 1.3 µs
// slower at M = 4096 and the same at M = 20480). The quantizer warps (one per
// SM) encode about 0.19 G elements per ms in all (measured on GB300), enough to stay
// ahead of a GEMM that reads its A rows no faster than a 12288-wide one does; a
// narrower GEMM (the attention output projection, N = 3072, measured) gains
// nothing from encoding part of its rows in-kernel, so below kQaMinN all rows are
// encoded up front and the GEMM runs without its quantizer warp.
constexpr int kQaStrip = 1024;     // columns of one in-kernel quantize item (one per lane: 32 blocks)
constexpr int kQaGroup = 4;        // items a quantize warp loads at once (divides 128 rows x strips)
constexpr int64_t kQaMinN = 12288;

inline int64_t qa_strips(int64_t k) { return (k + kQaStrip - 1) / kQaStrip; }

inline int64_t qa_lead_rows(int64_t m, int64_t n, int clusters) {
  if (n < kQaMinN) return m;
  const int64_t tiles = gemm_pair_tiles(m, n), num_n = n / kPairTileCols;
  const int64_t lead = static_cast<int64_t>(clusters) < tiles ? static_cast<int64_t>(clusters) : tiles;
  const int64_t rows = lead > 0 ? ((lead - 1) / num_n + 1) * kPairTileRows : 0;
  return rows < m ? rows : m;
}

// Counter words of the in-kernel quantizer: one per 128-row block.
inline int64_t qa_counter_words(int64_t m) { return (m + 127) / 128; }

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
  void* workspace;         // split-tail workspace (256-byte aligned, counters zero) or null
  size_t workspace_bytes;
  // in-kernel quantizer (x null: A is already quantized): A = MXFP6(x) is written to
  // a_codes / a_scales; rows below qa_lead_rows are already there, and `ready`
  // (qa_counter_words words) is zero at the launch. No split tail with it.
  const void* x;           // bf16 [M][K], row stride ld_x elements
  int64_t ld_x;
  int64_t lead_rows;       // a multiple of 256 below M
  unsigned* ready;
};

// Returns cudaSuccess or the first CUDA error; `encode_failed` is set when the
// tensor-map encoder rejected the operands.
cudaError_t launch_gemm(const GemmArgs& args, int num_sms, cudaStream_t stream, bool* encode_failed);

// Shape rules shared by mx_mlp, mx_gated_mlp, mx_dit_mlp_block and mx_mlp_noalloc:
// MX_ERR_INVALID_ARG for a negative size, MX_ERR_UNSUPPORTED_SHAPE for d or ff of 0,
// d % 256, ff % 128, an up-projection width (ff, or 2 ff for the stacked SwiGLU
// weight) % 256, or a size of 2^31 or more; MX_OK otherwise (M == 0 included).
mx_status mlp_check_shape(int64_t M, int64_t d, int64_t ff, bool swiglu);

// Smallest workspace mx_mlp / mx_gated_mlp / mx_dit_mlp_block run with: the MXFP6
// activations and intermediate, without the split-tail region.
size_t mlp_min_workspace_bytes(int64_t M, int64_t d, int64_t ff);

// Unique ID of the calling thread's current CUDA context (cuCtxGetId); false when
// no context is current or the driver cannot say. A device's primary context gets
// a new ID when cudaDeviceReset destroys and recreates it, so caches of
// context-bound state (a device symbol's address, a kernel's shared-memory
// attribute) are kept per context ID rather than per device.
bool current_context_id(unsigned long long* id);

// Co-resident CTA pairs of the GEMM kernel on the current device (cached per device).
cudaError_t gemm_max_clusters(int* clusters);

cudaError_t launch_wait_selftest(cudaStream_t stream);

// Reads (and optionally clears) the device error word of the current device.
cudaError_t read_device_error(unsigned* flags, bool clear);

}  // namespace mxk
