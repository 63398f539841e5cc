/*
 * mx.h -- C ABI of the GB300 (sm_103a) MXFP6 MLP library.
 *
 * The operation is the MXFP6 hot path of a diffusion transformer's MLP, as the
 * page "Optimizing Krea 3 on AMD Instinct MI355X" describes it:
 *   - section "Quality set the precision limit": MXFP6 = 6-bit floating-point
 *     elements with one shared scale per block;
 *   - section "We built a faster MXFP6 kernel" (Figure 1): the MLP's GEMMs run
 *     in MXFP6 with the 6-bit values packed in memory;
 *   - section "Fusion cut intermediate memory traffic": the activations are
 *     quantized once, and the down-projection reads the up-projection's MXFP6
 *     output directly (no BF16 round trip, no separate requantization pass).
 * The number format (which the pages leave open) is OCP MX v1.0's: E2M3
 * elements, one E8M0 scale per 32 consecutive K-elements, shared exponent
 * floor(log2(block amax)) - 2, round-to-nearest-even, saturation at +-7.5.
 *
 * Conventions for every entry point
 *   - Every pointer except the ones marked "host" is a device pointer on the
 *     current CUDA device; the caller allocates and owns every buffer. The
 *     library allocates no device memory and keeps no per-call state.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream).
 *   - Argument errors are detected on the host before anything is launched and
 *     nothing is written. CUDA launch errors return MX_ERR_CUDA. Kernels never
 *     trap: a device-side wait that runs out (2 s) sets a bit that
 *     mx_device_error() reports, and the kernel returns.
 *   - Only compute capability 10.3 (GB300) is supported; anything else returns
 *     MX_ERR_UNSUPPORTED_DEVICE. There is no CPU fallback.
 *
 * Storage format (MXFP6 tensor of `rows` x K, K-major)
 *   codes : rows * 3K/4 bytes, 32-byte aligned. Row r holds its K 6-bit codes
 *           packed little-endian: code j at bits [6j, 6j+6) of the row's bits.
 *           A code is E2M3: bit 5 sign, bits 4..3 exponent (bias 1), bits 2..0
 *           mantissa.
 *   scales: mx_scales_bytes(rows, K) bytes, 16-byte aligned, one E8M0 byte per
 *           (row, 32-element K-block) in the tiled order of the tensor cores'
 *           scale-factor copy: 512-byte atoms per (128-row group, 4 K-blocks),
 *           atoms of a row group consecutive along K; inside an atom row
 *           r = 32*r1 + r0 and K-block j are at byte 16*r0 + 4*r1 + j. Rows are
 *           padded to a multiple of 128; padding scales are 0.
 *           mx_scales_to_plain() converts to plain [rows][K/32] order.
 */
#ifndef MX_H_
#define MX_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1,          /* null pointer, negative size, bad enum, ld_x < K   */
  MX_ERR_UNSUPPORTED_SHAPE = 2,    /* K % 128 != 0 or K == 0; N % 256 != 0; too large   */
  MX_ERR_MISALIGNED = 3,           /* codes not 32-byte aligned, others not 16-byte      */
  MX_ERR_WORKSPACE_TOO_SMALL = 4,  /* mx_mlp workspace below mx_mlp_workspace_bytes()    */
  MX_ERR_UNSUPPORTED_DEVICE = 5,   /* current device is not compute capability 10.3      */
  MX_ERR_CUDA = 6                  /* a CUDA runtime/driver call or a launch failed       */
} mx_status;

typedef enum {
  MX_EPI_BIAS_BF16 = 0,          /* out = bf16_rne(acc + bias): the down-projection (K2)       */
  MX_EPI_BIAS_GELU_MXFP6 = 1,    /* out = MXFP6(gelu_tanh(acc + bias)): the up-projection (K3)  */
  MX_EPI_BIAS_SWIGLU_MXFP6 = 2,  /* stacked gate/up weight: out = MXFP6(silu(g) * u)            */
  MX_EPI_GATE_RESIDUAL_BF16 = 3  /* out = bf16(residual + gate * (acc + bias)): mx_quantize_gemm
                                    only (mx_gemm_gate_residual is this epilogue on MXFP6 input) */
} mx_epilogue;

typedef enum {
  MX_ACT_GELU_TANH = 0,   /* up-projection W1 [ff][d], h = gelu_tanh(x W1^T + b1)                 */
  MX_ACT_SWIGLU = 1       /* stacked [W_g; W_u] [2ff][d], h = silu(x W_g^T + b_g) * (x W_u^T + b_u) */
} mx_activation;

/* Bytes of the packed codes of a rows x K MXFP6 tensor: rows * 3K/4. */
size_t mx_codes_bytes(int64_t rows, int64_t K);

/* Bytes of the tiled scales of a rows x K MXFP6 tensor: ceil(rows/128)*128 * K/32. */
size_t mx_scales_bytes(int64_t rows, int64_t K);

/*
 * mx_quantize -- K1: BF16 [rows][K] (row stride ld_x elements) -> MXFP6.
 * Per 32-element block: amax; scale exponent s = floor(log2 amax) - 2 clamped to
 * [-127, 127] (E8M0 code s + 127; an all-zero block gets code 0); each element
 * is v * 2^-s rounded to the nearest E2M3 value, ties to the even code, magnitude
 * saturated to 7.5, sign kept (so -0 -> 0x20). A block holding Inf/NaN gets scale
 * 0xFF and zero codes. Used for activations (every MLP call) and once for weights.
 *   x      : device, 16-byte aligned, rows x ld_x BF16 (only the first K of a row are read)
 *   rows   : >= 0 (0 is a no-op)          K: multiple of 128, > 0
 *   ld_x   : >= K, multiple of 8
 *   codes  : device, mx_codes_bytes(rows, K) bytes, 32-byte aligned (written)
 *   scales : device, mx_scales_bytes(rows, K) bytes, 16-byte aligned (written,
 *            padding rows included)
 */
mx_status mx_quantize(const void* x, int64_t rows, int64_t K, int64_t ld_x, void* codes, void* scales,
                      cudaStream_t stream);

/*
 * mx_quantize_stacked -- K1 over several BF16 matrices with the same K into one
 * stacked MXFP6 tensor of R = sum(part_rows) rows: the weights that one GEMM reads
 * as a single B operand ("Optimizing Krea 3 on AMD Instinct MI355X", section
 * "Fusion cut intermediate memory traffic": the stacked projections are quantized
 * and read once) -- [W_g; W_u] for MX_EPI_BIAS_SWIGLU_MXFP6 / mx_gated_mlp, or the
 * query/key/value/gate weights of one projection. Rows are quantized independently,
 * so the result equals mx_quantize of the concatenated matrix.
 * Scale-atom offset rule: part i starts at stacked row R_i = part_rows[0] + ... +
 * part_rows[i-1]; its codes at byte mx_codes_bytes(R_i, K) of `codes` and its
 * scales at byte mx_scales_bytes(R_i, K) of `scales`. That is where its own
 * mx_quantize output would go, because every part but the last has a multiple of
 * 128 rows, so each part's tiled scales begin on a 512-byte atom.
 *   x_parts   : host array of n_parts device pointers; part i is BF16
 *               [part_rows[i]][K] with row stride ld_x[i], 16-byte aligned
 *   part_rows : host array of n_parts row counts >= 0; all but the last % 128 == 0
 *   ld_x      : host array of n_parts row strides (>= K, % 8 == 0), or NULL for K
 *   n_parts   : >= 1
 *   K         : as mx_quantize
 *   codes, scales : the stacked tensor, mx_codes_bytes(R, K) and mx_scales_bytes(R, K)
 *               bytes (32- and 16-byte aligned), written
 * Every part is checked on the host before the first launch (one launch per part,
 * in order, on `stream`); a bad part returns its mx_quantize status and nothing is
 * written. R < 2^31.
 */
mx_status mx_quantize_stacked(const void* const* x_parts, const int64_t* part_rows, const int64_t* ld_x, int n_parts,
                              int64_t K, void* codes, void* scales, cudaStream_t stream);

/*
 * mx_quantize_rmsnorm_modulate -- K1 with the step before it fused in: row-wise
 * RMS normalisation, modulation, then MXFP6 quantization of the result
 * ("Optimizing Krea 3 on AMD Instinct MI355X", section "Fusion cut intermediate
 * memory traffic": modulation merged with RMSNorm; "Creating Custom Kernels for
 * the AMD MI300", section "Fused RMS Norm Kernel").
 *   y[m][k] = x[m][k] / sqrt(mean_k' x[m][k']^2 + eps) * (1 + scale[k]) + shift[k]
 * in fp32 (sum of squares in fp32, rstd = rsqrtf(sum / K + eps) within 2 ulp, then
 * fma(x * rstd, 1 + scale, shift)); codes/scales = MXFP6(y) by the mx_quantize rule.
 *   x, rows, K, ld_x, codes, scales : as mx_quantize, and K <= 8192
 *   shift, scale : device BF16 [K] (one conditioning vector for all rows), 16-byte
 *                  aligned, or NULL for zeros
 *   eps          : >= 0 and finite (with eps = 0 an all-zero row gives NaN, whose
 *                  blocks get scale 0xFF and zero codes)
 *   debug_y      : NULL, or device fp32 [rows][K] (16-byte aligned) that receives y,
 *                  the exact values the quantization rounded (test hook)
 */
mx_status mx_quantize_rmsnorm_modulate(const void* x, int64_t rows, int64_t K, int64_t ld_x, const void* shift,
                                       const void* scale, float eps, void* codes, void* scales, float* debug_y,
                                       cudaStream_t stream);

/*
 * mx_gemm -- K2/K3: C = A * B^T on MXFP6 operands, fp32 accumulation in tensor
 * memory, then the fused epilogue `epi`:
 *   MX_EPI_BIAS_BF16      : out = BF16 [M][N] row-major, bf16_rne(C + bias)
 *   MX_EPI_BIAS_GELU_MXFP6: g = gelu_tanh(C + bias) in fp32, with
 *                           gelu_tanh(v) = 0.5 v (1 + tanh(sqrt(2/pi)(v + 0.044715 v^3)));
 *                           out = MXFP6 codes of g [M][N] (same rule as mx_quantize,
 *                           blocks of 32 along N), out_scales = its tiled scales.
 *   MX_EPI_BIAS_SWIGLU_MXFP6: the gate and up projections of a SwiGLU MLP as one
 *                           GEMM ("Optimizing Krea 3 on AMD Instinct MI355X", section
 *                           "Fusion cut intermediate memory traffic"; "Creating Custom
 *                           Kernels for the AMD MI300", section "Fused SwiGLU Kernel").
 *                           B is the stacked weight [W_g; W_u]: its first F = N/2 rows
 *                           are the gate rows, the next F the up rows (quantize W_g and
 *                           W_u into the two halves of one buffer); bias likewise
 *                           [b_g; b_u] (2F values). With C = [G | U]:
 *                           h = silu(G + b_g) * (U + b_u) in fp32, silu(v) = v/(1+e^-v);
 *                           out = MXFP6 codes of h [M][F], out_scales its tiled
 *                           scales (mx_scales_bytes(M, F)).
 *   a_codes/a_scales : A, M x K MXFP6 (activations)
 *   b_codes/b_scales : B, N x K MXFP6 (weights, nn.Linear layout)
 *   bias             : device BF16 [N], 16-byte aligned, or NULL (no bias)
 *   M >= 0 (any value; 0 is a no-op), N % 256 == 0, K % 128 == 0 and K > 0,
 *   M, N, K < 2^31.
 *   out              : BF16 [M][N] (16-byte aligned) or codes mx_codes_bytes(M, W),
 *                      W = N (GELU) or N/2 (SwiGLU), 32-byte aligned
 *   out_scales       : MXFP6 epilogues only: mx_scales_bytes(M, W) bytes; else ignored
 *   debug_prequant   : MXFP6 epilogues only, may be NULL: fp32 [M][W] receives g
 *                      (or h), the exact value the requantization rounded (test hook).
 *   workspace        : NULL, or device scratch of workspace_bytes bytes (256-byte
 *                      aligned, overlapping no other argument) for the split tail:
 *                      when the 256 x 256 output tiles leave a last round at most a
 *                      quarter full for the GPU's CTA pairs (76 on GB300) and K >= 4096,
 *                      the first pairs + (tiles mod pairs) tiles are divided along K so
 *                      every pair does the same work, and a tile two pairs share is
 *                      summed through the workspace (the two fp32 partial sums are
 *                      added once, so the result is deterministic but may differ from
 *                      the unsplit one by fp32 rounding). Used when workspace_bytes >=
 *                      mx_gemm_workspace_bytes(M, N, K) (> 0); otherwise, and for other
 *                      shapes, the GEMM runs unsplit (mx_gemm_launch_plan tells which). Its first
 *                      MX_GEMM_WORKSPACE_COUNTER_BYTES bytes are arrival counters that
 *                      must be zero when the GEMM starts: zero them once when the
 *                      workspace is new (e.g. cudaMemsetAsync); every launch that
 *                      completes leaves them zero again (after mx_device_error
 *                      reports a timeout, zero them anew). Calls sharing one
 *                      workspace must not overlap on the GPU.
 */
mx_status mx_gemm(const void* a_codes, const void* a_scales, const void* b_codes, const void* b_scales,
                  const void* bias, int64_t M, int64_t N, int64_t K, mx_epilogue epi, void* out,
                  void* out_scales, float* debug_prequant, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream);

/*
 * mx_gemm_gate_residual -- an output projection fused with its gate and the
 * residual add ("Optimizing Krea 3 on AMD Instinct MI355X", section "Fusion cut
 * intermediate memory traffic"):
 *   out[m][n] = bf16_rne(residual[m][n] + gate[n] * (C[m][n] + bias[n])),  C = A * B^T
 * computed in fp32 as fma(gate, C + bias, residual).
 *   A, B, bias, M, N, K : as mx_gemm (MXFP6 operands, N % 256 == 0, K % 128 == 0)
 *   gate     : device BF16 [N] (one conditioning vector for all rows), 16-byte
 *              aligned, or NULL for a gate of 1 (plain residual add)
 *   residual : device BF16 [M][N] row-major, 16-byte aligned; required
 *   out      : device BF16 [M][N] row-major, 16-byte aligned (written). It may be
 *              residual itself (in-place update: the warp that reads a block of
 *              the residual issues that block's store only after its loads); any
 *              other overlap returns MX_ERR_INVALID_ARG.
 *   workspace, workspace_bytes : the optional split-tail scratch, as mx_gemm.
 */
mx_status mx_gemm_gate_residual(const void* a_codes, const void* a_scales, const void* b_codes,
                                const void* b_scales, const void* bias, const void* gate, const void* residual,
                                int64_t M, int64_t N, int64_t K, void* out, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes that let mx_gemm / mx_gemm_gate_residual of this shape split
 * their tail: MX_GEMM_WORKSPACE_COUNTER_BYTES of arrival counters plus two 256 KB
 * partial-sum slots per CTA pair, for at most 80 pairs (about 42 MB; GB300 runs
 * 76); 0 when the shape never splits (K < 4096, a single tile, or an unsupported
 * shape). Host only; depends on nothing but the shape (whether a launch splits
 * also depends on the device's pair count: mx_gemm_launch_plan).
 */
#define MX_GEMM_WORKSPACE_COUNTER_BYTES ((size_t)10240)

size_t mx_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * mx_gemm_launch_plan -- what a GEMM of this shape does on the current device:
 *   pairs       (host, written): CTA pairs of the whole-tile plan (co-resident pairs,
 *                                at most one per tile)
 *   split_tiles (host, written): leading tiles divided along K when called with a
 *                                workspace of workspace_bytes bytes (0: no split)
 * Shape rules as mx_gemm; M == 0 or N == 0 gives 0 and 0. Without a split, a GEMM
 * with an epilogue other than MX_EPI_BIAS_SWIGLU_MXFP6 and no debug output also
 * runs its last round's tiles as two 128-column halves each when they fit in one
 * round (tiles mod pairs <= pairs / 2), and all its tiles as halves, on twice as
 * many pairs, when it has at most pairs / 2 tiles; the result is the same.
 */
mx_status mx_gemm_launch_plan(int64_t M, int64_t N, int64_t K, size_t workspace_bytes, int* pairs,
                              int* split_tiles);

/*
 * mx_quantize_gemm -- mx_quantize of BF16 activations fused with the GEMM that
 * reads them ("Optimizing Krea 3 on AMD Instinct MI355X", section "Fusion cut
 * intermediate memory traffic": activations quantized on the fly, once):
 *   xq = MXFP6(x) (the mx_quantize rule, bit for bit), then
 *   out = epilogue(xq * B^T + bias) as mx_gemm (epi 0-2), or, with
 *   MX_EPI_GATE_RESIDUAL_BF16, as mx_gemm_gate_residual (gate, residual).
 * The quantize kernel encodes the leading rows (and zeroes the workspace's
 * counters); the GEMM quantizes the remaining rows itself, in an extra warp per
 * CTA, while its main loop runs, so the encoding of most of x overlaps the
 * tensor-core work. The leading rows are those the GEMM's first round of tiles
 * reads; for N < 12288 (where the extra warps would fall behind the GEMM's
 * reads) they are all M rows, and the GEMM runs as mx_gemm. Two launches on `stream`.
 *   x        : device BF16 [M][K] row-major, row stride ld_x elements (ld_x % 8 == 0),
 *              16-byte aligned; must not overlap out or the workspace
 *   b_*, bias, N, K, out, out_scales : as mx_gemm (K % 128 == 0, N % 256 == 0)
 *   gate, residual : MX_EPI_GATE_RESIDUAL_BF16 only, as mx_gemm_gate_residual
 *              (residual required; out may be residual itself; neither may overlap
 *              the workspace); ignored otherwise
 *   workspace: device, mx_quantize_gemm_workspace_bytes(M, K) bytes, 256-byte
 *              aligned, any contents. After the call (in stream order) it holds
 *              MXFP6(x): codes at offset 0 (mx_codes_bytes(M, K) bytes), tiled
 *              scales at offset mx_codes_bytes(M, K) rounded up to 256, then one
 *              counter word per 128 rows (zeroed by the call's quantize kernel).
 * No split tail, no debug output. M == 0 or N == 0: nothing is launched.
 * Not for two calls at once on one workspace.
 * The GEMM's CTAs wait for rows that other CTAs' quantizer warps encode; those
 * warps claim their rows from a counter, so a CTA that has not started holds
 * none, and the call runs correctly beside other streams' kernels.
 */
size_t mx_quantize_gemm_workspace_bytes(int64_t M, int64_t K);

mx_status mx_quantize_gemm(const void* x, int64_t M, int64_t K, int64_t ld_x, const void* b_codes,
                           const void* b_scales, const void* bias, int64_t N, mx_epilogue epi, const void* gate,
                           const void* residual, void* out, void* out_scales, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

/*
 * Workspace bytes of mx_mlp, mx_gated_mlp and mx_dit_mlp_block for M tokens:
 * MXFP6 x (M x d), MXFP6 h (M x ff), one counter word per 128 rows (the
 * up-projection's in-kernel quantizer) and the split-tail region both GEMMs use in
 * turn (as mx_gemm_workspace_bytes, for the wider of the two), each part starting
 * on a 256-byte boundary. A smaller workspace that still holds the first five
 * parts runs without the split tail.
 */
size_t mx_mlp_workspace_bytes(int64_t M, int64_t d, int64_t ff);

/*
 * mx_mlp -- the whole MXFP6 MLP block in three launches on `stream`:
 *   K1 xq = MXFP6(x); K3 hq = MXFP6(gelu_tanh(xq W1^T + b1)); K2 y = bf16(hq W2^T + b2).
 *   As in mx_quantize_gemm, K1 encodes only the leading rows of x (those K3's
 *   first round of tiles reads), and K3 encodes the rest itself while it runs
 *   (when its width, ff or 2 ff, is at least 12288, it does not split its tail, and
 *   the leading rows are not all of x); the result is the same bit for bit.
 *   x        : BF16 [M][d] (16-byte aligned); y: BF16 [M][d] (written)
 *   w1_*     : W1 as MXFP6, ff x d (quantized once with mx_quantize)
 *   w2_*     : W2 as MXFP6, d x ff
 *   b1, b2   : BF16 [ff], [d], or NULL
 *   d % 256 == 0, ff % 256 == 0 (both are K of one GEMM and N of the other)
 *   workspace: device, mx_mlp_workspace_bytes(M, d, ff) bytes, 256-byte aligned;
 *              holds xq, hq, the row-block counters and the split-tail scratch (the
 *              first kernel zeroes the counters, so no initialisation is needed); must not overlap
 *              any other argument. Without
 *              room for the split-tail region the GEMMs run unsplit; without room
 *              for xq and hq the call returns MX_ERR_WORKSPACE_TOO_SMALL.
 */
mx_status mx_mlp(const void* x, int64_t M, int64_t d, int64_t ff, const void* w1_codes, const void* w1_scales,
                 const void* b1, const void* w2_codes, const void* w2_scales, const void* b2, void* y,
                 void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * mx_gated_mlp -- the SwiGLU MLP block in three launches on `stream`:
 *   K1 xq = MXFP6(x); up hq = MXFP6(silu(xq W_g^T + b_g) * (xq W_u^T + b_u));
 *   K2 y = bf16(hq W2^T + b2).
 *   wgu_*    : the stacked [W_g; W_u] as MXFP6, 2ff x d (gate rows first)
 *   bgu      : BF16 [2ff] = [b_g; b_u], or NULL
 *   w2_*     : W2 as MXFP6, d x ff;  b2: BF16 [d] or NULL
 *   d % 256 == 0, ff % 128 == 0; workspace as mx_mlp (mx_mlp_workspace_bytes(M, d, ff)).
 */
mx_status mx_gated_mlp(const void* x, int64_t M, int64_t d, int64_t ff, const void* wgu_codes,
                       const void* wgu_scales, const void* bgu, const void* w2_codes, const void* w2_scales,
                       const void* b2, void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * mx_dit_mlp_block -- the MLP half of a diffusion-transformer block, with both
 * neighbouring fusions of "Optimizing Krea 3 on AMD Instinct MI355X", section
 * "Fusion cut intermediate memory traffic", in three launches on `stream`:
 *   1. xq = MXFP6(x / rms(x) * (1 + scale) + shift)    (mx_quantize_rmsnorm_modulate)
 *   2. hq = MXFP6(act(xq W_up^T + b_up))                (GELU, or SwiGLU on [W_g; W_u])
 *   3. y  = bf16(x + gate * (hq W2^T + b2))             (mx_gemm_gate_residual, residual x)
 *   x          : BF16 [M][d]; y: BF16 [M][d], may be x itself (in place), no other overlap
 *   shift, scale, gate : BF16 [d] conditioning vectors (one sample), or NULL (0, 0, 1)
 *   eps        : as mx_quantize_rmsnorm_modulate
 *   activation : MX_ACT_GELU_TANH (w_up = W1, ff x d; b_up [ff]) or MX_ACT_SWIGLU
 *                (w_up = [W_g; W_u], 2ff x d; b_up [2ff])
 *   w2_*, b2   : W2 as MXFP6, d x ff; BF16 [d] or NULL
 *   d % 256 == 0, d <= 8192, ff % 128 == 0 (ff % 256 == 0 for GELU);
 *   workspace  : >= mx_mlp_workspace_bytes(M, d, ff), 256-byte aligned.
 */
mx_status mx_dit_mlp_block(const void* x, int64_t M, int64_t d, int64_t ff, const void* shift, const void* scale,
                           const void* gate, float eps, mx_activation activation, const void* w_up_codes,
                           const void* w_up_scales, const void* b_up, const void* w2_codes, const void* w2_scales,
                           const void* b2, void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Capacity of the static scratch of mx_mlp_noalloc: 64 MiB per GPU. */
#define MX_MLP_NOALLOC_WORKSPACE_BYTES ((size_t)64 << 20)

/*
 * mx_mlp_noalloc -- mx_mlp for callers that cannot allocate device memory.
 * The paper has no counterpart for this entry point; it exists for callers such
 * as code hosted in a runtime whose allocator owns all device memory, callers
 * with a device-memory budget fixed at start-up, and paths that cannot afford
 * cudaMalloc's implicit synchronization.
 *   Same arguments and results as mx_mlp, without workspace/workspace_bytes: the
 *   scratch (MXFP6 x and MXFP6 h, and the split-tail region when it also fits)
 *   lives in a static device array of MX_MLP_NOALLOC_WORKSPACE_BYTES inside the
 *   library, which every GPU that loads the library holds until the process exits.
 *   The call allocates nothing. Sizes whose MXFP6 x and h exceed that capacity
 *   return MX_ERR_WORKSPACE_TOO_SMALL before anything is launched (for d = 3072,
 *   ff = 12288 that is M > 5590 tokens).
 *   Argument checks run in mx_mlp's order (shape rules first, then M == 0 is a
 *   no-op, then the capacity, then null pointers), all before any launch.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, and so does the first call
 *   in a new context of the device (cudaDeviceReset recreates the context, and
 *   the array may then sit elsewhere); make such a first call before any stream
 *   capture.
 *   Every call on a device shares the one array, and the kernels write all of it
 *   that they read before reading it (the first kernel zeroes the split-tail
 *   counters), so nothing needs clearing between calls; but calls whose
 *   executions overlap on the GPU (different streams, no ordering between them)
 *   race on the array and must be serialized by the caller.
 */
mx_status mx_mlp_noalloc(const void* x, int64_t M, int64_t d, int64_t ff, const void* w1_codes,
                         const void* w1_scales, const void* b1, const void* w2_codes, const void* w2_scales,
                         const void* b2, void* y, cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* mx_status_string(mx_status status);

/*
 * mx_scales_to_plain -- host-side layout helper: tiled scales (host, as written
 * by the kernels) -> plain row-major [rows][K/32] (host). K % 128 == 0.
 */
mx_status mx_scales_to_plain(const void* tiled_host, void* plain_host, int64_t rows, int64_t K);

/* Inverse of mx_scales_to_plain (host). Padding rows of `tiled_host` are set to 0. */
mx_status mx_scales_from_plain(const void* plain_host, void* tiled_host, int64_t rows, int64_t K);

/*
 * mx_device_error -- synchronizes the current device and reads the device-side
 * error word of the library's kernels (0 = none; bit 0: a producer wait ran out,
 * bit 1: an MMA wait, bit 2: an epilogue wait, bit 3: draining after an abort ran
 * out, bit 4: mx_selftest_wait_timeout ran, bit 5: a GEMM that quantizes its own
 * activations (mx_quantize_gemm, mx_mlp, mx_gated_mlp) gave up waiting for a block
 * of them). clear != 0 resets it. Returns MX_ERR_CUDA if the read itself fails.
 */
mx_status mx_device_error(unsigned* flags_host, int clear);

/*
 * mx_selftest_wait_timeout -- failure-detection self test. Launches a one-warp
 * kernel whose single mbarrier wait can never complete (nothing arrives on it).
 * The wait gives up after the kernels' bound (2 s), sets bit 4 of the device
 * error word and returns; the CUDA context stays usable. No GPU fault, trap or
 * hang is involved. Asynchronous on `stream`; read the result with
 * mx_device_error().
 */
mx_status mx_selftest_wait_timeout(cudaStream_t stream);

/* Library ABI version (major * 100 + minor). */
int mx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MX_H_ */
