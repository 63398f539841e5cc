"""Plain, slow CPU restatement of the MXFP6 MLP hot path (numpy, fp64).

TEST INFRASTRUCTURE ONLY: the product path never imports this module. Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (``cpu_baseline`` and
``--impl reference``) may import it. It shares no code with the CUDA library.

What it restates
----------------
"Optimizing Krea 3 on AMD Instinct MI355X", section "Quality set the precision
limit": MXFP6 stores 6-bit floating-point elements with one shared scale per
block. Section "Fusion cut intermediate memory traffic": the up-projection's
output is quantized to MXFP6 and the down-projection reads it directly.
Section "We built a faster MXFP6 kernel" (Figure 1): the GEMMs of one GPU's
share of the MLP are the measured work.

The pages do not spell out the number format. This library's contract fixes it,
and it is the one of the OCP Microscaling Formats (MX) v1.0 specification:

* element: FP6 E2M3 -- 1 sign bit, 2 exponent bits (bias 1), 3 mantissa bits,
  no Inf/NaN, largest magnitude 7.5;
* scale: E8M0 -- an unsigned biased exponent, value 2**(code - 127), 0xFF = NaN;
* block: 32 consecutive elements along K of one row;
* shared exponent: s = floor(log2(amax)) - 2, where 2 is the largest exponent
  of E2M3, so that the block maximum lands in [4, 8);
* element: round v * 2**-s to the nearest E2M3 value, ties to the even code,
  saturating to +-7.5.

Each function below says which of these steps it follows. Readings taken where
the pages and the contract are silent are listed in each docstring.

The neighbouring fusions of the same section -- the gate and up projections
stacked with the SwiGLU activation, modulation merged with RMSNorm before the
quantizer, and an output projection merged with its gate and the residual add
-- are restated at the end of the module ("Fused neighbours").

Parity pins (tests/test_oracle.py): every function here is pinned against
something other than itself -- the OCP MX value table typed in by hand, CUDA's
own host-side fp6 conversion routine, brute-force integer GEMMs, mpmath, and
hand-derived fixtures under tests/golden/.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "BLOCK",
    "E2M3_MAX",
    "e2m3_value",
    "E2M3_TABLE",
    "e8m0_value",
    "bf16_bits_to_f64",
    "f32_to_f64",
    "shared_exponent",
    "nearest_e2m3_code",
    "quantize",
    "quantize_bf16",
    "quantize_f32",
    "dequantize",
    "pack_codes",
    "unpack_codes",
    "scales_tiled_to_plain",
    "scales_plain_to_tiled",
    "scales_tiled_bytes",
    "gemm",
    "gelu_tanh",
    "up_projection",
    "down_projection",
    "mlp",
    "silu",
    "swiglu_up_projection",
    "gated_mlp",
    "rms_norm_modulate",
    "gate_residual",
    "dit_mlp_block",
]

BLOCK = 32          # elements sharing one scale (OCP MX v1.0, block size k = 32)
E2M3_MAX = 7.5      # largest E2M3 magnitude
E2M3_EMAX = 2       # exponent of the largest E2M3 binade ([4, 8))


# --------------------------------------------------------------------------
# Element and scale types
# --------------------------------------------------------------------------

def e2m3_value(code: int) -> float:
    """Value of one 6-bit E2M3 code (OCP MX v1.0, FP6 E2M3 definition).

    Bit 5 is the sign, bits 4..3 the exponent field e (bias 1), bits 2..0 the
    mantissa m. e == 0 is subnormal: m/8. Otherwise (1 + m/8) * 2**(e - 1).
    """
    if not 0 <= code < 64:
        raise ValueError("E2M3 codes are 6-bit")
    sign = -1.0 if code & 0x20 else 1.0
    e = (code >> 3) & 0x3
    m = code & 0x7
    if e == 0:
        mag = m / 8.0
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 1)
    return sign * mag


#: value of every code 0..63, decoded one by one from the definition.
E2M3_TABLE = np.array([e2m3_value(c) for c in range(64)], dtype=np.float64)
#: the 32 non-negative magnitudes (codes 0x00..0x1F), increasing.
_MAGNITUDES = E2M3_TABLE[:32].copy()


def e8m0_value(code):
    """Value of an E8M0 scale code: 2**(code - 127); 0xFF is NaN (OCP MX v1.0)."""
    code = np.asarray(code, dtype=np.int64)
    out = np.ldexp(1.0, (code - 127).astype(np.int64))
    return np.where(code == 0xFF, np.nan, out)


# --------------------------------------------------------------------------
# Input decoding (exact)
# --------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> exact fp64 values (BF16 is the top half of fp32)."""
    bits = np.asarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):   # NaN patterns widen to NaN; numpy warns about them
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_f64(x) -> np.ndarray:
    """fp32 -> fp64, exact."""
    return np.asarray(x, dtype=np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# Quantization (OCP MX v1.0 conversion: shared exponent, then per element)
# --------------------------------------------------------------------------

def shared_exponent(amax) -> np.ndarray:
    """s = floor(log2(amax)) - 2, clamped to the E8M0 range [-127, 127].

    floor(log2(a)) is taken exactly from the binary exponent (np.frexp gives
    a = f * 2**e with f in [0.5, 1), so floor(log2 a) = e - 1), never from a
    floating-point log2. Reading: an all-zero block (amax == 0) takes the
    smallest scale, s = -127 (E8M0 code 0x00); its codes are all zero anyway.
    """
    amax = np.asarray(amax, dtype=np.float64)
    _, e = np.frexp(amax)
    s = (e.astype(np.int64) - 1) - E2M3_EMAX
    s = np.where(amax == 0.0, -127, s)
    return np.clip(s, -127, 127)


def _nearest_chunk(f: np.ndarray) -> np.ndarray:
    # Every |t| >= 8 has 7.5 as its nearest value, as 8 does; capping at 8
    # keeps each distance below exact in fp64 (huge |t| would round them).
    a = np.minimum(np.abs(f), 8.0)
    best = np.abs(a - _MAGNITUDES[0])
    code = np.zeros(a.shape, dtype=np.uint8)
    for j in range(1, 32):
        d = np.abs(a - _MAGNITUDES[j])
        # strictly nearer wins; on an exact tie with code j - 1 the even one wins
        take = (d < best) | ((d == best) & (j % 2 == 0))
        best = np.where(take, d, best)
        code = np.where(take, np.uint8(j), code)
    return code | np.where(np.signbit(f), 0x20, 0).astype(np.uint8)


def nearest_e2m3_code(t) -> np.ndarray:
    """Round each value to the nearest E2M3 code by brute-force search.

    The magnitude |t| is compared with all 32 non-negative E2M3 values; the
    nearest wins, a tie goes to the even code (code LSB 0 -- for a binary
    floating-point format this is the even-mantissa rule of round-to-nearest-
    even). Values beyond 7.5 are nearest to 7.5 (code 0x1F), which is the
    saturation the contract asks for. The sign bit copies the sign of t,
    negative zero included (so -0.01 gives 0x20, as IEEE rounding does).
    Independent chunks of elements are searched on a thread pool.
    """
    t = np.asarray(t, dtype=np.float64)
    flat = t.reshape(-1)
    chunk = 1 << 16
    pieces = [flat[lo:lo + chunk] for lo in range(0, flat.size, chunk)]
    if len(pieces) <= 1:
        out = _nearest_chunk(flat)
    else:
        with ThreadPoolExecutor(max_workers=min(len(pieces), os.cpu_count() or 1)) as ex:
            out = np.concatenate(list(ex.map(_nearest_chunk, pieces)))
    return out.reshape(t.shape)


def quantize(v) -> tuple[np.ndarray, np.ndarray]:
    """Quantize rows of exact values to MXFP6 along the last axis.

    v: float64 [rows][K], K a multiple of 32, holding values that are exact
    (they come from BF16 or fp32). Returns (codes uint8 [rows][K], one 6-bit
    code per byte; scales uint8 [rows][K/32], E8M0, plain row-major order).

    Per block of 32: amax = max |v|; s = shared_exponent(amax); codes =
    nearest_e2m3_code(v * 2**-s) (the multiply by a power of two is exact in
    fp64). Reading for non-finite input, which the contract does not cover: a
    block holding Inf or NaN gets scale 0xFF (the E8M0 NaN) and all-zero codes.
    """
    v = np.asarray(v, dtype=np.float64)
    if v.ndim != 2 or v.shape[1] % BLOCK:
        raise ValueError("quantize wants [rows][K] with K a multiple of 32")
    rows, k = v.shape
    blocks = v.reshape(rows, k // BLOCK, BLOCK)
    finite = np.isfinite(blocks).all(axis=2)
    safe = np.where(np.isfinite(blocks), blocks, 0.0)
    amax = np.abs(safe).max(axis=2)
    s = shared_exponent(amax)
    t = np.ldexp(safe, (-s)[:, :, None])
    codes = nearest_e2m3_code(t)
    codes = np.where(finite[:, :, None], codes, 0).astype(np.uint8)
    scales = np.where(finite, s + 127, 0xFF).astype(np.uint8)
    return codes.reshape(rows, k), scales


def quantize_bf16(x_bits) -> tuple[np.ndarray, np.ndarray]:
    """quantize() of a BF16 matrix given as uint16 bit patterns."""
    return quantize(bf16_bits_to_f64(x_bits))


def quantize_f32(x) -> tuple[np.ndarray, np.ndarray]:
    """quantize() of an fp32 matrix (used for the fused requantization)."""
    return quantize(f32_to_f64(x))


def dequantize(codes, scales) -> np.ndarray:
    """fp64 value of each element: E2M3 value of its code times 2**(scale - 127)."""
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint8)
    rows, k = codes.shape
    if scales.shape != (rows, k // BLOCK):
        raise ValueError("scales must be [rows][K/32]")
    vals = E2M3_TABLE[codes & 0x3F]
    factor = np.repeat(e8m0_value(scales), BLOCK, axis=1)
    return vals * factor


# --------------------------------------------------------------------------
# Storage formats
# --------------------------------------------------------------------------

def pack_codes(codes) -> np.ndarray:
    """Pack 6-bit codes densely, little-endian: code j of a row occupies bits
    [6j, 6j + 6) of the row's bit string, byte b holds bits [8b, 8b + 8).

    So every 4 codes fill 3 bytes and every 16 codes 12 bytes (the 16 x U6
    group the GPU's tensor-memory-access unit moves). [rows][K] -> [rows][3K/4].
    """
    codes = np.asarray(codes, dtype=np.uint8)
    rows, k = codes.shape
    if k % 4:
        raise ValueError("K must be a multiple of 4")
    q = codes.reshape(rows, k // 4, 4).astype(np.uint32) & 0x3F
    word = q[..., 0] | (q[..., 1] << 6) | (q[..., 2] << 12) | (q[..., 3] << 18)
    out = np.empty((rows, k // 4, 3), dtype=np.uint8)
    out[..., 0] = word & 0xFF
    out[..., 1] = (word >> 8) & 0xFF
    out[..., 2] = (word >> 16) & 0xFF
    return out.reshape(rows, 3 * k // 4)


def unpack_codes(packed, k: int) -> np.ndarray:
    """Inverse of pack_codes: [rows][3K/4] bytes -> [rows][K] codes."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows = packed.shape[0]
    b = packed.reshape(rows, k // 4, 3).astype(np.uint32)
    word = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16)
    out = np.empty((rows, k // 4, 4), dtype=np.uint8)
    for j in range(4):
        out[..., j] = (word >> (6 * j)) & 0x3F
    return out.reshape(rows, k)


def scales_tiled_bytes(rows: int, k: int) -> int:
    """Bytes of the tiled scale array: rows rounded up to 128, K/32 per row."""
    return ((rows + 127) // 128) * 128 * (k // BLOCK)


def _tiled_offset(r, kb, k):
    """Byte offset of the scale of (row r, K-block kb) in the tiled order.

    The tiled order is the one the tensor cores' scale-factor copy consumes:
    512-byte atoms, one per (128-row group, 4 consecutive K-blocks); atoms of
    one row group are consecutive along K. Inside an atom, row r = 32*r1 + r0
    (r0 < 32, r1 < 4) and K-block j < 4 sit at byte 16*r0 + 4*r1 + j.
    """
    atom = (r // 128) * (k // 128) + kb // 4
    r0 = r % 32
    r1 = (r % 128) // 32
    return atom * 512 + 16 * r0 + 4 * r1 + (kb % 4)


def scales_tiled_to_plain(tiled, rows: int, k: int) -> np.ndarray:
    """Tiled scale bytes (see _tiled_offset) -> plain [rows][K/32] array."""
    tiled = np.asarray(tiled, dtype=np.uint8).reshape(-1)
    if k % 128:
        raise ValueError("tiled scales need K % 128 == 0")
    r = np.arange(rows)[:, None]
    kb = np.arange(k // BLOCK)[None, :]
    return tiled[_tiled_offset(r, kb, k)]


def scales_plain_to_tiled(plain, rows: int, k: int, pad_value: int = 0) -> np.ndarray:
    """Plain [rows][K/32] -> tiled bytes; padding rows (up to 128) get pad_value."""
    plain = np.asarray(plain, dtype=np.uint8)
    out = np.full(scales_tiled_bytes(rows, k), pad_value, dtype=np.uint8)
    r = np.arange(rows)[:, None]
    kb = np.arange(k // BLOCK)[None, :]
    out[_tiled_offset(r, kb, k)] = plain
    return out


# --------------------------------------------------------------------------
# GEMM, activation and the MLP
# --------------------------------------------------------------------------

def gemm(a_codes, a_scales, b_codes, b_scales, bias_bits=None) -> np.ndarray:
    """C[m][n] = sum_k deq(A)[m][k] * deq(B)[n][k] (+ bias[n]) in fp64.

    A is [M][K] and B is [N][K], both K-major with K-blocks of 32, as in
    nn.Linear (y = x W^T). bias_bits are BF16 bit patterns, decoded exactly.
    The matmul is a library primitive on exactly dequantized operands.
    """
    a = dequantize(a_codes, a_scales)
    b = dequantize(b_codes, b_scales)
    c = a @ b.T
    if bias_bits is not None:
        c = c + bf16_bits_to_f64(bias_bits)[None, :]
    return c


def gelu_tanh(v) -> np.ndarray:
    """tanh-approximated GELU in fp64: 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3)))."""
    v = np.asarray(v, dtype=np.float64)
    return 0.5 * v * (1.0 + np.tanh(np.sqrt(2.0 / np.pi) * (v + 0.044715 * v ** 3)))


def up_projection(xq_codes, xq_scales, w1_codes, w1_scales, b1_bits):
    """Up-projection with its fused epilogue, fp64: gelu_tanh(x W1^T + b1).

    Returns the fp64 pre-quantization activation [M][ff]. Requantizing it
    needs a precision decision: the GPU rounds its own fp32 accumulation, so
    parity requantizes the GPU's fp32 values (quantize_f32) instead.
    """
    return gelu_tanh(gemm(xq_codes, xq_scales, w1_codes, w1_scales, b1_bits))


def down_projection(hq_codes, hq_scales, w2_codes, w2_scales, b2_bits):
    """Down-projection with bias, fp64 (the BF16 store is compared with tolerance)."""
    return gemm(hq_codes, hq_scales, w2_codes, w2_scales, b2_bits)


def mlp(x_bits, w1_codes, w1_scales, b1_bits, w2_codes, w2_scales, b2_bits):
    """The whole MLP, independent of any GPU value.

    x (BF16) -> MXFP6 -> up-projection + bias + GELU -> rounded to fp32 ->
    MXFP6 -> down-projection + bias. Reading: the intermediate is rounded to
    fp32 before requantization, the precision the fused epilogue keeps.
    Returns (y fp64 [M][d], intermediate dict).
    """
    xq, xs = quantize_bf16(x_bits)
    g = up_projection(xq, xs, w1_codes, w1_scales, b1_bits)
    hq, hs = quantize_f32(g.astype(np.float32))
    y = down_projection(hq, hs, w2_codes, w2_scales, b2_bits)
    return y, {"xq": xq, "xs": xs, "g": g, "hq": hq, "hs": hs}


# --------------------------------------------------------------------------
# Fused neighbours of the MLP
#
# "Optimizing Krea 3 on AMD Instinct MI355X", section "Fusion cut intermediate
# memory traffic": the MLP's gate and up projections merge with the SwiGLU
# activation; modulation merges with RMSNorm; an output projection merges with
# its gate and the residual add. "Creating Custom Kernels for the AMD MI300",
# sections "Fused RMS Norm Kernel" and "Fused SwiGLU Kernel": row-wise RMS
# normalisation and the SwiGLU activation, each followed by the quantization of
# its output in the same kernel.
# --------------------------------------------------------------------------

def silu(v) -> np.ndarray:
    """SiLU in fp64: v * sigmoid(v) = v / (1 + exp(-v)).

    For v below about -709, exp(-v) overflows to +inf and the quotient is -0,
    the correctly rounded value of a number below 1e-300 in magnitude.
    """
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def swiglu_up_projection(xq_codes, xq_scales, wgu_codes, wgu_scales, bgu_bits):
    """Gate and up projections as one stacked GEMM, SwiGLU epilogue, fp64.

    The stacked weight holds the F gate rows first and the F up rows after them
    (N = 2F rows of K, each row quantized on its own, so stacking is a plain
    concatenation of the two MXFP6 weights); the stacked bias likewise [b_g; b_u].
      g = x W_g^T + b_g,  u = x W_u^T + b_u,  h = silu(g) * u.
    Returns h [M][F] in fp64. As for the GELU epilogue, parity requantizes the
    GPU's own fp32 h (quantize_f32).
    """
    c = gemm(xq_codes, xq_scales, wgu_codes, wgu_scales, bgu_bits)
    f = c.shape[1] // 2
    return silu(c[:, :f]) * c[:, f:]


def gated_mlp(x_bits, wgu_codes, wgu_scales, bgu_bits, w2_codes, w2_scales, b2_bits):
    """The SwiGLU MLP, independent of any GPU value.

    x (BF16) -> MXFP6 -> stacked gate/up projection + SwiGLU -> rounded to fp32
    -> MXFP6 -> down-projection + bias. Same readings as mlp().
    Returns (y fp64 [M][d], intermediate dict).
    """
    xq, xs = quantize_bf16(x_bits)
    h = swiglu_up_projection(xq, xs, wgu_codes, wgu_scales, bgu_bits)
    hq, hs = quantize_f32(h.astype(np.float32))
    y = down_projection(hq, hs, w2_codes, w2_scales, b2_bits)
    return y, {"xq": xq, "xs": xs, "h": h, "hq": hq, "hs": hs}


def rms_norm_modulate(x_bits, shift_bits, scale_bits, eps: float) -> np.ndarray:
    """Row-wise RMS normalisation followed by modulation, fp64.

      y[m][k] = x[m][k] / sqrt(mean_k' x[m][k']^2 + eps) * (1 + scale[k]) + shift[k]

    x is BF16 [M][K]; shift and scale are BF16 [K] (one conditioning vector per
    sample; this library's workloads are one sample). Readings: the norm carries
    no learned weight of its own (the modulation is its affine part) and eps is
    added to the mean square inside the root. The quantizer that follows rounds
    y to fp32 first (the precision the fused kernel keeps), so parity
    requantizes the GPU's own fp32 y (quantize_f32).
    """
    x = bf16_bits_to_f64(x_bits)
    shift = bf16_bits_to_f64(shift_bits)
    scale = bf16_bits_to_f64(scale_bits)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * (1.0 + scale) + shift


def gate_residual(c, gate_bits, residual_bits) -> np.ndarray:
    """Output-projection epilogue with gate and residual, fp64.

      y[m][n] = residual[m][n] + gate[n] * c[m][n]

    c is the projection with its bias already added (gemm(..., bias)); gate is
    BF16 [N] (one conditioning vector per sample), residual BF16 [M][N]. The BF16
    store of y is compared with tolerance.
    """
    c = np.asarray(c, dtype=np.float64)
    return bf16_bits_to_f64(residual_bits) + bf16_bits_to_f64(gate_bits)[None, :] * c


def dit_mlp_block(x_bits, shift_bits, scale_bits, gate_bits, eps: float, w_up_codes, w_up_scales, b_up_bits,
                  w2_codes, w2_scales, b2_bits, activation: str = "gelu"):
    """The MLP half of a diffusion-transformer block, independent of any GPU value.

      y = x + gate * (MLP(MXFP6(rms_norm_modulate(x))) + b2)

    with MLP = up-projection + activation ("gelu": tanh-GELU, w_up is W1 [F][d];
    "swiglu": w_up is the stacked [W_g; W_u] [2F][d]), the intermediate rounded
    to fp32 and requantized, then the down-projection. Each rounding to fp32
    before a quantization is the reading the fused kernels take.
    Returns (y fp64 [M][d], intermediate dict).
    """
    a = rms_norm_modulate(x_bits, shift_bits, scale_bits, eps)
    xq, xs = quantize_f32(a.astype(np.float32))
    if activation == "gelu":
        h = up_projection(xq, xs, w_up_codes, w_up_scales, b_up_bits)
    elif activation == "swiglu":
        h = swiglu_up_projection(xq, xs, w_up_codes, w_up_scales, b_up_bits)
    else:
        raise ValueError(f"unknown activation {activation!r}")
    hq, hs = quantize_f32(h.astype(np.float32))
    c = down_projection(hq, hs, w2_codes, w2_scales, b2_bits)
    y = gate_residual(c, gate_bits, x_bits)
    return y, {"a": a, "xq": xq, "xs": xs, "h": h, "hq": hq, "hs": hs, "c": c}
