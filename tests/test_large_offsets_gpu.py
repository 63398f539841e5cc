"""Maximum sizes: every kernel at tensor sizes whose element offsets pass 2^31 and
whose byte offsets pass 2^31 or 2^32, with ragged row counts, checked on the rows
that straddle each of those boundaries, the first and last rows and seeded
random rows.

A 32-bit offset anywhere (a source row, a code or scale store, the debug hooks)
would move or wrap exactly those rows. The BF16 inputs of the quantizers hold
several GB, so the device fills them with the counter-based generator of the
synthetic-input module, and the oracle regenerates only the checked rows on the
host. The MXFP6 GEMM operands are drawn on the host as usual. Tolerances and
exactness are those of the small-size tests: quantizer codes bit-exact, GEMM
outputs within 2^-7 |ref| + 1e-3 rms(ref), and requantized codes bit-exact given
the kernel's own fp32 values.
"""

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import (REL_TOL, RMS_TOL, assert_codes_equal, assert_gemm_close, assert_swiglu_close, bf16_from_device,
                    bf16_to_device, f32_from_bf16_bits, mx_upload, requant_flip_report)
from test_norm_block_gpu import assert_norm_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# quantizers: 1,300,001 rows (33 in the last 128-row group) of K = 2304
QR, QK = 1_300_001, 2304
# GEMMs: M = 245,837 (77 rows in the last tile) x N = 12288, K = 256
GM, GN, GK = 245_837, 12288, 256


def _rows(m: int, boundaries, seed: int) -> np.ndarray:
    """Rows that straddle each boundary (the row holding it and the next), the
    first and last rows, the first rows of a tile, and eight seeded random rows."""
    picked = {0, 1, 127, 128, 255, 256, m - 3, m - 2, m - 1}
    for b in boundaries:
        picked |= {b, b + 1}
    picked |= set(np.random.default_rng(seed).integers(0, m, size=8).tolist())
    return np.array(sorted(r for r in picked if 0 <= r < m), dtype=np.int64)


def _crossing_row(byte_boundary: int, row_bytes: int) -> int:
    return byte_boundary // row_bytes


def _codes_rows(mxt, rows) -> np.ndarray:
    import torch

    idx = torch.as_tensor(rows, device=mxt.codes.device)
    return O.unpack_codes(mxt.codes.index_select(0, idx).cpu().numpy(), mxt.k)


def _scale_rows(mxt, rows) -> np.ndarray:
    """Plain scales of the given rows, read from their 128-row groups of the tiled
    array only (each group is one contiguous run of (K/128) 512-byte atoms)."""
    group = (mxt.k // 128) * 512
    out = []
    for r in rows:
        g = int(r) // 128
        chunk = mxt.scales[g * group:(g + 1) * group].cpu().numpy()
        out.append(O.scales_tiled_to_plain(chunk, 128, mxt.k)[int(r) % 128])
    return np.stack(out)


def _padding_scales_zero(mxt):
    """The scale rows past the last row, up to the 128-row boundary, are zero."""
    rows, group = mxt.rows, (mxt.k // 128) * 512
    if rows % 128 == 0:
        return
    g = rows // 128
    chunk = mxt.scales[g * group:(g + 1) * group].cpu().numpy()
    assert not O.scales_tiled_to_plain(chunk, 128, mxt.k)[rows % 128:].any()


def _free():
    import torch

    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _hash_input(seed: int):
    import torch

    x = torch.empty((QR, QK), dtype=torch.bfloat16, device="cuda")
    return synth.hash_bf16_fill_(x, seed=seed)


def test_quantize_beyond_32bit_offsets(lib):
    """x: 3.0e9 elements, 6.0 GB (source offsets past 2^31 elements and 2^32 bytes);
    codes: 2.25 GB (store offsets past 2^31 bytes)."""
    x = _hash_input(seed=11)
    q = lib.mx_quantize(x)
    del x
    rows = _rows(QR, [_crossing_row(1 << 31, QK), _crossing_row(1 << 31, QK * 3 // 4)], seed=1)
    ref_codes, ref_scales = O.quantize_bf16(synth.hash_bf16_rows(rows, QK, seed=11))
    assert_codes_equal(_codes_rows(q, rows), ref_codes, _scale_rows(q, rows), ref_scales,
                       f"quantize {QR}x{QK} rows {rows.tolist()}")
    _padding_scales_zero(q)
    del q
    _free()


def test_norm_quantize_beyond_32bit_offsets(lib):
    """The fused RMSNorm + modulation quantizer on the same input, with its fp32
    debug output (12 GB: offsets past 2^33 bytes)."""
    import torch

    rng = np.random.default_rng(12)
    shift = synth.bf16_round((rng.standard_normal(QK) * 0.5).astype(np.float32))
    scale = synth.bf16_round((rng.standard_normal(QK) * 0.5).astype(np.float32))
    x = _hash_input(seed=12)
    dbg = torch.full((QR, QK), float("nan"), dtype=torch.float32, device="cuda")
    out_dbg = lib.mx_quantize_rmsnorm_modulate(x, bf16_to_device(shift), bf16_to_device(scale), 1e-6, debug_y=dbg)
    out = lib.mx_quantize_rmsnorm_modulate(x, bf16_to_device(shift), bf16_to_device(scale), 1e-6)
    del x
    assert torch.equal(out.codes, out_dbg.codes) and torch.equal(out.scales, out_dbg.scales)
    del out_dbg
    rows = _rows(QR, [_crossing_row(1 << 32, 4 * QK), _crossing_row(1 << 33, 4 * QK),
                      _crossing_row(1 << 31, QK * 3 // 4)], seed=2)
    y = dbg.index_select(0, torch.as_tensor(rows, device="cuda")).cpu().numpy()
    del dbg
    assert np.isfinite(y).all()
    assert_norm_close(y, synth.hash_bf16_rows(rows, QK, seed=12), shift, scale, 1e-6, "norm y")
    rc, rs = O.quantize_f32(y)
    assert_codes_equal(_codes_rows(out, rows), rc, _scale_rows(out, rows), rs, "norm codes")
    _padding_scales_zero(out)
    del out
    _free()


def test_quantize_gemm_beyond_32bit_offsets(lib):
    """The GEMM that quantizes its own activations, on the quantizers' 6.0 GB input
    (x offsets past 2^31 elements and 2^32 bytes; its MXFP6 codes, written into the
    workspace, past 2^31 bytes), N = 12288, so every row past the first 512 is
    encoded by the GEMM's quantizer warps; the BF16 output holds 32 GB (store
    offsets past 2^34 bytes). The in-kernel codes and scales are bit-exact against
    the oracle on the boundary rows, padding-row scales zero, and the output within
    the GEMM tolerance."""
    import torch

    rng = np.random.default_rng(14)
    w_bits = synth.bf16_round(rng.standard_normal((GN, QK)).astype(np.float32) * 0.02)
    bias = synth.bf16_round((rng.standard_normal(GN) * 0.01).astype(np.float32))
    wq = lib.mx_quantize(bf16_to_device(w_bits))
    x = _hash_input(seed=14)
    ws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(QR, QK), dtype=torch.uint8, device="cuda")
    y = lib.mx_quantize_gemm(x, wq, bf16_to_device(bias), lib.MX_EPI_BIAS_BF16, workspace=ws)
    del x
    xq = lib.mx_quantize_gemm_xq(ws, QR, QK)
    rows = _rows(QR, [_crossing_row(1 << 31, QK), _crossing_row(1 << 32, 2 * QK),
                      _crossing_row(1 << 31, QK * 3 // 4), _crossing_row(1 << 34, 2 * GN)], seed=4)
    rq, rs = O.quantize_bf16(synth.hash_bf16_rows(rows, QK, seed=14))
    assert_codes_equal(_codes_rows(xq, rows), rq, _scale_rows(xq, rows), rs, "in-kernel MXFP6(x)")
    _padding_scales_zero(xq)
    got = f32_from_bf16_bits(bf16_from_device(y.index_select(0, torch.as_tensor(rows, device="cuda"))))
    del y, xq, ws
    r_wq, r_ws = O.quantize_bf16(w_bits)
    assert_gemm_close(got.astype(np.float64), O.gemm(rq, rs, r_wq, r_ws, bias), "fused quantize + GEMM")
    assert lib.mx_device_error() == 0
    _free()


def _gemm_operands(seed: int):
    rng = np.random.default_rng(seed)
    a = rng.integers(0, 64, size=(GM, GK), dtype=np.uint8)
    sa = rng.integers(118, 125, size=(GM, GK // 32), dtype=np.uint8)
    b = rng.integers(0, 64, size=(GN, GK), dtype=np.uint8)
    sb = rng.integers(118, 125, size=(GN, GK // 32), dtype=np.uint8)
    bias = synth.bf16_round(rng.standard_normal(GN).astype(np.float32))
    return a, sa, b, sb, bias


def test_gemm_bf16_beyond_32bit_offsets(lib):
    """Output 3.0e9 BF16 elements, 6.0 GB: store offsets past 2^31 elements and 2^32 bytes."""
    import torch

    a, sa, b, sb, bias = _gemm_operands(13)
    y = lib.mx_gemm(mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias), lib.MX_EPI_BIAS_BF16)
    rows = _rows(GM, [_crossing_row(1 << 31, GN), _crossing_row(1 << 32, 2 * GN), GM - 77], seed=3)
    got = f32_from_bf16_bits(bf16_from_device(y.index_select(0, torch.as_tensor(rows, device="cuda"))))
    del y
    assert_gemm_close(got.astype(np.float64), O.gemm(a[rows], sa[rows], b, sb, bias), "bf16 epilogue")
    _free()


def test_gemm_gelu_requant_beyond_32bit_offsets(lib):
    """GELU + MXFP6 requantization: codes 2.27 GB (offsets past 2^31 bytes) and the
    fp32 debug output 12 GB (past 2^33 bytes)."""
    import torch

    a, sa, b, sb, bias = _gemm_operands(14)
    A, B, bias_d = mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias)
    dbg = torch.full((GM, GN), float("nan"), dtype=torch.float32, device="cuda")
    out_dbg = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=dbg)
    out = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_GELU_MXFP6)
    assert torch.equal(out.codes, out_dbg.codes) and torch.equal(out.scales, out_dbg.scales)
    del out_dbg
    rows = _rows(GM, [_crossing_row(1 << 32, 4 * GN), _crossing_row(1 << 33, 4 * GN),
                      _crossing_row(1 << 31, GN * 3 // 4), GM - 77], seed=4)
    g = dbg.index_select(0, torch.as_tensor(rows, device="cuda")).cpu().numpy()
    del dbg
    assert np.isfinite(g).all()
    assert_gemm_close(g, O.up_projection(a[rows], sa[rows], b, sb, bias), "gelu pre-quant")
    rc, rs = O.quantize_f32(g)
    assert_codes_equal(_codes_rows(out, rows), rc, _scale_rows(out, rows), rs, "gelu requant")
    _padding_scales_zero(out)
    del out
    _free()


def test_gemm_swiglu_requant_beyond_32bit_offsets(lib):
    """SwiGLU on a stacked [W_g; W_u] of 2 x 12288 rows: codes of h 2.27 GB (offsets
    past 2^31 bytes), the fp32 debug output 12 GB (past 2^33 bytes)."""
    import torch

    rng = np.random.default_rng(16)
    a, sa, _, _, _ = _gemm_operands(16)
    b = rng.integers(0, 64, size=(2 * GN, GK), dtype=np.uint8)
    sb = rng.integers(118, 125, size=(2 * GN, GK // 32), dtype=np.uint8)
    bias = synth.bf16_round(rng.standard_normal(2 * GN).astype(np.float32))
    A, B, bias_d = mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias)
    dbg = torch.full((GM, GN), float("nan"), dtype=torch.float32, device="cuda")
    out_dbg = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_SWIGLU_MXFP6, debug_prequant=dbg)
    out = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_SWIGLU_MXFP6)
    assert torch.equal(out.codes, out_dbg.codes) and torch.equal(out.scales, out_dbg.scales)
    del out_dbg, A, B
    rows = _rows(GM, [_crossing_row(1 << 32, 4 * GN), _crossing_row(1 << 33, 4 * GN),
                      _crossing_row(1 << 31, GN * 3 // 4), GM - 77], seed=6)
    h = dbg.index_select(0, torch.as_tensor(rows, device="cuda")).cpu().numpy()
    del dbg
    assert np.isfinite(h).all()
    assert_swiglu_close(h, O.gemm(a[rows], sa[rows], b, sb, bias), "swiglu pre-quant")
    rc, rs = O.quantize_f32(h)
    assert_codes_equal(_codes_rows(out, rows), rc, _scale_rows(out, rows), rs, "swiglu requant")
    _padding_scales_zero(out)
    del out
    _free()


def test_gemm_gate_residual_in_place_beyond_32bit_offsets(lib):
    """Gate + residual, in place on a 6.0 GB BF16 residual: loads and stores at
    element offsets past 2^31 and byte offsets past 2^32."""
    import torch

    a, sa, b, sb, bias = _gemm_operands(17)
    rng = np.random.default_rng(17)
    gate = synth.bf16_round((rng.standard_normal(GN) * 0.5).astype(np.float32))
    y = torch.empty((GM, GN), dtype=torch.bfloat16, device="cuda")
    synth.hash_bf16_fill_(y, seed=17)
    out = lib.mx_gemm_gate_residual(mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias), bf16_to_device(gate),
                                    y, out=y)
    assert out.data_ptr() == y.data_ptr()
    rows = _rows(GM, [_crossing_row(1 << 31, GN), _crossing_row(1 << 32, 2 * GN), GM - 77], seed=7)
    got = f32_from_bf16_bits(bf16_from_device(y.index_select(0, torch.as_tensor(rows, device="cuda"))))
    del y, out
    c = O.gemm(a[rows], sa[rows], b, sb, bias)
    ref = O.gate_residual(c, gate, synth.hash_bf16_rows(rows, GN, seed=17))
    gate_f = f32_from_bf16_bits(gate).astype(np.float64)
    bound = (np.abs(gate_f)[None, :] * (REL_TOL * np.abs(c) + RMS_TOL * np.sqrt(np.mean(c ** 2))) +
             2.0 ** -8 * np.abs(ref) + 1e-30)
    err = np.abs(got.astype(np.float64) - ref)
    assert not (err > bound).any(), f"{int((err > bound).sum())} outside, worst {float((err / bound).max())}"
    _free()


def test_mlp_beyond_32bit_offsets(lib):
    """mx_mlp at M = 240,077 tokens, d = 3072, ff = 12288: the MXFP6 intermediate in
    its workspace holds 2.2 GB (offsets past 2^31 bytes). Activations from the
    counter-based generator, weights of the full DiT MLP workload. Stage-wise on the
    boundary rows as in the full-size MLP tests, then end to end against an
    independent oracle run (differing codes only near rounding boundaries)."""
    import torch

    from mxutil import gemm_tolerance_report

    M, d, ff = 240_077, 3072, 12288
    w = synth.full_mlp(M=1, d=d, ff=ff)
    x = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
    synth.hash_bf16_fill_(x, seed=15)
    w1q = lib.mx_quantize(bf16_to_device(w["w1"]))
    w2q = lib.mx_quantize(bf16_to_device(w["w2"]))
    b1, b2 = bf16_to_device(w["b1"]), bf16_to_device(w["b2"])
    y = lib.mx_mlp(x, w1q, b1, w2q, b2)
    xq = lib.mx_quantize(x)
    del x
    dbg = torch.empty((M, ff), dtype=torch.float32, device="cuda")
    hq = lib.mx_gemm(xq, w1q, b1, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=dbg)
    assert torch.equal(y, lib.mx_gemm(hq, w2q, b2, lib.MX_EPI_BIAS_BF16)), "mx_mlp differs from its three stages"

    rows = _rows(M, [_crossing_row(1 << 32, 4 * ff), _crossing_row(1 << 33, 4 * ff),
                     _crossing_row(1 << 31, ff * 3 // 4), M - 77], seed=5)
    idx = torch.as_tensor(rows, device="cuda")
    x_rows = synth.hash_bf16_rows(rows, d, seed=15)
    r_w1q, r_w1s = O.quantize_bf16(w["w1"])
    r_w2q, r_w2s = O.quantize_bf16(w["w2"])
    rxq, rxs = O.quantize_bf16(x_rows)
    assert_codes_equal(_codes_rows(xq, rows), rxq, _scale_rows(xq, rows), rxs, "xq")
    g = dbg.index_select(0, idx).cpu().numpy()
    del dbg
    assert_gemm_close(g, O.up_projection(rxq, rxs, r_w1q, r_w1s, w["b1"]), "gelu(x W1^T + b1)")
    ghq, ghs = _codes_rows(hq, rows), _scale_rows(hq, rows)
    rhq, rhs = O.quantize_f32(g)
    assert_codes_equal(ghq, rhq, ghs, rhs, "hq")
    _padding_scales_zero(hq)
    got = f32_from_bf16_bits(bf16_from_device(y.index_select(0, idx))).astype(np.float64)
    assert_gemm_close(got, O.down_projection(ghq, ghs, r_w2q, r_w2s, w["b2"]), "y")
    # end to end against an independent oracle run: every intermediate code that
    # differs lies within the stage-2 tolerance of a rounding boundary, and the
    # output within the GEMM tolerance plus those codes' exact contribution
    y_ref, mid = O.mlp(x_rows, r_w1q, r_w1s, w["b1"], r_w2q, r_w2s, w["b2"])
    g_tol = REL_TOL * np.abs(mid["g"]) + RMS_TOL * np.sqrt(np.mean(mid["g"] ** 2))
    requant_flip_report(ghq, ghs, mid["hq"], mid["hs"], mid["g"].astype(np.float32), g_tol)
    c_gpu = O.down_projection(ghq, ghs, r_w2q, r_w2s, w["b2"])
    bound = REL_TOL * np.abs(c_gpu) + RMS_TOL * np.sqrt(np.mean(c_gpu ** 2)) + np.abs(c_gpu - y_ref)
    assert not (np.abs(got - y_ref) > bound).any(), gemm_tolerance_report(got, y_ref)
    assert lib.mx_device_error() == 0
    del y, xq, hq
    _free()
