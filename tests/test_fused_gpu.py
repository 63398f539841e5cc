"""Parity of the fused neighbours of the MLP GEMM against the fp64 oracle.

* SwiGLU up-projection (stacked [W_g; W_u] weight, MX_EPI_BIAS_SWIGLU_MXFP6):
  the kernel's fp32 h = silu(g) * u (debug hook) within the tolerance derived
  below, and the requantized codes bit-exact given that h.
* SwiGLU MLP (mx_gated_mlp): stage-wise as the GELU MLP, end to end >= 99.9%.
* Output projection with gate and residual (mx_gemm_gate_residual).
* Stacked query/key/value/gate projection: one mx_gemm with N = 4d.

Tolerance of h. The GEMM contract bounds each accumulator: |dg| <= tg =
2^-7 |g| + 1e-3 rms(g), likewise |du| <= tu. With L = max |silu'| < 1.1,
|silu(g + dg)(u + du) - silu(g) u| <= L tg (|u| + tu) + |silu(g)| tu; the fp32
evaluation (approximate 2^x and reciprocal, two roundings) adds below 1e-6 |h|.

Tolerance of the gated residual output y = r + gate (c + bias), stored as BF16:
|gate| times the GEMM bound on c, plus 2^-8 |y| for the BF16 rounding (half an
ulp is 2^-9 relative) and the fp32 fma.
"""

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import (REL_TOL, RMS_TOL, assert_codes_equal, assert_gemm_close, assert_swiglu_close,
                    bf16_from_device, bf16_to_device, f32_from_bf16_bits, gemm_tolerance_report, mx_rows_to_host,
                    mx_to_host, mx_upload, requant_flip_report, sample_rows, swiglu_bound)

pytestmark = pytest.mark.gpu

def _random_mx(rng, rows, k, lo=118, hi=124):
    codes = rng.integers(0, 64, size=(rows, k)).astype(np.uint8)
    scales = rng.integers(lo, hi, size=(rows, k // 32)).astype(np.uint8)
    return codes, scales


def _swiglu(lib, a, b, bias_bits, m, f):
    import torch

    bias = None if bias_bits is None else bf16_to_device(bias_bits)
    dbg = torch.full((m, f), float("nan"), dtype=torch.float32, device="cuda")
    out_dbg = lib.mx_gemm(a, b, bias, lib.MX_EPI_BIAS_SWIGLU_MXFP6, debug_prequant=dbg)
    out = lib.mx_gemm(a, b, bias, lib.MX_EPI_BIAS_SWIGLU_MXFP6)
    assert out.rows == m and out.k == f
    # the production variant writes exactly what the instrumented one does
    assert torch.equal(out.codes, out_dbg.codes) and torch.equal(out.scales, out_dbg.scales)
    return out, dbg


def test_swiglu_gate_and_up_halves(lib):
    """Up rows all zero with up bias 1 -> h = silu(g); gate rows zero, gate bias 1 -> h = silu(1) u.

    Exposes which half of the stacked weight each CTA of the pair stages and which
    accumulator columns the epilogue pairs."""
    M, F, K = 256, 256, 256
    rng = np.random.default_rng(21)
    a, sa = _random_mx(rng, M, K)
    for zero_half in ("up", "gate"):
        b, sb = _random_mx(rng, 2 * F, K)
        lo = F if zero_half == "up" else 0
        b[lo:lo + F] = 0
        bias = np.zeros(2 * F, np.uint16)
        bias[lo:lo + F] = synth.bf16_round(np.ones(F, np.float32))
        out, dbg = _swiglu(lib, mx_upload(a, sa), mx_upload(b, sb), bias, M, F)
        c = O.gemm(a, sa, b, sb, bias)
        assert_swiglu_close(dbg.cpu().numpy(), c, f"{zero_half} half zero")


@pytest.mark.parametrize("M,F,K", [(300, 384, 640), (129, 128, 128), (512, 1024, 1024), (1, 256, 256)])
def test_swiglu_random_multitile(lib, M, F, K):
    rng = np.random.default_rng(7 * M + F + K)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, 2 * F, K)
    bias = synth.bf16_round(rng.standard_normal(2 * F).astype(np.float32))
    out, dbg = _swiglu(lib, mx_upload(a, sa), mx_upload(b, sb), bias, M, F)
    h = dbg.cpu().numpy()
    assert np.isfinite(h).all()
    assert_swiglu_close(h, O.gemm(a, sa, b, sb, bias), f"swiglu pre-quant {M}x{F}x{K}")
    codes, scales = mx_to_host(out)
    rc, rs = O.quantize_f32(h)
    assert_codes_equal(codes, rc, scales, rs, f"swiglu requant {M}x{F}x{K}")
    tiled = out.scales.cpu().numpy()
    assert np.count_nonzero(tiled) == np.count_nonzero(O.scales_plain_to_tiled(rs, M, F))


def test_swiglu_no_bias(lib):
    rng = np.random.default_rng(23)
    M, F, K = 200, 256, 256
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, 2 * F, K)
    out, dbg = _swiglu(lib, mx_upload(a, sa), mx_upload(b, sb), None, M, F)
    assert_swiglu_close(dbg.cpu().numpy(), O.gemm(a, sa, b, sb), "swiglu no bias")


def test_quantize_stacked_is_concatenation(lib):
    import torch

    w = synth.gated_mlp(M=8, d=256, ff=384)
    parts = [bf16_to_device(w["wgu"][:384]), bf16_to_device(w["wgu"][384:])]
    st = lib.mx_quantize_stacked(parts)
    whole = lib.mx_quantize(bf16_to_device(w["wgu"]))
    assert torch.equal(st.codes, whole.codes) and torch.equal(st.scales, whole.scales)


def test_quantize_stacked_strided_parts_and_ragged_last(lib):
    """Four parts (the query/key/value/gate layout) with their own row strides, the
    last one ragged: equal to quantizing the concatenation, and to the oracle, code
    for code; the padding rows' scales are zero."""
    import torch

    rng = np.random.default_rng(21)
    k, rows = 384, [256, 128, 384, 100]
    mats = [synth.bf16_round(rng.standard_normal((r, k)).astype(np.float32) * (0.5 + i)) for i, r in enumerate(rows)]
    parts = []
    for i, m in enumerate(mats):
        pad = 8 * (i + 1)                               # row stride k + pad elements
        buf = torch.zeros((m.shape[0], k + pad), dtype=torch.bfloat16, device="cuda")
        buf[:, :k] = bf16_to_device(m)
        parts.append(buf[:, :k])
    st = lib.mx_quantize_stacked(parts)
    cat = np.concatenate(mats)
    whole = lib.mx_quantize(bf16_to_device(cat))
    assert torch.equal(st.codes, whole.codes) and torch.equal(st.scales, whole.scales)
    codes = O.unpack_codes(st.codes.cpu().numpy(), k)
    scales = O.scales_tiled_to_plain(st.scales.cpu().numpy(), sum(rows), k)
    rq, rs = O.quantize_bf16(cat)
    assert_codes_equal(codes, rq, scales, rs, "stacked")
    padded = (sum(rows) + 127) // 128 * 128
    all_scales = O.scales_tiled_to_plain(st.scales.cpu().numpy(), padded, k)
    assert np.all(all_scales[sum(rows):] == 0)


def _run_gated_mlp(lib, w, rows):
    import torch

    x = bf16_to_device(w["x"])
    M, d = w["x"].shape
    ff = w["w2"].shape[1]
    wgu = lib.mx_quantize(bf16_to_device(w["wgu"]))
    w2q = lib.mx_quantize(bf16_to_device(w["w2"]))
    bgu = bf16_to_device(w["bgu"])
    b2 = bf16_to_device(w["b2"])
    y = lib.mx_gated_mlp(x, wgu, bgu, w2q, b2)

    xq = lib.mx_quantize(x)
    dbg = torch.empty((M, ff), dtype=torch.float32, device="cuda")
    hq = lib.mx_gemm(xq, wgu, bgu, lib.MX_EPI_BIAS_SWIGLU_MXFP6, debug_prequant=dbg)
    y2 = lib.mx_gemm(hq, w2q, b2, lib.MX_EPI_BIAS_BF16)
    assert torch.equal(y, y2), "mx_gated_mlp differs from its three stages"

    idx = torch.as_tensor(rows, device="cuda")
    r_wq, r_ws = O.quantize_bf16(w["wgu"])
    r_w2q, r_w2s = O.quantize_bf16(w["w2"])
    rxq, rxs = O.quantize_bf16(w["x"][rows])
    gxq, gxs = mx_rows_to_host(xq, rows)
    assert_codes_equal(gxq, rxq, gxs, rxs, "xq")
    h = dbg[idx].cpu().numpy()
    c_up = O.gemm(rxq, rxs, r_wq, r_ws, w["bgu"])
    assert_swiglu_close(h, c_up, "silu(g) * u")
    ghq, ghs = mx_rows_to_host(hq, rows)
    rhq, rhs = O.quantize_f32(h)
    assert_codes_equal(ghq, rhq, ghs, rhs, "hq")
    got = f32_from_bf16_bits(bf16_from_device(y[idx])).astype(np.float64)
    assert_gemm_close(got, O.down_projection(ghq, ghs, r_w2q, r_w2s, w["b2"]), "y")
    # end to end against an independent oracle run: differing intermediate codes
    # only within the SwiGLU stage's tolerance of a rounding boundary, and the output
    # within the GEMM tolerance plus those codes' exact contribution
    y_ref, mid = O.gated_mlp(w["x"][rows], r_wq, r_ws, w["bgu"], r_w2q, r_w2s, w["b2"])
    flips, _ = requant_flip_report(ghq, ghs, mid["hq"], mid["hs"], mid["h"].astype(np.float32), swiglu_bound(c_up))
    c_gpu = O.down_projection(ghq, ghs, r_w2q, r_w2s, w["b2"])
    bound = REL_TOL * np.abs(c_gpu) + RMS_TOL * np.sqrt(np.mean(c_gpu ** 2)) + np.abs(c_gpu - y_ref)
    rep = gemm_tolerance_report(got, y_ref)
    rep.update(flips)
    rep["n_outside_derived_bound"] = int((np.abs(got - y_ref) > bound).sum())
    print(f"gated MLP end-to-end vs independent oracle: {rep}")
    assert rep["n_outside_derived_bound"] == 0, rep
    assert lib.mx_device_error() == 0


def test_small_gated_mlp_all_rows(lib):
    _run_gated_mlp(lib, synth.gated_mlp(M=300, d=256, ff=384), np.arange(300))


@pytest.mark.slow
def test_full_gated_mlp(lib):
    """M=20480, d=3072, ff=8192: stacked gate/up GEMM N = 16384, down-projection K = 8192."""
    _run_gated_mlp(lib, synth.gated_mlp(), sample_rows(20480, n_random=128))


# ---------------------------------------------------------------- gate + residual

def assert_gate_residual_close(y_gpu, c_ref, gate_f, y_ref, what):
    rms = np.sqrt(np.mean(c_ref * c_ref))
    bound = np.abs(gate_f)[None, :] * (REL_TOL * np.abs(c_ref) + RMS_TOL * rms) + 2.0 ** -8 * np.abs(y_ref) + 1e-30
    err = np.abs(y_gpu - y_ref)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, f"{what}: {len(bad)} outside, first {bad[:4].tolist()}"


@pytest.mark.parametrize("M,N,K,gated,in_place", [(300, 768, 640, True, False), (129, 256, 128, False, False),
                                                  (512, 512, 1024, True, True), (1, 256, 256, True, False)])
def test_gate_residual_random(lib, M, N, K, gated, in_place):
    import torch

    rng = np.random.default_rng(3 * M + N + K)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, N, K)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32))
    gate = synth.bf16_round(rng.standard_normal(N).astype(np.float32)) if gated else None
    if gate is not None:
        gate[:7] = 0   # a zero gate passes the residual through
    res = synth.bf16_round((rng.standard_normal((M, N)) * 4).astype(np.float32))
    res_dev = bf16_to_device(res)
    out = res_dev if in_place else None
    y = lib.mx_gemm_gate_residual(mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias),
                                  None if gate is None else bf16_to_device(gate), res_dev, out=out)
    if in_place:
        assert y.data_ptr() == res_dev.data_ptr()
    got = f32_from_bf16_bits(bf16_from_device(y)).astype(np.float64)
    c = O.gemm(a, sa, b, sb, bias)
    gate_bits = gate if gate is not None else synth.bf16_round(np.ones(N, np.float32))
    y_ref = O.gate_residual(c, gate_bits, res)
    gate_f = f32_from_bf16_bits(gate_bits).astype(np.float64)
    assert_gate_residual_close(got, c, gate_f, y_ref, f"gate residual {M}x{N}x{K}")
    if gate is not None:
        np.testing.assert_array_equal(bf16_from_device(y)[:, :7], res[:, :7])
    torch.cuda.synchronize()
    assert lib.mx_device_error() == 0


# ---------------------------------------------------------------- stacked QKV + gate projection

@pytest.mark.slow
def test_stacked_qkv_gate_projection_full_size(lib):
    """M=20480, K=3072, N=4*3072: the four projections that read the same normalized
    activations as one MXFP6 GEMM with a BF16 store (activations quantized once)."""
    import torch

    w = synth.qkv_proj()
    xq = lib.mx_quantize(bf16_to_device(w["x"]))
    d = w["x"].shape[1]
    parts = [bf16_to_device(w["w"][i * d:(i + 1) * d]) for i in range(4)]
    wq = lib.mx_quantize_stacked(parts)
    y = lib.mx_gemm(xq, wq, bf16_to_device(w["b"]), lib.MX_EPI_BIAS_BF16)
    rows = sample_rows(20480, n_random=96)
    rxq, rxs = O.quantize_bf16(w["x"][rows])
    rwq, rws = O.quantize_bf16(w["w"])
    ref = O.gemm(rxq, rxs, rwq, rws, w["b"])
    got = f32_from_bf16_bits(bf16_from_device(y[torch.as_tensor(rows, device="cuda")])).astype(np.float64)
    assert_gemm_close(got, ref, "qkv+gate")
    assert lib.mx_device_error() == 0
