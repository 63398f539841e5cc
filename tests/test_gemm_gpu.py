"""K2/K3 parity: the tcgen05 block-scaled GEMM against the fp64 oracle.

Structured cases first (they pin the operand, swizzle and scale layouts one at a
time), then seeded random multi-tile shapes with ragged M, then the two DiT
projections at full size on sampled rows. Tolerance: |gpu - oracle| <=
2^-7 |oracle| + 1e-3 rms(oracle). The fused requantization is bit-exact given the
kernel's own fp32 GELU output, which the debug hook exports.
"""

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import (assert_codes_equal, assert_gemm_close, bf16_from_device, bf16_to_device, f32_from_bf16_bits,
                    mx_rows_to_host, mx_to_host, mx_upload, sample_rows)

pytestmark = pytest.mark.gpu


def _gemm_bf16(lib, a, b, bias_bits=None):
    bias = None if bias_bits is None else bf16_to_device(bias_bits)
    y = lib.mx_gemm(a, b, bias, lib.MX_EPI_BIAS_BF16)
    return f32_from_bf16_bits(bf16_from_device(y)).astype(np.float64)


def _unit(rows, k, code=0x08, scale=127):
    return np.full((rows, k), code, np.uint8), np.full((rows, k // 32), scale, np.uint8)


def test_all_ones_unit_scales(lib):
    a, sa = _unit(128, 128)
    b, sb = _unit(256, 128)
    y = _gemm_bf16(lib, mx_upload(a, sa), mx_upload(b, sb))
    assert np.all(y == 128.0), np.unique(y)[:10]


def test_code_bit_order_one_hot(lib):
    """A[m][k] = 1.0 at k = m % K only: C[m][n] = deq(B)[n][m % K] exposes the code order."""
    M, N, K = 128, 256, 128
    a = np.zeros((M, K), np.uint8)
    a[np.arange(M), np.arange(M) % K] = 0x08
    sa = np.full((M, K // 32), 127, np.uint8)
    rng = np.random.default_rng(1)
    b = rng.integers(0, 64, size=(N, K)).astype(np.uint8)
    sb = np.full((N, K // 32), 127, np.uint8)
    y = _gemm_bf16(lib, mx_upload(a, sa), mx_upload(b, sb))
    want = O.gemm(a, sa, b, sb)
    bad = np.argwhere(y != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first {bad[:5].tolist()}: {y[tuple(bad[:5].T)]} vs {want[tuple(bad[:5].T)]}"


@pytest.mark.parametrize("which", ["a", "b"])
def test_scale_layout(lib, which):
    """All codes 1.0; one operand's scales vary per (row, K-block): exposes the tiled scale layout."""
    M, N, K = 256, 512, 512
    rng = np.random.default_rng(2 if which == "a" else 3)
    a, sa = _unit(M, K)
    b, sb = _unit(N, K)
    if which == "a":
        sa = rng.integers(120, 135, size=sa.shape).astype(np.uint8)
    else:
        sb = rng.integers(120, 135, size=sb.shape).astype(np.uint8)
    y = _gemm_bf16(lib, mx_upload(a, sa), mx_upload(b, sb))
    assert_gemm_close(y, O.gemm(a, sa, b, sb), f"scale layout {which}")


def test_pr1(lib):
    w = synth.pr1()
    xq = lib.mx_quantize(bf16_to_device(w["x"]))
    wq = lib.mx_quantize(bf16_to_device(w["w"]))
    y = _gemm_bf16(lib, xq, wq, w["b"])
    rxq, rxs = O.quantize_bf16(w["x"])
    rwq, rws = O.quantize_bf16(w["w"])
    assert_gemm_close(y, O.gemm(rxq, rxs, rwq, rws, w["b"]), "pr1")


def _random_mx(rng, rows, k, lo=110, hi=140):
    codes = rng.integers(0, 64, size=(rows, k)).astype(np.uint8)
    scales = rng.integers(lo, hi, size=(rows, k // 32)).astype(np.uint8)
    return codes, scales


@pytest.mark.parametrize("M,N,K", [(300, 768, 640), (128, 256, 128), (1, 256, 128), (129, 512, 256),
                                   (1000, 1024, 1152)])
def test_random_multitile_bias_bf16(lib, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, N, K)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32) * 1000)
    y = _gemm_bf16(lib, mx_upload(a, sa), mx_upload(b, sb), bias)
    assert_gemm_close(y, O.gemm(a, sa, b, sb, bias), f"bf16 {M}x{N}x{K}")


def test_no_bias(lib):
    rng = np.random.default_rng(4)
    a, sa = _random_mx(rng, 200, 256)
    b, sb = _random_mx(rng, 256, 256)
    y = _gemm_bf16(lib, mx_upload(a, sa), mx_upload(b, sb), None)
    assert_gemm_close(y, O.gemm(a, sa, b, sb), "no bias")


def _gelu_mx(lib, a, b, bias_bits, m, n):
    import torch

    bias = bf16_to_device(bias_bits)
    dbg = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    out_dbg = lib.mx_gemm(a, b, bias, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=dbg)
    out = lib.mx_gemm(a, b, bias, lib.MX_EPI_BIAS_GELU_MXFP6)
    # the production variant writes exactly what the instrumented one does
    assert torch.equal(out.codes, out_dbg.codes) and torch.equal(out.scales, out_dbg.scales)
    return out, dbg


@pytest.mark.parametrize("M,N,K", [(300, 768, 640), (129, 256, 128), (512, 1024, 1024)])
def test_random_multitile_gelu_requant(lib, M, N, K):
    rng = np.random.default_rng(10 * M + N + K)
    a, sa = _random_mx(rng, M, K, 118, 124)
    b, sb = _random_mx(rng, N, K, 118, 124)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32))
    out, dbg = _gelu_mx(lib, mx_upload(a, sa), mx_upload(b, sb), bias, M, N)
    g = dbg.cpu().numpy()
    assert np.isfinite(g).all()
    assert_gemm_close(g, O.up_projection(a, sa, b, sb, bias), f"gelu pre-quant {M}x{N}x{K}")
    codes, scales = mx_to_host(out)
    rc, rs = O.quantize_f32(g)
    assert_codes_equal(codes, rc, scales, rs, f"requant {M}x{N}x{K}")
    tiled = out.scales.cpu().numpy()
    assert np.count_nonzero(tiled) == np.count_nonzero(O.scales_plain_to_tiled(rs, M, N))


@pytest.mark.slow
def test_dit_up_projection_full_size(lib):
    """M=4096, K=3072, N=12288, fused bias + GELU + MXFP6 requant, sampled rows."""
    w = synth.dit_up()
    xq = lib.mx_quantize(bf16_to_device(w["x"]))
    wq = lib.mx_quantize(bf16_to_device(w["w"]))
    M, N = 4096, 12288
    out, dbg = _gelu_mx(lib, xq, wq, w["b"], M, N)
    rows = sample_rows(M)
    rxq, rxs = O.quantize_bf16(w["x"][rows])
    gxq, gxs = mx_rows_to_host(xq, rows)
    assert_codes_equal(gxq, rxq, gxs, rxs, "x rows")
    rwq, rws = O.quantize_bf16(w["w"])
    g = dbg.cpu().numpy()[rows]
    assert_gemm_close(g, O.up_projection(rxq, rxs, rwq, rws, w["b"]), "up pre-quant")
    codes, scales = mx_rows_to_host(out, rows)
    rc, rs = O.quantize_f32(g)
    assert_codes_equal(codes, rc, scales, rs, "up requant")
    assert lib.mx_device_error() == 0


@pytest.mark.slow
def test_dit_down_projection_full_size(lib):
    """M=16384, K=12288, N=3072, bias + BF16 store; input MXFP6 of BF16(GELU(z)), sampled rows."""
    import torch

    w = synth.dit_down()
    z = torch.from_numpy(w["z"]).cuda()
    h_bf16 = torch.nn.functional.gelu(z, approximate="tanh").to(torch.bfloat16)
    del z
    hq = lib.mx_quantize(h_bf16)
    w2q = lib.mx_quantize(bf16_to_device(w["w"]))
    y = lib.mx_gemm(hq, w2q, bf16_to_device(w["b"]), lib.MX_EPI_BIAS_BF16)
    rows = sample_rows(16384)
    h_rows = bf16_from_device(h_bf16[torch.as_tensor(rows, device="cuda")])
    rhq, rhs = O.quantize_bf16(h_rows)
    ghq, ghs = mx_rows_to_host(hq, rows)
    assert_codes_equal(ghq, rhq, ghs, rhs, "h rows")
    rwq, rws = O.quantize_bf16(w["w"])
    ref = O.gemm(rhq, rhs, rwq, rws, w["b"])
    got = f32_from_bf16_bits(bf16_from_device(y[torch.as_tensor(rows, device="cuda")])).astype(np.float64)
    assert_gemm_close(got, ref, "down")
    assert lib.mx_device_error() == 0


def test_no_device_errors(lib):
    assert lib.mx_device_error() == 0


def test_extreme_scale_exponents(lib):
    """E8M0 scales over the whole range (codes 1..254) on both operands, paired so
    that every product 2^(sa + sb - 254) stays inside fp32's normal range: K-block j
    gives B a scale near a code drawn across 1..254 and A the complementary one, so
    the tensor cores must apply the full scale range exactly (bias-free, BF16 store)."""
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(11)
    a = rng.integers(0, 64, size=(M, K)).astype(np.uint8)
    b = rng.integers(0, 64, size=(N, K)).astype(np.uint8)
    kb = K // 32
    base_b = rng.permutation(np.linspace(4, 250, kb).round().astype(np.int64))
    d = rng.integers(-6, 7, size=kb)                       # per-block size of the products
    sb = base_b[None, :] + rng.integers(-3, 4, size=(N, kb))
    sa = (254 + d - base_b)[None, :] + rng.integers(-3, 4, size=(M, kb))
    assert sa.min() >= 1 and sa.max() <= 254 and sb.min() >= 1 and sb.max() <= 254
    sa, sb = sa.astype(np.uint8), sb.astype(np.uint8)
    y = _gemm_bf16(lib, mx_upload(a, sa), mx_upload(b, sb))
    assert_gemm_close(y, O.gemm(a, sa, b, sb), "extreme scales")


def test_nan_scale_block_propagates(lib):
    """A block whose E8M0 scale is 0xFF (NaN: what the quantizer writes for a block
    holding Inf/NaN) makes every output that sums it NaN, as in the oracle; other
    rows are unaffected; a requantizing epilogue turns the NaN row into NaN blocks."""
    M, N, K = 128, 256, 256
    rng = np.random.default_rng(12)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, N, K)
    sa = sa.copy()
    a = a.copy()
    sa[5, 2] = 0xFF
    a[5, 64:96] = 0
    y = _gemm_bf16(lib, mx_upload(a, sa), mx_upload(b, sb))
    ref = O.gemm(a, sa, b, sb)
    assert np.isnan(ref[5]).all()
    assert np.isnan(y[5]).all(), f"row 5: {np.isnan(y[5]).sum()} NaN of {N}, sample {y[5, :4]}"
    keep = np.arange(M) != 5
    assert_gemm_close(y[keep], ref[keep], "rows without the NaN block")
    # through the GELU + requantization epilogue: the NaN row's blocks get scale 0xFF
    # and zero codes, the quantizer's rule for a block holding NaN
    bias = np.zeros(N, np.uint16)
    out, dbg = _gelu_mx(lib, mx_upload(a, sa), mx_upload(b, sb), bias, M, N)
    g = dbg.cpu().numpy()
    assert np.isnan(g[5]).all()
    codes, scales = mx_to_host(out)
    rc, rs = O.quantize_f32(g)
    assert_codes_equal(codes, rc, scales, rs, "requant with a NaN row")
    assert (scales[5] == 0xFF).all() and (codes[5] == 0).all()
