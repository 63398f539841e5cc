"""The GEMM that quantizes its own BF16 activations (mx_quantize_gemm, and the
up-projection inside mx_mlp / mx_gated_mlp).

The quantize kernel encodes the leading rows -- those the GEMM's first round of
tiles reads; all rows when N < 12288 -- and the GEMM's quantizer warps the rest
while its main loop runs. With N = 12288 or 16384 (48 or 64 column tiles) the
first round of 76 pairs reads the first 512 rows, so on the shapes
below most rows are encoded inside the GEMM (in several 128-row blocks, the last
one ragged, with 1, 2 or 3 column strips of 1024, the last one partial); at
N = 3072 none.

Checks: the MXFP6(x) the call leaves in its workspace equals mx_quantize(x) byte
for byte (padding-row scales included), and the output equals mx_quantize followed
by mx_gemm / mx_gemm_gate_residual bit for bit (the same MMAs on the same codes).
Those two are pinned to the oracle by the quantizer and GEMM tests; sampled rows
are also compared with the oracle here, codes bit-exact and the GEMM within its
tolerance.
"""

import threading

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import (assert_codes_equal, assert_gemm_close, bf16_from_device, bf16_to_device, f32_from_bf16_bits,
                    mx_rows_to_host)

pytestmark = pytest.mark.gpu


def _inputs(seed, M, K, N, ld_pad=0):
    """BF16 activations (row stride K + ld_pad), an MXFP6 weight and a bias."""
    import torch

    rng = np.random.default_rng(seed)
    x_bits = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32) * rng.lognormal(0, 0.5, K))
    x = bf16_to_device(x_bits)
    if ld_pad:
        buf = torch.zeros((M, K + ld_pad), dtype=torch.bfloat16, device="cuda")
        buf[:, :K] = x
        x = buf[:, :K]
    w_bits = synth.bf16_round(rng.standard_normal((N, K)).astype(np.float32) * 0.02)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32) * 0.01)
    return x_bits, x, w_bits, bias


def _check_xq(lib, ws, x, x_bits, rows):
    import torch

    M, K = x_bits.shape
    got = lib.mx_quantize_gemm_xq(ws, M, K)
    ref = lib.mx_quantize(x)
    assert torch.equal(got.codes, ref.codes), "in-kernel codes differ from mx_quantize"
    assert torch.equal(got.scales, ref.scales), "in-kernel scales (padding rows included) differ from mx_quantize"
    gq, gs = mx_rows_to_host(got, rows)
    rq, rs = O.quantize_bf16(x_bits[rows])
    assert_codes_equal(gq, rq, gs, rs, "MXFP6(x)")
    return ref


def _rows(M):
    # the lead rows' last, the first encoded in-kernel, block boundaries, the last
    return np.unique(np.array([0, 511, 512, 639, 640, 1023, 1024, M // 2, M - 2, M - 1]).clip(0, M - 1))


# ld_pad 8: a row stride of 8 mod 16 elements, so the quantizer warp takes its
# 16-byte load path (32-byte loads need 32-byte aligned rows)
@pytest.mark.parametrize("M,K,N,ld_pad", [(3000, 1152, 16384, 0), (2000, 384, 12288, 64), (1300, 3072, 12288, 0),
                                          (1500, 512, 12288, 8)])
def test_bf16_epilogue(lib, M, K, N, ld_pad):
    import torch

    x_bits, x, w_bits, bias = _inputs(M + K, M, K, N, ld_pad)
    wq = lib.mx_quantize(bf16_to_device(w_bits))
    b = bf16_to_device(bias)
    ws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y = lib.mx_quantize_gemm(x, wq, b, lib.MX_EPI_BIAS_BF16, workspace=ws)
    rows = _rows(M)
    xq = _check_xq(lib, ws, x, x_bits, rows)
    assert torch.equal(y, lib.mx_gemm(xq, wq, b, lib.MX_EPI_BIAS_BF16, split=False)), "differs from the two calls"
    # a second call on the same workspace (the counters are zeroed again)
    y2 = lib.mx_quantize_gemm(x, wq, b, lib.MX_EPI_BIAS_BF16, workspace=ws)
    assert torch.equal(y, y2)
    rq, rs = O.quantize_bf16(x_bits[rows])
    wq_r, ws_r = O.quantize_bf16(w_bits)
    got = f32_from_bf16_bits(bf16_from_device(y[torch.as_tensor(rows, device="cuda")])).astype(np.float64)
    assert_gemm_close(got, O.gemm(rq, rs, wq_r, ws_r, bias), "x W^T + b")
    assert lib.mx_device_error() == 0


def test_gelu_requant_epilogue(lib):
    import torch

    M, K, N = 2500, 2176, 12288
    x_bits, x, w_bits, bias = _inputs(7, M, K, N)
    wq = lib.mx_quantize(bf16_to_device(w_bits))
    b = bf16_to_device(bias)
    ws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    hq = lib.mx_quantize_gemm(x, wq, b, lib.MX_EPI_BIAS_GELU_MXFP6, workspace=ws)
    xq = _check_xq(lib, ws, x, x_bits, _rows(M))
    ref = lib.mx_gemm(xq, wq, b, lib.MX_EPI_BIAS_GELU_MXFP6)
    assert torch.equal(hq.codes, ref.codes) and torch.equal(hq.scales, ref.scales)
    assert lib.mx_device_error() == 0


def test_swiglu_epilogue(lib):
    import torch

    M, K, F = 1800, 1024, 6144
    x_bits, x, w_bits, bias = _inputs(8, M, K, 2 * F)
    wq = lib.mx_quantize(bf16_to_device(w_bits))
    b = bf16_to_device(bias)
    ws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    hq = lib.mx_quantize_gemm(x, wq, b, lib.MX_EPI_BIAS_SWIGLU_MXFP6, workspace=ws)
    assert hq.rows == M and hq.k == F
    xq = _check_xq(lib, ws, x, x_bits, _rows(M))
    ref = lib.mx_gemm(xq, wq, b, lib.MX_EPI_BIAS_SWIGLU_MXFP6)
    assert torch.equal(hq.codes, ref.codes) and torch.equal(hq.scales, ref.scales)
    assert lib.mx_device_error() == 0


@pytest.mark.parametrize("gated,in_place,N", [(True, True, 12288), (False, False, 12288), (True, False, 3072)])
def test_gate_residual_epilogue(lib, gated, in_place, N):
    import torch

    M, K = 1700 if N > 3072 else 5000, 640
    x_bits, x, w_bits, bias = _inputs(9 + gated, M, K, N)
    rng = np.random.default_rng(5)
    gate = bf16_to_device(synth.bf16_round(rng.standard_normal(N).astype(np.float32))) if gated else None
    res = bf16_to_device(synth.bf16_round(rng.standard_normal((M, N)).astype(np.float32)))
    res_copy = res.clone()
    wq = lib.mx_quantize(bf16_to_device(w_bits))
    b = bf16_to_device(bias)
    ws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y = lib.mx_quantize_gemm(x, wq, b, lib.MX_EPI_GATE_RESIDUAL_BF16, gate=gate, residual=res,
                             out=res if in_place else None, workspace=ws)
    if in_place:
        assert y.data_ptr() == res.data_ptr()
    xq = _check_xq(lib, ws, x, x_bits, _rows(M))
    ref = lib.mx_gemm_gate_residual(xq, wq, b, gate, res_copy, split=False)
    assert torch.equal(y, ref)
    assert lib.mx_device_error() == 0


def test_rows_all_in_the_lead(lib):
    """N = 512: the first round reads every row, so the quantize kernel encodes
    all of x and the GEMM runs without its quantizer warp."""
    import torch

    M, K, N = 700, 256, 512
    x_bits, x, w_bits, bias = _inputs(11, M, K, N)
    wq = lib.mx_quantize(bf16_to_device(w_bits))
    b = bf16_to_device(bias)
    ws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y = lib.mx_quantize_gemm(x, wq, b, lib.MX_EPI_BIAS_BF16, workspace=ws)
    xq = _check_xq(lib, ws, x, x_bits, np.array([0, 255, 256, M - 1]))
    assert torch.equal(y, lib.mx_gemm(xq, wq, b, lib.MX_EPI_BIAS_BF16))


def test_empty(lib):
    import torch

    wq = lib.mx_quantize(bf16_to_device(np.zeros((12288, 256), np.uint16)))
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    y = lib.mx_quantize_gemm(x, wq, None, lib.MX_EPI_BIAS_BF16)
    assert y.shape == (0, 12288)


@pytest.mark.parametrize("gated", [False, True])
def test_mlp_up_projection_quantizes_in_kernel(lib, gated):
    """mx_mlp / mx_gated_mlp at M = 2048, ff = 12288: the up-projection encodes rows
    512.. of x itself. The workspace's MXFP6 x equals mx_quantize(x), and the
    result equals the three stages run one by one."""
    import torch

    M, d, ff = 2048, 512, 12288
    rng = np.random.default_rng(12 + gated)
    x_bits = synth.bf16_round(rng.standard_normal((M, d)).astype(np.float32))
    x = bf16_to_device(x_bits)
    rows_up = 2 * ff if gated else ff
    wu = lib.mx_quantize(bf16_to_device(synth.bf16_round(rng.standard_normal((rows_up, d)).astype(np.float32) * .02)))
    w2 = lib.mx_quantize(bf16_to_device(synth.bf16_round(rng.standard_normal((d, ff)).astype(np.float32) * .02)))
    bu = bf16_to_device(synth.bf16_round(rng.standard_normal(rows_up).astype(np.float32) * .01))
    b2 = bf16_to_device(synth.bf16_round(rng.standard_normal(d).astype(np.float32) * .01))
    ws = torch.empty(lib.mx_mlp_workspace_bytes(M, d, ff), dtype=torch.uint8, device="cuda")
    run = lib.mx_gated_mlp if gated else lib.mx_mlp
    y = run(x, wu, bu, w2, b2, workspace=ws)
    xq = lib.mx_quantize(x)
    got = lib.mx_quantize_gemm_xq(ws, M, d)   # xq sits at the start of the MLP workspace, scales 256-aligned
    assert torch.equal(got.codes, xq.codes) and torch.equal(got.scales, xq.scales)
    epi = lib.MX_EPI_BIAS_SWIGLU_MXFP6 if gated else lib.MX_EPI_BIAS_GELU_MXFP6
    hq = lib.mx_gemm(xq, wu, bu, epi)
    assert torch.equal(y, lib.mx_gemm(hq, w2, b2, lib.MX_EPI_BIAS_BF16)), "differs from its three stages"
    assert lib.mx_device_error() == 0


def test_threads_on_separate_streams(lib):
    """Three host threads, each on its own stream and workspace, run the fused GEMM
    five times at once; every result equals the one computed alone. The calls'
    grids cannot all be resident together, so producers wait on row groups that
    only the running CTAs' quantizer warps have claimed."""
    import torch

    n_threads, M, K, N = 3, 2048, 1024, 12288
    inputs = [_inputs(30 + i, M, K, N) for i in range(n_threads)]
    wq = lib.mx_quantize(bf16_to_device(inputs[0][2]))
    b = bf16_to_device(inputs[0][3])
    ref = [lib.mx_quantize_gemm(inp[1], wq, b, lib.MX_EPI_BIAS_BF16) for inp in inputs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(n_threads)]
    outs = [torch.empty_like(r) for r in ref]
    wss = [torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
           for _ in range(n_threads)]
    errors = []
    start = threading.Barrier(n_threads)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            start.wait()
            for _ in range(5):
                lib.mx_quantize_gemm(inputs[i][1], wq, b, lib.MX_EPI_BIAS_BF16, out=outs[i], workspace=wss[i],
                                     stream=streams[i])
            streams[i].synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    assert all(not t.is_alive() for t in threads)
    torch.cuda.synchronize()
    for i in range(n_threads):
        assert torch.equal(outs[i], ref[i]), f"thread {i} differs from the serial result"
    assert lib.mx_device_error() == 0


def test_nan_and_inf_blocks_in_kernel(lib):
    """NaN and Inf in rows the GEMM encodes itself: those blocks get the E8M0 NaN
    scale and zero codes exactly as the quantize kernel writes them, and the output
    equals K1 followed by mx_gemm bit for bit (NaN rows included)."""
    import torch

    M, K, N = 1400, 512, 12288
    x_bits, x, w_bits, bias = _inputs(13, M, K, N)
    nan, inf, ninf = 0x7FC0, 0x7F80, 0xFF80
    x_bits = x_bits.copy()
    x_bits[700, 5] = nan          # in-kernel rows (the lead is the first 512)
    x_bits[901, 300] = inf
    x_bits[1399, 511] = ninf
    x_bits[100, 64] = nan         # a lead row, for comparison
    x = bf16_to_device(x_bits)
    wq = lib.mx_quantize(bf16_to_device(w_bits))
    b = bf16_to_device(bias)
    ws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, K), dtype=torch.uint8, device="cuda")
    y = lib.mx_quantize_gemm(x, wq, b, lib.MX_EPI_BIAS_BF16, workspace=ws)
    rows = np.array([100, 700, 901, 1399, 1398])
    xq = _check_xq(lib, ws, x, x_bits, rows)
    ref = lib.mx_gemm(xq, wq, b, lib.MX_EPI_BIAS_BF16)
    assert torch.equal(y.view(torch.int16), ref.view(torch.int16))
    got = bf16_from_device(y)
    assert np.isnan(f32_from_bf16_bits(got[[100, 700, 901, 1399]])).all()
    assert not np.isnan(f32_from_bf16_bits(got[1398])).any()
    assert lib.mx_device_error() == 0

