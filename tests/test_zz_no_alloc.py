"""mx_mlp_noalloc: the MLP block for callers that cannot allocate device memory.

Such callers (code hosted by a runtime whose allocator owns all device memory, or
running under a device-memory budget fixed at start-up) cannot hand mx_mlp a
workspace, so this entry point keeps its scratch in a static device array inside
the library. The test calls it through the C ABI twice in a row, on two different
token batches (the second smaller and ragged, so it reuses the array a larger call
left behind), and requires each result to be bit-identical to the existing mx_mlp
entry point with a caller-provided workspace: both run the same kernels with the
same launch plan. A sampled row set of each call is also checked stage-wise
against the oracle. The host-side checks (shape rules, the capacity limit) are in
tests/test_abi.py; this file also checks on the GPU that a size beyond the
capacity is refused.
"""

import ctypes

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import assert_gemm_close, bf16_from_device, bf16_to_device, f32_from_bf16_bits, sample_rows

pytestmark = pytest.mark.gpu

MX_ERR_WORKSPACE_TOO_SMALL = 4


def _noalloc_fn(lib):
    fn = lib.load().mx_mlp_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    return fn


def test_noalloc_matches_mx_mlp_on_two_calls(lib):
    import torch

    fn = _noalloc_fn(lib)
    d, ff = 1024, 4096
    w = synth.full_mlp(M=2048, d=d, ff=ff)
    w1 = lib.mx_quantize(bf16_to_device(w["w1"]))
    w2 = lib.mx_quantize(bf16_to_device(w["w2"]))
    b1 = bf16_to_device(w["b1"])
    b2 = bf16_to_device(w["b2"])
    r_w1q, r_w1s = O.quantize_bf16(w["w1"])
    r_w2q, r_w2s = O.quantize_bf16(w["w2"])
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row on different batches (the second smaller and ragged)
    for rows in (slice(0, 2048), slice(100, 1100)):
        xb = w["x"][rows]
        x = bf16_to_device(xb)
        m = x.shape[0]
        ref = lib.mx_mlp(x, w1, b1, w2, b2)
        y = torch.full((m, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = fn(x.data_ptr(), m, d, ff, w1.codes.data_ptr(), w1.scales.data_ptr(), b1.data_ptr(),
                w2.codes.data_ptr(), w2.scales.data_ptr(), b2.data_ptr(), y.data_ptr(), stream)
        assert st == 0, lib.mx_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), "mx_mlp_noalloc differs from mx_mlp"
        # stage-wise against the oracle on sampled rows: the GPU's intermediate is
        # recomputed by the same kernels (bit-identical to the one the call used),
        # checked bit-exact given its fp32 pre-quantization values, then the
        # down-projection within the GEMM tolerance given that intermediate
        pick = sample_rows(m, n_random=48)
        idx = torch.as_tensor(pick, device="cuda")
        dbg = torch.empty((m, ff), dtype=torch.float32, device="cuda")
        hq = lib.mx_gemm(lib.mx_quantize(x), w1, b1, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=dbg)
        g = dbg[idx].cpu().numpy()
        rxq, rxs = O.quantize_bf16(xb[pick])
        assert_gemm_close(g, O.up_projection(rxq, rxs, r_w1q, r_w1s, w["b1"]), "gelu(x W1^T + b1)")
        rhq, rhs = O.quantize_f32(g)
        codes = O.unpack_codes(hq.codes.index_select(0, idx).cpu().numpy(), ff)
        scales = O.scales_tiled_to_plain(hq.scales.cpu().numpy(), m, ff)[pick]
        assert np.array_equal(codes, rhq) and np.array_equal(scales, rhs), "intermediate differs from the oracle"
        got = f32_from_bf16_bits(bf16_from_device(y[idx])).astype(np.float64)
        assert_gemm_close(got, O.down_projection(rhq, rhs, r_w2q, r_w2s, w["b2"]), "y")
    assert lib.mx_device_error() == 0


def test_noalloc_binding_matches_mx_mlp(lib):
    """The Python binding's mx_mlp_noalloc (argument marshalling only) gives mx_mlp's
    result bit for bit, and a size beyond the scratch raises."""
    import torch

    w = synth.full_mlp(M=300, d=256, ff=512)
    x = bf16_to_device(w["x"])
    w1, w2 = lib.mx_quantize(bf16_to_device(w["w1"])), lib.mx_quantize(bf16_to_device(w["w2"]))
    b1, b2 = bf16_to_device(w["b1"]), bf16_to_device(w["b2"])
    assert torch.equal(lib.mx_mlp_noalloc(x, w1, b1, w2, b2), lib.mx_mlp(x, w1, b1, w2, b2))
    assert lib.mx_device_error() == 0


def test_noalloc_with_the_quantizer_inside_the_gemm(lib):
    """At ff = 12288 the up-projection encodes x in-kernel (rows 512 onwards), with
    its row-block counters in the static scratch too: mx_mlp's result bit for bit,
    on two calls in a row (the second smaller and ragged)."""
    import torch

    d, ff = 512, 12288
    w = synth.full_mlp(M=2048, d=d, ff=ff)
    w1, w2 = lib.mx_quantize(bf16_to_device(w["w1"])), lib.mx_quantize(bf16_to_device(w["w2"]))
    b1, b2 = bf16_to_device(w["b1"]), bf16_to_device(w["b2"])
    for rows in (slice(0, 2048), slice(37, 1837)):
        x = bf16_to_device(w["x"][rows])
        assert torch.equal(lib.mx_mlp_noalloc(x, w1, b1, w2, b2), lib.mx_mlp(x, w1, b1, w2, b2))
    assert lib.mx_device_error() == 0


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    fn = _noalloc_fn(lib)
    # 5591 tokens of a d=3072, ff=12288 block need more than the 64 MiB scratch;
    # the host refuses before anything launches, so no buffers are needed
    st = fn(None, 5591, 3072, 12288, None, None, None, None, None, None, None, None)
    assert st == MX_ERR_WORKSPACE_TOO_SMALL
