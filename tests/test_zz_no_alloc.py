"""mx_mlp_noalloc: the MLP block for callers that cannot allocate device memory.

Such callers (code hosted by a runtime whose allocator owns all device memory, or
running under a device-memory budget fixed at start-up) cannot hand mx_mlp a
workspace, so this entry point keeps its scratch in a static device array inside
the library. The test calls it through the C ABI twice in a row, on two different
token batches, and checks each result against the existing mx_mlp entry point
(caller-provided workspace) with the library's GEMM tolerance. It also checks
that a size beyond the static capacity is refused on the host.
"""

import ctypes

import numpy as np
import pytest

import synth
from mxutil import bf16_from_device, bf16_to_device, f32_from_bf16_bits, gemm_tolerance_report

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
    stream = torch.cuda.current_stream().cuda_stream
    # two calls in a row on different batches (the second smaller and ragged)
    for rows in (slice(0, 2048), slice(100, 1100)):
        x = bf16_to_device(w["x"][rows])
        m = x.shape[0]
        ref = lib.mx_mlp(x, w1, b1, w2, b2)
        y = torch.full((m, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = fn(x.data_ptr(), m, d, ff, w1.codes.data_ptr(), w1.scales.data_ptr(), b1.data_ptr(),
                w2.codes.data_ptr(), w2.scales.data_ptr(), b2.data_ptr(), y.data_ptr(), stream)
        assert st == 0, lib.mx_status_string(st)
        torch.cuda.synchronize()
        got = f32_from_bf16_bits(bf16_from_device(y)).astype(np.float64)
        want = f32_from_bf16_bits(bf16_from_device(ref)).astype(np.float64)
        rep = gemm_tolerance_report(got, want)
        assert rep["n_bad"] == 0, rep
    assert lib.mx_device_error() == 0


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    fn = _noalloc_fn(lib)
    # 5591 tokens of a d=3072, ff=12288 block need more than the 64 MiB scratch;
    # the host refuses before anything launches, so no buffers are needed
    st = fn(None, 5591, 3072, 12288, None, None, None, None, None, None, None, None)
    assert st == MX_ERR_WORKSPACE_TOO_SMALL
