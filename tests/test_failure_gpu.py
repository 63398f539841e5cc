"""Failure detection without a GPU fault: a kernel wait that can never complete
must give up after its bound, report it through the device error word, and leave
the context usable for the next launch."""

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import assert_gemm_close, bf16_from_device, bf16_to_device, f32_from_bf16_bits

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_and_context_survives(lib):
    assert lib.mx_device_error(clear=True) == 0
    lib.mx_selftest_wait_timeout()
    flags = lib.mx_device_error(clear=True)
    assert flags == 1 << 4, hex(flags)
    # the context still works: a GEMM right after matches the oracle
    w = synth.pr1()
    xq = lib.mx_quantize(bf16_to_device(w["x"]))
    wq = lib.mx_quantize(bf16_to_device(w["w"]))
    y = lib.mx_gemm(xq, wq, bf16_to_device(w["b"]), lib.MX_EPI_BIAS_BF16)
    rxq, rxs = O.quantize_bf16(w["x"])
    rwq, rws = O.quantize_bf16(w["w"])
    got = f32_from_bf16_bits(bf16_from_device(y)).astype(np.float64)
    assert_gemm_close(got, O.gemm(rxq, rxs, rwq, rws, w["b"]), "after self test")
    assert lib.mx_device_error() == 0
