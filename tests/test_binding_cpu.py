"""The Python binding refuses host tensors before it calls the library: the
kernels take raw device pointers, so a CPU tensor must fail loudly on the host
rather than reach a launch. Runs without a GPU (the library loads; no compute
call is made)."""

import pytest

torch = pytest.importorskip("torch")

import microscaled_precision_gemm_gb300 as mx  # noqa: E402


def _mx(rows, k):
    return mx.MxTensor(torch.zeros((rows, k * 3 // 4), dtype=torch.uint8),
                       torch.zeros(max(1, ((rows + 127) // 128) * 128 * (k // 32)), dtype=torch.uint8), rows, k)


def _bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


@pytest.fixture(scope="module")
def lib():
    try:
        mx.load()
    except Exception as e:  # noqa: BLE001
        pytest.skip(f"library not built: {e}")
    return mx


CALLS = {
    "mx_quantize": lambda: mx.mx_quantize(_bf16(256, 256)),
    "mx_quantize_rmsnorm_modulate": lambda: mx.mx_quantize_rmsnorm_modulate(_bf16(256, 256)),
    "mx_gemm": lambda: mx.mx_gemm(_mx(256, 256), _mx(256, 256)),
    "mx_gemm gelu": lambda: mx.mx_gemm(_mx(256, 256), _mx(256, 256), None, mx.MX_EPI_BIAS_GELU_MXFP6),
    "mx_gemm_gate_residual": lambda: mx.mx_gemm_gate_residual(_mx(256, 256), _mx(256, 256), None, None,
                                                              _bf16(256, 256)),
    "mx_mlp": lambda: mx.mx_mlp(_bf16(256, 256), _mx(512, 256), None, _mx(256, 512), None),
    "mx_gated_mlp": lambda: mx.mx_gated_mlp(_bf16(256, 256), _mx(1024, 256), None, _mx(256, 512), None),
    "mx_dit_mlp_block": lambda: mx.mx_dit_mlp_block(_bf16(256, 256), None, None, None, _mx(512, 256), None,
                                                    _mx(256, 512), None),
    "mx_quantize_gemm": lambda: mx.mx_quantize_gemm(_bf16(256, 256), _mx(512, 256)),
    "mx_quantize_gemm gate residual": lambda: mx.mx_quantize_gemm(_bf16(256, 256), _mx(512, 256), None,
                                                                  mx.MX_EPI_GATE_RESIDUAL_BF16,
                                                                  residual=_bf16(256, 512)),
    "mx_mlp_noalloc": lambda: mx.mx_mlp_noalloc(_bf16(256, 256), _mx(512, 256), None, _mx(256, 512), None),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused_before_any_launch(lib, name):
    with pytest.raises(ValueError, match="CUDA"):
        CALLS[name]()
