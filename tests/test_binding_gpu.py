"""The Python binding refuses buffers the library would read or write out of
bounds (short, mis-typed, strided or misshapen outputs, vectors and MXFP6
operands) with a ValueError before any launch, and valid calls are unaffected."""

import pytest

pytestmark = pytest.mark.gpu


def _mx(lib, rows, k, short_codes=0, short_scales=0):
    import torch

    codes = torch.zeros(lib.mx_codes_bytes(rows, k) - short_codes, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(lib.mx_scales_bytes(rows, k) - short_scales, dtype=torch.uint8, device="cuda")
    return lib.MxTensor(codes, scales, rows, k)


def _bf16(*shape):
    import torch

    return torch.zeros(shape, dtype=torch.bfloat16, device="cuda")


def test_gemm_refuses_bad_buffers(lib):
    import torch

    M, N, K = 300, 512, 256
    a, b = _mx(lib, M, K), _mx(lib, N, K)
    bad = {
        "short out": dict(out=_bf16(M * N - 1)),
        "fp32 out": dict(out=torch.zeros((M, N), device="cuda")),
        "strided out": dict(out=_bf16(N, M).t()),
        "short bias": dict(bias=_bf16(N - 1)),
        "fp32 bias": dict(bias=torch.zeros(N, device="cuda")),
        "int64 workspace": dict(workspace=torch.zeros(4096, dtype=torch.int64, device="cuda")),
    }
    for what, kw in bad.items():
        with pytest.raises(ValueError):
            lib.mx_gemm(a, b, kw.get("bias"), lib.MX_EPI_BIAS_BF16, out=kw.get("out"),
                        workspace=kw.get("workspace"))
    # the requantizing epilogues check their MXFP6 output and debug buffer too
    with pytest.raises(ValueError):
        lib.mx_gemm(a, b, None, lib.MX_EPI_BIAS_GELU_MXFP6, out=_mx(lib, M, N, short_scales=1))
    with pytest.raises(ValueError):
        lib.mx_gemm(a, b, None, lib.MX_EPI_BIAS_GELU_MXFP6, out=_mx(lib, M - 1, N))
    with pytest.raises(ValueError):
        lib.mx_gemm(a, b, None, lib.MX_EPI_BIAS_GELU_MXFP6,
                    debug_prequant=torch.zeros((M, N - 1), device="cuda"))
    with pytest.raises(ValueError):
        lib.mx_gemm(a, b, None, lib.MX_EPI_BIAS_SWIGLU_MXFP6, out=_mx(lib, M, N))   # SwiGLU writes N/2
    for short in (dict(short_codes=1), dict(short_scales=1)):
        with pytest.raises(ValueError):
            lib.mx_gemm(_mx(lib, M, K, **short), b)
        with pytest.raises(ValueError):
            lib.mx_gemm(a, _mx(lib, N, K, **short))
    assert lib.mx_device_error() == 0


def test_quantizers_refuse_bad_buffers(lib):
    import torch

    x = _bf16(300, 256)
    with pytest.raises(ValueError):
        lib.mx_quantize(x, out=_mx(lib, 300, 256, short_codes=1))
    with pytest.raises(ValueError):
        lib.mx_quantize(x, out=_mx(lib, 299, 256))
    with pytest.raises(ValueError):
        lib.mx_quantize_rmsnorm_modulate(x, shift=_bf16(255))
    with pytest.raises(ValueError):
        lib.mx_quantize_rmsnorm_modulate(x, debug_y=torch.zeros((299, 256), device="cuda"))
    with pytest.raises(ValueError):
        lib.mx_quantize_rmsnorm_modulate(x, out=_mx(lib, 300, 256, short_scales=1))
    assert lib.mx_device_error() == 0


def test_fused_entry_points_refuse_bad_buffers(lib):
    import torch

    M, d, ff = 300, 256, 512
    x = _bf16(M, d)
    w1, w2, wgu = _mx(lib, ff, d), _mx(lib, d, ff), _mx(lib, 2 * ff, d)
    for kw in (dict(y=_bf16(M * d - 1)), dict(workspace=torch.zeros(1 << 20, dtype=torch.float32, device="cuda"))):
        with pytest.raises(ValueError):
            lib.mx_mlp(x, w1, None, w2, None, **kw)
        with pytest.raises(ValueError):
            lib.mx_gated_mlp(x, wgu, None, w2, None, **kw)
        with pytest.raises(ValueError):
            lib.mx_dit_mlp_block(x, None, None, None, w1, None, w2, None, **kw)
    with pytest.raises(ValueError):
        lib.mx_mlp(x, w1, _bf16(ff - 1), w2, None)
    with pytest.raises(ValueError):
        lib.mx_mlp(x, _mx(lib, ff, d, short_scales=1), None, w2, None)
    with pytest.raises(ValueError):
        lib.mx_mlp(_bf16(d, M).t(), w1, None, w2, None)          # strided activations
    with pytest.raises(ValueError):
        lib.mx_gated_mlp(x, wgu, _bf16(ff), w2, None)             # bias of the stacked weight is 2 ff long
    with pytest.raises(ValueError):
        lib.mx_dit_mlp_block(x, _bf16(d - 1), None, None, w1, None, w2, None)
    a, b = _mx(lib, M, ff), _mx(lib, d, ff)
    with pytest.raises(ValueError):
        lib.mx_gemm_gate_residual(a, b, None, None, _bf16(M + 1, d))
    with pytest.raises(ValueError):
        lib.mx_gemm_gate_residual(a, b, None, _bf16(d + 1), _bf16(M, d))
    with pytest.raises(ValueError):
        lib.mx_gemm_gate_residual(a, b, None, None, _bf16(M, d), out=_bf16(M, d - 1))
    assert lib.mx_device_error() == 0


def test_quantize_gemm_refuses_bad_buffers(lib):
    """mx_quantize_gemm: the activations, the weight, the bias, the gate and residual,
    the output and the workspace are checked as the other entry points check them."""
    import torch

    M, K, N = 300, 256, 512
    x, b = _bf16(M, K), _mx(lib, N, K)
    need = lib.mx_quantize_gemm_workspace_bytes(M, K)
    bad = [
        dict(x=_bf16(K, M).t()),                                     # strided activations
        dict(x=torch.zeros((M, K), device="cuda")),                  # fp32 activations
        dict(b=_mx(lib, N, K, short_scales=1)),
        dict(b=_mx(lib, N, K + 128)),                                # inner dimensions differ
        dict(bias=_bf16(N - 1)),
        dict(out=_bf16(M * N - 1)),
        dict(workspace=torch.zeros(need, dtype=torch.int32, device="cuda")),
        dict(epi=lib.MX_EPI_GATE_RESIDUAL_BF16),                    # no residual
        dict(epi=lib.MX_EPI_GATE_RESIDUAL_BF16, residual=_bf16(M + 1, N)),
        dict(epi=lib.MX_EPI_GATE_RESIDUAL_BF16, residual=_bf16(M, N), gate=_bf16(N + 1)),
        dict(epi=lib.MX_EPI_BIAS_GELU_MXFP6, out=_mx(lib, M, N, short_scales=1)),
        dict(epi=lib.MX_EPI_BIAS_SWIGLU_MXFP6, out=_mx(lib, M, N)),  # SwiGLU writes N/2
    ]
    for kw in bad:
        with pytest.raises(ValueError):
            lib.mx_quantize_gemm(kw.get("x", x), kw.get("b", b), kw.get("bias"), kw.get("epi", lib.MX_EPI_BIAS_BF16),
                                 gate=kw.get("gate"), residual=kw.get("residual"), out=kw.get("out"),
                                 workspace=kw.get("workspace"))
    # a workspace below mx_quantize_gemm_workspace_bytes is refused by the library
    with pytest.raises(lib.MxError):
        lib.mx_quantize_gemm(x, b, None, lib.MX_EPI_BIAS_BF16,
                             workspace=torch.zeros(need - 256, dtype=torch.uint8, device="cuda"))
    assert lib.mx_device_error() == 0
