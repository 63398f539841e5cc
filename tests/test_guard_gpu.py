"""Out-of-bounds and unwritten-output checks without a sanitizer.

Every output buffer sits inside a larger allocation with 4 KB canary bands on
both sides. Each kernel runs twice, into buffers pre-filled with two different
poison patterns (0x00 and 0xA5): the two results must be byte-identical (every
output byte is written, padding-row scales included, none is left over from the
poison) and every canary byte must still hold its poison (nothing is written
outside the output). Ragged row counts put the last tiles partly past the end.
"""

import numpy as np
import pytest

import synth
from mxutil import bf16_to_device, mx_upload

pytestmark = pytest.mark.gpu

GUARD = 4096


class Guarded:
    """`nbytes` usable bytes at a 4096-byte offset inside a poisoned allocation."""

    def __init__(self, nbytes: int, poison: int):
        import torch

        self.n = int(nbytes)
        self.poison = poison
        self.raw = torch.full((self.n + 2 * GUARD,), poison, dtype=torch.uint8, device="cuda")
        self.body = self.raw[GUARD:GUARD + self.n]

    def canaries_intact(self) -> bool:
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        return bool((head == self.poison).all().item() and (tail == self.poison).all().item())


def _mx_out(lib, rows, k, poison):
    codes = Guarded(lib.mx_codes_bytes(rows, k), poison)
    scales = Guarded(lib.mx_scales_bytes(rows, k), poison)
    return codes, scales, lib.MxTensor(codes.body.view(rows, -1), scales.body, rows, k)


def _check_twice(run):
    """run(poison) -> list of Guarded outputs; compares the two poisons' results."""
    import torch

    outs = [run(p) for p in (0x00, 0xA5)]
    torch.cuda.synchronize()
    for g in outs[0] + outs[1]:
        assert g.canaries_intact(), "a kernel wrote outside its output buffer"
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.body, b.body), "an output byte was left unwritten (poison shows through)"


def _random_mx(rng, rows, k):
    return (rng.integers(0, 64, size=(rows, k)).astype(np.uint8),
            rng.integers(118, 124, size=(rows, k // 32)).astype(np.uint8))


def test_quantize_guards(lib):
    x = bf16_to_device(synth.bf16_round(np.random.default_rng(1).standard_normal((300, 640)).astype(np.float32)))

    def run(p):
        c, s, t = _mx_out(lib, 300, 640, p)
        lib.mx_quantize(x, out=t)
        return [c, s]

    _check_twice(run)


def test_norm_quantize_guards(lib):
    rng = np.random.default_rng(2)
    x = bf16_to_device(synth.bf16_round(rng.standard_normal((130, 1024)).astype(np.float32)))
    vec = bf16_to_device(synth.bf16_round(rng.standard_normal(1024).astype(np.float32) * 0.5))

    def run(p):
        c, s, t = _mx_out(lib, 130, 1024, p)
        lib.mx_quantize_rmsnorm_modulate(x, vec, vec, 1e-6, out=t)
        return [c, s]

    _check_twice(run)


@pytest.mark.parametrize("epi", ["bf16", "gelu", "swiglu", "gate_res"])
def test_gemm_epilogue_guards(lib, epi):
    import torch

    M, N, K = 300, 768, 256
    rng = np.random.default_rng(3)
    a = mx_upload(*_random_mx(rng, M, K))
    b = mx_upload(*_random_mx(rng, N, K))
    bias = bf16_to_device(synth.bf16_round(rng.standard_normal(N).astype(np.float32)))
    gate = bf16_to_device(synth.bf16_round(rng.standard_normal(N).astype(np.float32)))
    res = bf16_to_device(synth.bf16_round(rng.standard_normal((M, N)).astype(np.float32)))

    def run(p):
        if epi in ("bf16", "gate_res"):
            y = Guarded(M * N * 2, p)
            out = y.body.view(torch.bfloat16).view(M, N)
            if epi == "bf16":
                lib.mx_gemm(a, b, bias, lib.MX_EPI_BIAS_BF16, out=out)
            else:
                lib.mx_gemm_gate_residual(a, b, bias, gate, res, out=out)
            return [y]
        w = N // 2 if epi == "swiglu" else N
        c, s, t = _mx_out(lib, M, w, p)
        e = lib.MX_EPI_BIAS_SWIGLU_MXFP6 if epi == "swiglu" else lib.MX_EPI_BIAS_GELU_MXFP6
        lib.mx_gemm(a, b, bias, e, out=t)
        return [c, s]

    _check_twice(run)


def test_mlp_workspace_and_output_guards(lib):
    """mx_mlp writes only its workspace (fully overwritten each call) and y."""
    import torch

    w = synth.full_mlp(M=257, d=256, ff=512)
    w1 = lib.mx_quantize(bf16_to_device(w["w1"]))
    w2 = lib.mx_quantize(bf16_to_device(w["w2"]))
    x = bf16_to_device(w["x"])
    b1, b2 = bf16_to_device(w["b1"]), bf16_to_device(w["b2"])
    need = lib.mx_mlp_workspace_bytes(257, 256, 512)

    def run(p):
        ws = Guarded(need, p)
        y = Guarded(257 * 256 * 2, p)
        lib.mx_mlp(x, w1, b1, w2, b2, y=y.body.view(torch.bfloat16).view(257, 256), workspace=ws.body)
        return [y, ws]

    outs = [run(p) for p in (0x00, 0xA5)]
    torch.cuda.synchronize()
    for g in outs[0] + outs[1]:
        assert g.canaries_intact(), "mx_mlp wrote outside y or its workspace"
    assert torch.equal(outs[0][0].body, outs[1][0].body), "y differs with the workspace's initial contents"
    assert lib.mx_device_error() == 0
