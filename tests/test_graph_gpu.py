"""The MLP entry points under CUDA graph capture.

A step of the hot path is a fixed sequence of launches on one stream, so it can
be captured once and replayed: every replay must equal an eager call on the
same inputs bit for bit (the kernels are deterministic: no atomics, fixed
reduction orders). Inputs are refreshed between replays by copying into the
captured buffers, as a serving loop would. The first eager call on a device
fills the library's per-device caches (kernel attributes, occupancy); capture
comes after it.
"""

import pytest

import synth
from mxutil import bf16_to_device, graph_capture as _capture, graph_replays_match as _replays_match

pytestmark = pytest.mark.gpu


def test_mlp_graph_replay(lib):
    import torch

    w = synth.full_mlp(M=384, d=512, ff=1024)
    w1 = lib.mx_quantize(bf16_to_device(w["w1"]))
    w2 = lib.mx_quantize(bf16_to_device(w["w2"]))
    b1, b2 = bf16_to_device(w["b1"]), bf16_to_device(w["b2"])
    ws = torch.empty(lib.mx_mlp_workspace_bytes(384, 512, 1024), dtype=torch.uint8, device="cuda")
    x = bf16_to_device(w["x"])
    y = torch.empty_like(x)

    def run(xi, yi):
        lib.mx_mlp(xi, w1, b1, w2, b2, y=yi, workspace=ws)

    run(x, y)   # fills the per-device caches outside capture
    _replays_match(lib, run, lambda s: bf16_to_device(synth.full_mlp(seed=s, M=384, d=512, ff=1024)["x"]), x, y)


def test_dit_block_graph_replay_in_place(lib):
    """The SwiGLU DiT sub-block updating its input in place, captured and replayed."""
    import torch

    w = synth.dit_block(M=300, d=256, ff=384, activation="swiglu")
    wup = lib.mx_quantize(bf16_to_device(w["w_up"]))
    w2 = lib.mx_quantize(bf16_to_device(w["w2"]))
    vec = {k: bf16_to_device(w[k]) for k in ("shift", "scale", "gate", "b_up", "b2")}
    ws = torch.empty(lib.mx_mlp_workspace_bytes(300, 256, 384), dtype=torch.uint8, device="cuda")

    def run(xi, yi):
        lib.mx_dit_mlp_block(xi, vec["shift"], vec["scale"], vec["gate"], wup, vec["b_up"], w2, vec["b2"],
                             eps=w["eps"], activation=lib.MX_ACT_SWIGLU, y=yi, workspace=ws)

    x = bf16_to_device(w["x"])
    run(x.clone(), torch.empty_like(x))
    # in place: the captured graph reads x and overwrites it with x + gate * MLP(x)
    g = _capture(lambda: run(x, x))
    for i in range(3):
        x_new = bf16_to_device(synth.dit_block(seed=50 + i, M=300, d=256, ff=384, activation="swiglu")["x"])
        x.copy_(x_new)
        g.replay()
        torch.cuda.synchronize()
        y_eager = torch.empty_like(x)
        run(x_new, y_eager)
        torch.cuda.synchronize()
        assert torch.equal(x, y_eager), f"in-place replay {i} differs from the eager call"
        assert not torch.equal(x, x_new)
    assert lib.mx_device_error() == 0


def test_quantize_then_gemm_graph_many_replays(lib):
    """K1 + a BF16-epilogue GEMM captured once, replayed 20 times on fresh inputs."""
    import torch

    w = synth.pr1(M=256, K=512, N=512)
    wq = lib.mx_quantize(bf16_to_device(w["w"]))
    b = bf16_to_device(w["b"])
    x = bf16_to_device(w["x"])
    xq = lib.mx_quantize(x)
    y = torch.empty((256, 512), dtype=torch.bfloat16, device="cuda")

    def run(xi, yi):
        q = lib.mx_quantize(xi, out=xq) if xi is x else lib.mx_quantize(xi)
        lib.mx_gemm(q, wq, b, lib.MX_EPI_BIAS_BF16, out=yi)

    _replays_match(lib, run, lambda s: bf16_to_device(synth.pr1(seed=s, M=256, K=512, N=512)["x"]), x, y, n=20)


def test_fused_quantizer_graph_replay(lib):
    """The GEMM that quantizes its own activations under capture: mx_mlp at a width
    whose up-projection encodes rows 512.. in-kernel (ff = 12288), and
    mx_quantize_gemm on its own, captured and replayed on fresh inputs; the
    captured quantize kernel zeroes the row-block counters (and the quantizer warps'
    work counter) on every replay, so each replay equals the eager call."""
    import torch

    M, d, ff = 1536, 256, 12288
    w = synth.full_mlp(M=M, d=d, ff=ff)
    w1 = lib.mx_quantize(bf16_to_device(w["w1"]))
    w2 = lib.mx_quantize(bf16_to_device(w["w2"]))
    b1, b2 = bf16_to_device(w["b1"]), bf16_to_device(w["b2"])
    ws = torch.empty(lib.mx_mlp_workspace_bytes(M, d, ff), dtype=torch.uint8, device="cuda")
    x = bf16_to_device(w["x"])
    y = torch.empty_like(x)

    def mlp(xi, yi):
        lib.mx_mlp(xi, w1, b1, w2, b2, y=yi, workspace=ws)

    mlp(x, y)
    _replays_match(lib, mlp, lambda s: bf16_to_device(synth.full_mlp(seed=s, M=M, d=d, ff=ff)["x"]), x, y)

    qws = torch.empty(lib.mx_quantize_gemm_workspace_bytes(M, d), dtype=torch.uint8, device="cuda")
    h = torch.empty((M, ff), dtype=torch.bfloat16, device="cuda")

    def up(xi, hi):
        lib.mx_quantize_gemm(xi, w1, b1, lib.MX_EPI_BIAS_BF16, out=hi, workspace=qws)

    up(x, h)
    _replays_match(lib, up, lambda s: bf16_to_device(synth.full_mlp(seed=60 + s, M=M, d=d, ff=ff)["x"]), x, h)
