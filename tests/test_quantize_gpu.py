"""K1 parity: the CUDA quantizer must reproduce the oracle's codes and scales bit
for bit (BF16 -> MXFP6, OCP MX rule), on every BF16 bit pattern, hand-derived
edge blocks, ragged and strided inputs and the workloads' activations/weights."""

import os

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import assert_codes_equal, bf16_to_device, mx_rows_to_host, mx_to_host, sample_rows

pytestmark = pytest.mark.gpu


def _check_full(lib, bits, what):
    x = bf16_to_device(bits)
    q = lib.mx_quantize(x)
    codes, scales = mx_to_host(q)
    rc, rs = O.quantize_bf16(bits)
    assert_codes_equal(codes, rc, scales, rs, what)
    # padding rows of the tiled scales are zero
    tiled = q.scales.cpu().numpy()
    rows, k = bits.shape
    assert np.count_nonzero(tiled) == np.count_nonzero(O.scales_plain_to_tiled(rs, rows, k))
    return q


def test_pr1_activations_and_weights(lib):
    w = synth.pr1()
    _check_full(lib, w["x"], "pr1 x")
    _check_full(lib, w["w"], "pr1 w")


def test_every_bf16_pattern(lib):
    """All 65,536 BF16 bit patterns (NaN and Inf included), in three arrangements:
    sequential, a seeded permutation, and each pattern beside anchors of many sizes."""
    allp = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    _check_full(lib, allp.reshape(512, 128), "sequential patterns")
    perm = np.random.default_rng(5).permutation(allp)
    _check_full(lib, perm.reshape(512, 128), "permuted patterns")
    finite = allp[np.isfinite(synth.bf16_to_f32(allp))]
    for e in (-130, -60, 0, 3, 60, 125):
        anchor = synth.bf16_round(np.array([7.75 * 2.0 ** e], dtype=np.float32))[0]
        n = finite.size // 31 * 31
        blocks = finite[:n].reshape(-1, 31)
        full = np.concatenate([np.full((blocks.shape[0], 1), anchor, np.uint16), blocks], axis=1)
        pad = (-full.shape[0]) % 4
        full = np.concatenate([full, np.zeros((pad, 32), np.uint16)])
        _check_full(lib, full.reshape(-1, 128), f"anchored 2^{e}")


def test_hand_derived_blocks(lib):
    """tests/golden/quant_blocks.txt, worked by hand, checked directly on the GPU."""
    vals, want_codes, want_scales = [], [], []
    with open(os.path.join(os.path.dirname(__file__), "golden", "quant_blocks.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            p = line.split()
            if p[0] == "block":
                want_scales.append(int(p[2]))
            else:
                vals.append(float.fromhex(p[0]))
                want_codes.append(int(p[1], 16))
    v = np.array(vals + [0.0] * 32, dtype=np.float32)     # 8 blocks -> two rows of 128
    bits = synth.bf16_round(v).reshape(2, 128)
    q = lib.mx_quantize(bf16_to_device(bits))
    codes, scales = mx_to_host(q)
    assert codes.reshape(-1)[:len(want_codes)].tolist() == want_codes
    assert scales.reshape(-1)[:len(want_scales)].tolist() == want_scales


def test_ragged_rows_and_row_stride(lib):
    import torch

    rng = np.random.default_rng(9)
    rows, k, ld = 300, 384, 520
    full = synth.bf16_round((rng.standard_normal((rows, ld)) * np.exp(rng.uniform(-8, 8, (rows, 1)))).astype(np.float32))
    xd = bf16_to_device(full)[:, :k]                      # strided view, ld_x = 520
    assert xd.stride(0) == ld
    q = lib.mx_quantize(xd)
    codes, scales = mx_to_host(q)
    rc, rs = O.quantize_bf16(full[:, :k])
    assert_codes_equal(codes, rc, scales, rs, "ragged/strided")
    tiled = q.scales.cpu().numpy()
    pad = O.scales_plain_to_tiled(np.full((rows, k // 32), 1, np.uint8), rows, k, pad_value=0) == 0
    assert np.all(tiled[pad] == 0)
    torch.cuda.synchronize()


def test_empty_and_single_row(lib):
    import torch

    q = lib.mx_quantize(torch.empty((0, 256), dtype=torch.bfloat16, device="cuda"))
    assert q.codes.numel() == 0 and q.scales.numel() == 0
    bits = synth.bf16_round(np.linspace(-9, 9, 128, dtype=np.float32)).reshape(1, 128)
    _check_full(lib, bits, "one row")


@pytest.mark.slow
@pytest.mark.parametrize("name", ["dit_up", "full_mlp", "outlier_mlp"])
def test_workload_activations_sampled(lib, name):
    w = synth.workload(name)
    x = w["x"]
    q = lib.mx_quantize(bf16_to_device(x))
    rows = sample_rows(x.shape[0], n_random=256)
    codes, scales = mx_rows_to_host(q, rows)
    rc, rs = O.quantize_bf16(x[rows])
    assert_codes_equal(codes, rc, scales, rs, name)


@pytest.mark.slow
def test_weights_full(lib):
    w = synth.full_mlp(M=128)
    for key in ("w1", "w2"):
        _check_full(lib, w[key], f"full_mlp {key}")
    assert lib.mx_device_error() == 0
