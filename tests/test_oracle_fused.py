"""Pins for the oracle's fused neighbours of the MLP (SwiGLU, RMSNorm + modulation,
gate + residual, the whole DiT MLP sub-block).

Sources of truth: printed values of the logistic function, the odd-part identity
of SiLU, scipy's expit, exact rational arithmetic in pure Python on tiny cases
(from the hand-typed OCP E2M3 table), and closed forms of the RMS normalisation.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_table():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m3_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            code, val = line.split()
            vals[int(code, 16)] = Fraction(val)
    assert sorted(vals) == list(range(32))
    return vals


def _exact_gemm(a, sa, b, sb, bias_bits=None):
    """C = deq(A) deq(B)^T (+ bias) as exact Fractions, from the golden table."""
    golden = _golden_table()

    def val(code, scale):
        v = golden[int(code) & 0x1F] * Fraction(2) ** (int(scale) - 127)
        return -v if int(code) & 0x20 else v

    M, K = a.shape
    N = b.shape[0]
    out = [[Fraction(0)] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += val(a[m, k], sa[m, k // 32]) * val(b[n, k], sb[n, k // 32])
            if bias_bits is not None:
                acc += Fraction(float(synth.bf16_to_f32(bias_bits[n])))
            out[m][n] = acc
    return out


def _bf16(x):
    return synth.bf16_round(np.asarray(x, dtype=np.float32))


# ---------------------------------------------------------------- SiLU

def test_silu_printed_values_and_limits():
    # sigmoid(1) = e / (1 + e) = 0.7310585786300049 (printed value of the logistic function)
    assert O.silu(0.0) == 0.0
    assert abs(O.silu(1.0) - 0.7310585786300049) < 1e-16
    assert abs(O.silu(-1.0) + 0.2689414213699951) < 1e-16
    assert abs(O.silu(2.0) - 2 * 0.8807970779778823) < 1e-15
    assert O.silu(60.0) == 60.0
    assert abs(O.silu(-60.0)) < 1e-24
    assert O.silu(-800.0) == 0.0 and O.silu(800.0) == 800.0


def test_silu_odd_part_identity_and_expit():
    # v sigma(v) - (-v) sigma(-v) = v (sigma(v) + sigma(-v)) = v: fails on a sign slip
    v = np.linspace(-30, 30, 6001)
    np.testing.assert_allclose(O.silu(v) - O.silu(-v), v, rtol=0, atol=1e-14 * 30)
    special = pytest.importorskip("scipy.special")
    np.testing.assert_allclose(O.silu(v), v * special.expit(v), rtol=2e-15, atol=1e-300)
    # minimum of SiLU: about -0.2784645 at v = -1.2784645 (root of 1 + v (1 - sigma(v)) = 0)
    grid = np.linspace(-3, 0, 300001)
    s = O.silu(grid)
    assert abs(s.min() + 0.27846454276) < 1e-9
    assert abs(grid[np.argmin(s)] + 1.27846454) < 1e-4


# ---------------------------------------------------------------- SwiGLU projection

@pytest.mark.parametrize("M,F,K", [(2, 3, 32), (3, 4, 64)])
def test_swiglu_projection_equals_exact_gate_times_up(M, F, K):
    rng = np.random.default_rng(10 * M + F + K)
    a = rng.integers(0, 64, size=(M, K)).astype(np.uint8)
    b = rng.integers(0, 64, size=(2 * F, K)).astype(np.uint8)
    sa = rng.integers(124, 131, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(124, 131, size=(2 * F, K // 32)).astype(np.uint8)
    bias = _bf16(rng.standard_normal(2 * F))
    h = O.swiglu_up_projection(a, sa, b, sb, bias)
    assert h.shape == (M, F)
    c = _exact_gemm(a, sa, b, sb, bias)
    for m in range(M):
        for n in range(F):
            g = float(c[m][n])            # gate rows come first in the stack
            u = float(c[m][F + n])
            ref = g / (1.0 + math.exp(-g)) * u
            assert abs(h[m, n] - ref) <= 1e-14 * abs(ref) + 1e-300, (m, n)


def test_swiglu_gate_and_up_are_not_swapped():
    # up rows all zero and up bias 1 -> h = silu(g); gate rows zero, bias 1 -> h = silu(1) u
    K, F = 32, 2
    a = np.zeros((1, K), np.uint8)
    a[0, 0] = 0x10                           # 2.0
    b = np.zeros((2 * F, K), np.uint8)
    b[0, 0] = 0x08                           # gate row 0: 1.0 -> g0 = 2
    b[1, 0] = 0x28                           # gate row 1: -1.0 -> g1 = -2
    sa = np.full((1, 1), 127, np.uint8)
    sb = np.full((2 * F, 1), 127, np.uint8)
    one = _bf16([1.0])[0]
    zero = _bf16([0.0])[0]
    bias = np.array([zero, zero, one, one], dtype=np.uint16)
    h = O.swiglu_up_projection(a, sa, b, sb, bias)
    np.testing.assert_allclose(h[0], [2 * 0.8807970779778823, -2 * 0.11920292202211755], rtol=1e-15)


def test_gated_mlp_chain_on_tiny_workload():
    w = synth.gated_mlp(M=8, d=128, ff=256)
    wq, ws = O.quantize_bf16(w["wgu"])
    w2q, w2s = O.quantize_bf16(w["w2"])
    y, mid = O.gated_mlp(w["x"], wq, ws, w["bgu"], w2q, w2s, w["b2"])
    assert y.shape == (8, 128) and mid["h"].shape == (8, 256)
    hq, hs = O.quantize_f32(mid["h"].astype(np.float32))
    assert np.array_equal(hq, mid["hq"]) and np.array_equal(hs, mid["hs"])
    # stacking is concatenation: quantizing the halves alone gives the same codes
    gq, gs = O.quantize_bf16(w["wgu"][:256])
    assert np.array_equal(gq, wq[:256]) and np.array_equal(gs, ws[:256])


# ---------------------------------------------------------------- RMSNorm + modulation

def test_rms_norm_closed_forms():
    K = 64
    zero = np.zeros(K, np.uint16)
    # +-1 alternating row: mean square 1, eps 0 -> y = x
    x = _bf16(np.tile([1.0, -1.0], K // 2)[None, :])
    np.testing.assert_array_equal(O.rms_norm_modulate(x, zero, zero, 0.0), np.tile([1.0, -1.0], K // 2)[None, :])
    # constant row c: y = sign(c) (1 + scale) + shift, whatever c's magnitude
    for c in (0.0078125, 3.0, -40.0):
        xc = _bf16(np.full((1, K), c))
        scale = _bf16(np.linspace(-0.5, 0.5, K))
        shift = _bf16(np.linspace(1.0, -1.0, K))
        y = O.rms_norm_modulate(xc, shift, scale, 0.0)
        ref = np.sign(c) * (1 + synth.bf16_to_f32(scale).astype(np.float64)) + synth.bf16_to_f32(shift)
        np.testing.assert_allclose(y[0], ref, rtol=1e-15, atol=1e-15)
    # [3, 4, 0, ...]: mean square 25 / K
    x = np.zeros((1, K), np.float32)
    x[0, :2] = [3.0, 4.0]
    y = O.rms_norm_modulate(_bf16(x), zero, zero, 0.0)
    np.testing.assert_allclose(y[0, :2], np.array([3.0, 4.0]) / math.sqrt(25.0 / K), rtol=1e-15)
    # all-zero row: only eps keeps the root finite -> y = shift
    shift = _bf16(np.arange(K) / 8.0)
    y = O.rms_norm_modulate(np.zeros((1, K), np.uint16), shift, zero, 1e-6)
    np.testing.assert_array_equal(y[0], synth.bf16_to_f32(shift).astype(np.float64))


def test_rms_norm_invariants():
    rng = np.random.default_rng(5)
    K = 96
    x = _bf16(rng.standard_normal((4, K)) * np.array([[0.01], [1.0], [30.0], [1000.0]]))
    zero = np.zeros(K, np.uint16)
    y = O.rms_norm_modulate(x, zero, zero, 0.0)
    # unit RMS per row
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)
    # invariant to a power-of-two rescaling of the row (exact in BF16)
    y4 = O.rms_norm_modulate(_bf16(synth.bf16_to_f32(x) * 4.0), zero, zero, 0.0)
    np.testing.assert_allclose(y4, y, rtol=1e-15)
    # eps is added to the mean square: with mean square 1 and eps 3, y = x / 2
    xs = _bf16(np.tile([1.0, -1.0], K // 2)[None, :])
    np.testing.assert_allclose(O.rms_norm_modulate(xs, zero, zero, 3.0)[0], np.tile([0.5, -0.5], K // 2))
    # the modulation is (1 + scale), not scale: scale = 0 keeps y, scale = -1 removes it
    minus_one = _bf16(np.full(K, -1.0))
    np.testing.assert_array_equal(O.rms_norm_modulate(x, zero, minus_one, 0.0), np.zeros((4, K)))


# ---------------------------------------------------------------- gate + residual

def test_gate_residual_definition():
    rng = np.random.default_rng(9)
    M, N, K = 3, 4, 64
    a = rng.integers(0, 64, size=(M, K)).astype(np.uint8)
    b = rng.integers(0, 64, size=(N, K)).astype(np.uint8)
    sa = np.full((M, K // 32), 127, np.uint8)
    sb = np.full((N, K // 32), 126, np.uint8)
    bias = _bf16(rng.standard_normal(N))
    gate = _bf16([0.0, 1.0, -0.5, 3.0])
    res = _bf16(rng.standard_normal((M, N)))
    c = O.gemm(a, sa, b, sb, bias)
    y = O.gate_residual(c, gate, res)
    exact = _exact_gemm(a, sa, b, sb, bias)
    for m in range(M):
        for n in range(N):
            ref = Fraction(float(synth.bf16_to_f32(res[m, n]))) + \
                Fraction(float(synth.bf16_to_f32(gate[n]))) * exact[m][n]
            assert abs(Fraction(y[m, n]) - ref) <= abs(ref) * Fraction(1, 2 ** 50), (m, n)
    # gate 0 passes the residual through untouched
    np.testing.assert_array_equal(y[:, 0], synth.bf16_to_f32(res[:, 0]).astype(np.float64))


# ---------------------------------------------------------------- DiT MLP sub-block

@pytest.mark.parametrize("activation", ["gelu", "swiglu"])
def test_dit_block_composes_its_steps(activation):
    w = synth.dit_block(M=8, d=128, ff=256, activation=activation)
    wuq, wus = O.quantize_bf16(w["w_up"])
    w2q, w2s = O.quantize_bf16(w["w2"])
    y, mid = O.dit_mlp_block(w["x"], w["shift"], w["scale"], w["gate"], w["eps"], wuq, wus, w["b_up"],
                             w2q, w2s, w["b2"], activation=activation)
    a = O.rms_norm_modulate(w["x"], w["shift"], w["scale"], w["eps"])
    xq, xs = O.quantize_f32(a.astype(np.float32))
    assert np.array_equal(xq, mid["xq"]) and np.array_equal(xs, mid["xs"])
    # a gate of zero returns the residual (x) exactly
    y0, _ = O.dit_mlp_block(w["x"], w["shift"], w["scale"], np.zeros_like(w["gate"]), w["eps"], wuq, wus,
                            w["b_up"], w2q, w2s, w["b2"], activation=activation)
    np.testing.assert_array_equal(y0, synth.bf16_to_f32(w["x"]).astype(np.float64))
    # with gate 1 the block adds the plain MLP output of the normalised input
    one = _bf16(np.ones_like(w["gate"], dtype=np.float32))
    y1, mid1 = O.dit_mlp_block(w["x"], w["shift"], w["scale"], one, w["eps"], wuq, wus, w["b_up"],
                               w2q, w2s, w["b2"], activation=activation)
    np.testing.assert_allclose(y1 - synth.bf16_to_f32(w["x"]), mid1["c"], rtol=1e-12, atol=1e-12)
