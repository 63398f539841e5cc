"""Pins for the CPU oracle: each check ties it to something other than itself.

Sources of truth used here: the OCP MX v1.0 E2M3 value table typed in by hand
(tests/golden/e2m3_values.txt), CUDA's own host-side fp6 conversion routines
(cuda_fp6.h, compiled for the host and called, never re-implemented),
hand-derived fixtures (tests/golden/quant_blocks.txt, pack_example.txt),
exact integer arithmetic in pure Python, closed-form GELU identities and the
erf-based GELU.
"""

import math
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HELPER_SRC = os.path.join(os.path.dirname(__file__), "helpers", "fp6_host_ref.cpp")
HELPER_BIN = os.path.join(os.path.dirname(__file__), "_bin", "fp6_host_ref")
CUDA_INC = "/usr/local/cuda/include"


def _golden_table():
    vals = {}
    with open(os.path.join(GOLDEN, "e2m3_values.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            code, val = line.split()
            vals[int(code, 16)] = float(val)
    assert sorted(vals) == list(range(32))
    return vals


def _helper():
    """Build (once) the host program that calls cuda_fp6.h's conversions."""
    cxx = shutil.which("g++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_fp6.h")):
        pytest.skip("g++ or cuda_fp6.h not available")
    if not os.path.exists(HELPER_BIN) or os.path.getmtime(HELPER_BIN) < os.path.getmtime(HELPER_SRC):
        os.makedirs(os.path.dirname(HELPER_BIN), exist_ok=True)
        subprocess.run([cxx, "-O1", "-I", CUDA_INC, HELPER_SRC, "-o", HELPER_BIN], check=True)
    return HELPER_BIN


def _cuda_encode(values_f32):
    out = subprocess.run([_helper(), "encode"], input=np.asarray(values_f32, np.float32).tobytes(),
                         capture_output=True, check=True).stdout
    return np.frombuffer(out, dtype=np.uint8)


# ---------------------------------------------------------------- element table

def test_e2m3_table_matches_ocp_table():
    golden = _golden_table()
    for c in range(32):
        assert O.E2M3_TABLE[c] == golden[c]
        neg = O.E2M3_TABLE[c | 0x20]
        assert neg == -golden[c] and math.copysign(1.0, neg) == -1.0


def test_e2m3_table_matches_cuda_header_decode():
    out = subprocess.run([_helper(), "decode"], capture_output=True, check=True, text=True).stdout
    halves = np.array([int(x) for x in out.split()], dtype=np.uint16).view(np.float16)
    assert halves.shape == (64,)
    np.testing.assert_array_equal(halves.astype(np.float64), O.E2M3_TABLE)
    assert np.array_equal(np.signbit(halves), np.signbit(O.E2M3_TABLE))


def test_e8m0_values():
    assert O.e8m0_value(127) == 1.0
    assert O.e8m0_value(0) == 2.0 ** -127
    assert O.e8m0_value(254) == 2.0 ** 127
    assert np.isnan(O.e8m0_value(255))


# ---------------------------------------------------------------- rounding

def test_nearest_matches_cuda_header_on_every_bf16_pattern():
    """Every finite BF16 value (scale 1): the brute-force nearest search must equal
    CUDA's host E2M3 round-to-nearest conversion, including saturation and -0."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = synth.bf16_to_f32(bits)
    f = f[np.isfinite(f)]
    ours = O.nearest_e2m3_code(f.astype(np.float64))
    theirs = _cuda_encode(f)
    bad = np.nonzero(ours != theirs)[0]
    assert bad.size == 0, [(float(f[i]), int(ours[i]), int(theirs[i])) for i in bad[:10]]


def test_nearest_matches_cuda_header_on_midpoints_and_random_f32():
    mags = O.E2M3_TABLE[:32]
    mids = (mags[1:] + mags[:-1]) / 2
    eps = np.ldexp(1.0, -20)
    pts = np.concatenate([mids, mids + eps, mids - eps, mags, [7.5 + eps, 7.75, 7.76, 8.0, 1e30]])
    pts = np.concatenate([pts, -pts])
    rng = np.random.default_rng(1234)
    pts = np.concatenate([pts, rng.uniform(-9.0, 9.0, 200000)]).astype(np.float32)
    ours = O.nearest_e2m3_code(pts.astype(np.float64))
    theirs = _cuda_encode(pts)
    np.testing.assert_array_equal(ours, theirs)


# ---------------------------------------------------------------- blocks

def _read_blocks():
    blocks = []
    with open(os.path.join(GOLDEN, "quant_blocks.txt")) as f:
        cur = None
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            parts = line.split()
            if parts[0] == "block":
                cur = {"name": parts[1], "scale": int(parts[2]), "v": [], "c": []}
                blocks.append(cur)
            else:
                cur["v"].append(float.fromhex(parts[0]))
                cur["c"].append(int(parts[1], 16))
    return blocks


def test_quantize_hand_derived_blocks():
    blocks = _read_blocks()
    assert len(blocks) == 7
    v = np.array([b["v"] for b in blocks], dtype=np.float64).reshape(1, -1)
    # every value is exact in BF16: round trip through the generator's rounding
    assert np.array_equal(synth.bf16_to_f32(synth.bf16_round(v.astype(np.float32))).astype(np.float64), v)
    codes, scales = O.quantize(v)
    assert scales.reshape(-1).tolist() == [b["scale"] for b in blocks]
    for i, b in enumerate(blocks):
        got = codes[0, 32 * i:32 * (i + 1)].tolist()
        assert got == b["c"], (b["name"], [hex(x) for x in got])


def test_shared_exponent_special_cases():
    # floor(log2 a) - 2, by hand
    cases = [(1.0, -2), (7.99, 0), (8.0, 1), (4.0, 0), (3.999, -1), (0.0, -127),
             (2.0 ** -126, -127), (2.0 ** -125, -127), (2.0 ** -124, -126),
             (2.0 ** -140, -127), (float(np.finfo(np.float32).max), 125), (6.0e4, 13)]
    for a, s in cases:
        assert int(O.shared_exponent(a)) == s, a


def test_round_trip_every_code_at_many_scales():
    """Dequantize -> quantize returns the same codes and scale, for all 64 codes
    at several scales, in blocks anchored by a top-binade element."""
    rng = np.random.default_rng(7)
    for anchor in (0x1F, 0x18, 0x3C):
        for s in (-127, -20, -1, 0, 1, 20, 125):
            codes = rng.integers(0, 64, size=(64, 32)).astype(np.uint8)
            codes[:, 0] = anchor
            codes[:, 1] = np.arange(64, dtype=np.uint8)
            scales = np.full((64, 1), s + 127, dtype=np.uint8)
            vals = O.dequantize(codes, scales)
            c2, s2 = O.quantize(vals)
            assert np.array_equal(s2, scales)
            # +0 and -0 are the same value but keep their sign bit
            assert np.array_equal(c2, codes), s


def _half_grid_step(t):
    a = np.abs(t)
    return np.where(a < 2.0, 0.0625, np.where(a < 4.0, 0.125, 0.25))


@pytest.mark.parametrize("law", ["normal", "student_t", "tiny", "huge", "mixed"])
def test_block_invariants(law):
    rng = np.random.default_rng({"normal": 1, "student_t": 2, "tiny": 3, "huge": 4, "mixed": 5}[law])
    shape = (256, 128)
    if law == "normal":
        v = rng.standard_normal(shape)
    elif law == "student_t":
        v = rng.standard_t(3.0, shape) * 100
    elif law == "tiny":
        v = rng.standard_normal(shape) * 2.0 ** -128
    elif law == "huge":
        v = rng.standard_normal(shape) * 2.0 ** 120
    else:
        v = rng.standard_normal(shape) * np.exp(rng.uniform(-30, 30, shape))
    v = synth.bf16_to_f32(synth.bf16_round(v.astype(np.float32))).astype(np.float64)
    v[:8, :32] = 0.0                       # all-zero blocks
    codes, scales = O.quantize(v)
    blocks = v.reshape(256, 4, 32)
    cb = codes.reshape(256, 4, 32)
    s = scales.astype(np.int64) - 127
    amax = np.abs(blocks).max(axis=2)
    t = blocks * np.ldexp(1.0, -s)[:, :, None]
    # (i) the block maximum lands in the top binade [4, 8) unless the scale clamps
    idx = np.abs(blocks).argmax(axis=2)
    top = np.take_along_axis(cb, idx[:, :, None], axis=2)[:, :, 0]
    live = (amax > 0) & (s > -127)
    assert np.all(((top >> 3) & 3)[live] == 3)
    tmax = np.abs(np.take_along_axis(t, idx[:, :, None], axis=2)[:, :, 0])
    assert np.all((tmax[live] >= 4.0) & (tmax[live] < 8.0))
    # (ii) an all-zero block gives zero codes and the zero-block scale
    assert np.all(codes[:8, :32] == 0) and np.all(scales[:8, 0] == 0)
    # (iii) saturation: |t| >= 7.5 gives magnitude code 0x1F
    sat = np.abs(t) >= 7.5
    assert np.all((cb[sat] & 0x1F) == 0x1F)
    # (iv) error bound: half a grid step (times the scale) for unsaturated elements
    deq = O.dequantize(codes, scales).reshape(256, 4, 32)
    err = np.abs(deq - blocks) * np.ldexp(1.0, -s)[:, :, None]
    assert np.all(err[~sat] <= _half_grid_step(t[~sat]))
    # sign bit follows the sign of the input
    assert np.array_equal((cb & 0x20) != 0, np.signbit(blocks))


def test_non_finite_block_reading():
    v = np.ones((1, 64))
    v[0, 3] = np.inf
    v[0, 40] = np.nan
    codes, scales = O.quantize(v)
    assert scales.tolist() == [[0xFF, 0xFF]]
    assert np.all(codes == 0)


# ---------------------------------------------------------------- storage formats

def test_pack_hand_derived_example():
    with open(os.path.join(GOLDEN, "pack_example.txt")) as f:
        lines = [l for l in f if not l.startswith("#") and l.strip()]
    pairs = list(zip(lines[0::2], lines[1::2]))
    assert len(pairs) == 2
    for c_line, b_line in pairs:
        codes = np.array([int(x, 16) for x in c_line.split(":")[1].split()], dtype=np.uint8)[None]
        want = np.array([int(x, 16) for x in b_line.split(":")[1].split()], dtype=np.uint8)[None]
        assert np.array_equal(O.pack_codes(codes), want)
        assert np.array_equal(O.unpack_codes(want, 16), codes)


def test_pack_matches_big_integer_bit_string():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 64, size=(5, 96)).astype(np.uint8)
    packed = O.pack_codes(codes)
    for r in range(5):
        big = 0
        for j, c in enumerate(codes[r].tolist()):
            big |= c << (6 * j)
        assert packed[r].tobytes() == big.to_bytes(72, "little")
    assert np.array_equal(O.unpack_codes(packed, 96), codes)


def test_tiled_scale_layout_positions():
    # rows 256, K 256 -> 2 atoms per 128-row group. By hand:
    # (row 33, kb 5): atom 0*2 + 1 = 1; r0 = 1, r1 = 1, j = 1 -> 512 + 16 + 4 + 1 = 533
    # (row 130, kb 0): atom 1*2 + 0 = 2; r0 = 2, r1 = 0 -> 1024 + 32 = 1056
    # (row 127, kb 7): atom 1; r0 = 31, r1 = 3, j = 3 -> 512 + 496 + 12 + 3 = 1023
    # (row 255, kb 4): atom 3; r0 = 31, r1 = 3, j = 0 -> 1536 + 496 + 12 = 2044
    plain = np.zeros((256, 8), dtype=np.uint8)
    marks = {(33, 5): 11, (130, 0): 22, (127, 7): 33, (255, 4): 44}
    for (r, kb), val in marks.items():
        plain[r, kb] = val
    tiled = O.scales_plain_to_tiled(plain, 256, 256)
    assert tiled.size == 256 * 8
    for (r, kb), off in {(33, 5): 533, (130, 0): 1056, (127, 7): 1023, (255, 4): 2044}.items():
        assert tiled[off] == marks[(r, kb)]
    # bijection + ragged rows padded to 128 with the pad value
    rng = np.random.default_rng(0)
    p = rng.integers(0, 255, size=(300, 12)).astype(np.uint8)
    t = O.scales_plain_to_tiled(p, 300, 384, pad_value=0)
    assert t.size == 384 * 12
    assert np.array_equal(O.scales_tiled_to_plain(t, 300, 384), p)
    assert np.count_nonzero(t) == np.count_nonzero(p)


# ---------------------------------------------------------------- GEMM

def _golden_int8_value(code, golden):
    """8 x E2M3 value as an exact integer, from the hand-typed OCP table."""
    v = golden[code & 0x1F] * 8
    assert v == int(v)
    return -int(v) if code & 0x20 else int(v)


@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (3, 5, 64), (8, 7, 128), (6, 8, 96)])
def test_tiny_gemm_equals_exact_integer_block_sums(M, N, K):
    golden = _golden_table()
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    a = rng.integers(0, 64, size=(M, K)).astype(np.uint8)
    b = rng.integers(0, 64, size=(N, K)).astype(np.uint8)
    sa = rng.integers(124, 131, size=(M, K // 32)).astype(np.uint8)
    sb = rng.integers(124, 131, size=(N, K // 32)).astype(np.uint8)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32))
    got = O.gemm(a, sa, b, sb, bias)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for blk in range(K // 32):
                isum = 0
                for k in range(32 * blk, 32 * blk + 32):
                    isum += _golden_int8_value(a[m, k], golden) * _golden_int8_value(b[n, k], golden)
                e = int(sa[m, blk]) + int(sb[n, blk]) - 254 - 6
                acc += Fraction(isum) * (Fraction(2) ** e)
            acc += Fraction(float(synth.bf16_to_f32(bias[n])))
            assert got[m, n] == float(acc), (m, n)


def test_gemm_is_not_transposed():
    # A = [[1, 0, ...]], B rows pick distinct columns: C[m][n] = A[m][n]
    a = np.zeros((2, 32), dtype=np.uint8)
    b = np.zeros((3, 32), dtype=np.uint8)
    a[0, 0] = 0x08   # 1.0
    a[1, 1] = 0x10   # 2.0
    b[0, 0] = 0x18   # 4.0
    b[1, 1] = 0x04   # 0.5
    b[2, 0] = 0x28   # -1.0
    s1 = np.full((2, 1), 127, np.uint8)
    s2 = np.full((3, 1), 127, np.uint8)
    c = O.gemm(a, s1, b, s2)
    assert c.tolist() == [[4.0, 0.0, -1.0], [0.0, 1.0, 0.0]]


# ---------------------------------------------------------------- GELU

def test_gelu_closed_forms():
    x = np.linspace(-6, 6, 2001)
    g = O.gelu_tanh(x)
    assert O.gelu_tanh(0.0) == 0.0
    # odd part: gelu(x) - gelu(-x) = x exactly in exact arithmetic
    np.testing.assert_allclose(g - O.gelu_tanh(-x), x, rtol=0, atol=4e-15)
    # limits
    assert abs(O.gelu_tanh(30.0) - 30.0) < 1e-12
    assert abs(O.gelu_tanh(-30.0)) < 1e-12
    # the tanh form approximates x * Phi(x) to within 1e-3 (textbook GELU)
    phi = 0.5 * (1 + np.vectorize(math.erf)(x / math.sqrt(2)))
    assert np.max(np.abs(g - x * phi)) < 1e-3


def test_gelu_fp64_accuracy_against_mpmath():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    xs = [-8.0, -3.3, -1.0, -0.25, 1e-3, 0.5, 1.7, 4.0, 9.0]
    for x in xs:
        u = mp.sqrt(2 / mp.pi) * (x + mp.mpf("0.044715") * x ** 3)
        ref = mp.mpf("0.5") * x * (1 + mp.tanh(u))
        got = O.gelu_tanh(x)
        # the 0.5 v (1 + tanh) form cancels for negative v: the error is
        # absolute there (1 + tanh rounds at 1 ulp of 1.0), relative elsewhere
        assert abs(mp.mpf(float(got)) - ref) <= 1e-14 * abs(ref) + 1e-15 * (1 + abs(x))


# ---------------------------------------------------------------- MLP chain

def test_mlp_chain_on_tiny_workload():
    w = synth.full_mlp(M=8, d=128, ff=256)
    w1q, w1s = O.quantize_bf16(w["w1"])
    w2q, w2s = O.quantize_bf16(w["w2"])
    y, mid = O.mlp(w["x"], w1q, w1s, w["b1"], w2q, w2s, w["b2"])
    assert y.shape == (8, 128)
    # intermediate is the fp32-rounded GELU of the up-projection, requantized
    g32 = mid["g"].astype(np.float32)
    hq, hs = O.quantize_f32(g32)
    assert np.array_equal(hq, mid["hq"]) and np.array_equal(hs, mid["hs"])
    # the requantized intermediate stays within the MXFP6 error bound of g
    deq = O.dequantize(hq, hs)
    # half a step of the top binade (0.25), or 0.5 where [7.5, 8) saturates
    step = np.repeat(np.ldexp(1.0, hs.astype(np.int64) - 127), 32, axis=1) * 0.5
    assert np.all(np.abs(deq - g32.astype(np.float64)) <= step)
