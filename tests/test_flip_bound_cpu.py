"""The derived bound the end-to-end GPU tests use for requantization flips
(mxutil.near_rounding_boundary / requant_flip_report), checked on the CPU with the
oracle's own encoder: inputs perturbed by at most tol must encode identically
outside the elements the helper marks as near a rounding boundary, and a value on
a boundary, at zero, or a block amax at a power of two must be marked."""

import numpy as np

import oracle as O
from mxutil import near_rounding_boundary, requant_flip_report


def test_perturbations_within_tol_only_flip_marked_elements():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal((96, 256)) * np.exp2(rng.integers(-6, 6, size=(96, 1)))).astype(np.float32)
    c0, s0 = O.quantize_f32(v)
    for scale in (1e-4, 1e-3, 1e-2):
        tol = scale * np.abs(v.astype(np.float64)) + scale * 1e-2
        total = 0
        for _ in range(8):
            p = (v + rng.uniform(-1, 1, v.shape) * tol).astype(np.float32)
            c1, s1 = O.quantize_f32(p)
            rep, _ = requant_flip_report(c1, s1, c0, s0, v, tol)   # asserts every flip is marked
            total += rep["differing"]
        assert total > 0   # the perturbations do reach boundaries


def test_marks_boundaries_zero_and_scale_edges():
    block = np.full((1, 32), 4.0)          # amax 4 = 2^2: scale exponent 0, values at t = 4
    block[0, 1] = 1.0625                   # t = 1.0625: midpoint between the E2M3 values 1.0 and 1.125
    block[0, 2] = 1e-9                     # next to zero: the sign bit could change
    block[0, 3] = 2.5                      # an E2M3 value itself, far from any boundary
    near = near_rounding_boundary(block, np.full(block.shape, 1e-6))
    assert near[0, 1] and near[0, 2]
    assert near.all()                      # the amax sits on a power of two: the scale could change
    block[0, 0] = 5.0
    block[0, 4:] = 5.0                     # amax 5: no scale edge within 1e-6
    near = near_rounding_boundary(block, np.full(block.shape, 1e-6))
    assert near[0, 1] and near[0, 2] and not near[0, 3] and not near[0, 0]
