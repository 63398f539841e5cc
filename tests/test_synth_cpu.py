"""The counter-based BF16 generator that fills tensors too large to draw on the
host: its numpy and torch forms give the same bits (so a test may fill the device
tensor with one and regenerate checked rows with the other), the values follow
the stated law, and rows far apart differ."""

import numpy as np
import pytest

import synth


def test_hash_generator_numpy_and_torch_agree_at_large_row_indices():
    torch = pytest.importorskip("torch")
    k = 2304
    for row0 in (0, 932066, 1_299_998, (1 << 31) - 3):
        t = torch.empty((3, k), dtype=torch.bfloat16)
        synth.hash_bf16_fill_(t, seed=5, row0=row0, slab_rows=2)
        got = t.view(torch.int16).numpy().view(np.uint16)
        np.testing.assert_array_equal(got, synth.hash_bf16_rows(np.arange(row0, row0 + 3), k, seed=5))


def test_hash_generator_value_law():
    bits = synth.hash_bf16_rows(np.arange(256), 1024, seed=0)
    exp = (bits >> 7) & 0xFF
    assert exp.min() == 118 and exp.max() == 133          # finite normal values, 2^-9 .. 2^7
    counts = np.bincount(exp.ravel(), minlength=134)[118:134]
    assert counts.min() > 0.9 * bits.size / 16 and counts.max() < 1.1 * bits.size / 16
    assert abs(float((bits >> 15).mean()) - 0.5) < 0.01    # signs balanced
    v = synth.bf16_to_f32(bits)
    assert np.isfinite(v).all() and np.abs(v).min() >= 2.0 ** -9 and np.abs(v).max() < 2.0 ** 7


def test_hash_generator_rows_and_seeds_differ():
    a = synth.hash_bf16_rows([0, 1, 1 << 20, (1 << 20) + 1], 512, seed=0)
    assert len({row.tobytes() for row in a}) == 4
    assert not np.array_equal(a, synth.hash_bf16_rows([0, 1, 1 << 20, (1 << 20) + 1], 512, seed=1))
    # lowbias32 of key 0 is 0: element (0, 0) of seed 0 is the smallest positive value
    assert a[0, 0] == (118 << 7)
