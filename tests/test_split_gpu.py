"""The GEMM's split tail on the GPU.

When the 256 x 256 output tiles leave a last round at most a quarter full for the
CTA pairs and the tiles are long (K >= 4096), the first pairs + (tiles mod pairs)
tiles are divided along K so that every pair does the same number of K-steps, and
a tile two pairs share is summed through the workspace. Checked here, on shapes
that split with GB300's 76 pairs:
  * the launch plan: the DiT down-projection splits, the full DiT block's GEMMs
    (whose last rounds are half full) do not;
  * the split result against the fp64 oracle (the library's GEMM tolerance);
  * tiles outside the split region bit-identical to the unsplit launch (same
    MMA sequence), split tiles within the tolerance of it;
  * the same result on repeated calls and in CUDA-graph replays (two partial
    sums are added in either order, and fp32 addition of two terms is commutative);
  * the fused GELU requantization bit-exact given the kernel's own fp32 values,
    SwiGLU and the gate/residual epilogue (in place) on split tiles;
  * the arrival counters zero again after every launch, partial slots holding
    garbage harmless, and an MLP workspace full of garbage harmless (its first
    kernel zeroes the counters).
"""

import numpy as np
import pytest

import oracle as O
import synth
from mxutil import (REL_TOL, RMS_TOL, assert_codes_equal, assert_gemm_close, assert_swiglu_close, bf16_from_device,
                    bf16_to_device, f32_from_bf16_bits, gemm_tolerance_report, graph_replays_match, mx_rows_to_host,
                    mx_to_host, mx_upload, requant_flip_report, sample_rows)

pytestmark = pytest.mark.gpu

TILE = 256


def _random_mx(rng, rows, k, lo=118, hi=124):
    codes = rng.integers(0, 64, size=(rows, k)).astype(np.uint8)
    scales = rng.integers(lo, hi, size=(rows, k // 32)).astype(np.uint8)
    return codes, scales


def _plan(lib, m, n, k):
    pairs, split = lib.mx_gemm_launch_plan(m, n, k)
    tiles = -(-m // TILE) * (n // TILE)
    if split == 0:
        pytest.skip(f"{tiles} tiles fill this device's {pairs} CTA pairs evenly: nothing to split")
    assert split == pairs + tiles % pairs
    assert lib.mx_gemm_launch_plan(m, n, k, 0) == (pairs, 0)   # no workspace: no split
    return tiles, split


def _split_mask(m, n, split_tiles):
    """[m][n] bool: outputs in the tiles divided along K (the first split_tiles, row-major)."""
    num_n = n // TILE
    mask = np.zeros((m, n), bool)
    for t in range(split_tiles):
        pm, nb = divmod(t, num_n)
        mask[pm * TILE:(pm + 1) * TILE, nb * TILE:(nb + 1) * TILE] = True
    return mask


def _bf16(y):
    return f32_from_bf16_bits(bf16_from_device(y)).astype(np.float64)


def test_launch_plan_policy(lib):
    """Split when the leftover round is at most a quarter full and K >= 4096."""
    for m, n, k in [(16384, 3072, 12288),   # DiT down-projection: 768 tiles
                    (20480, 3072, 12288),   # full block down-projection: 960 tiles
                    (20480, 12288, 3072),   # full block up-projection: K = 3072
                    (4096, 12288, 3072),    # DiT up-projection: K = 3072
                    (20480, 4096, 16384)]:  # outlier MLP down-projection: 1280 tiles
        pairs, split = lib.mx_gemm_launch_plan(m, n, k)
        tiles = -(-m // TILE) * (n // TILE)
        rem = tiles % pairs
        want = pairs + rem if (tiles > pairs and 0 < rem <= pairs // 4 and k >= 4096) else 0
        assert split == want, (m, n, k, pairs, split)
        if split:
            assert (tiles - split) % pairs == 0


@pytest.mark.parametrize("M,N,K", [(5000, 1024, 4096),    # 80 tiles: all in the split region
                                   (4900, 1024, 4096),    # the last pair's second CTA wholly past M
                                   (8292, 1280, 4096)])   # 165 tiles: one whole round + the split region
def test_split_bf16_matches_oracle_and_unsplit(lib, M, N, K):
    import torch

    tiles, split = _plan(lib, M, N, K)
    rng = np.random.default_rng(M + N + K)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, N, K)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32))
    A, B, bias_d = mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias)
    ys = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_BF16)
    ys2 = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_BF16)
    yu = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_BF16, split=False)
    assert torch.equal(ys, ys2), "split result differs between calls"
    got, unsplit = _bf16(ys), _bf16(yu)
    mask = _split_mask(M, N, split)
    assert np.array_equal(got[~mask], unsplit[~mask]), "whole tiles differ from the unsplit launch"
    assert_gemm_close(got[mask], unsplit[mask], "split tiles vs unsplit")
    rows = sample_rows(M, 256) if M * N * K > 3e10 else np.arange(M)
    assert_gemm_close(got[rows], O.gemm(a[rows], sa[rows], b, sb, bias), f"split bf16 {M}x{N}x{K}")
    assert lib.mx_device_error() == 0


def test_split_gelu_requant(lib):
    import torch

    M, N, K = 5000, 1024, 4096
    _, split = _plan(lib, M, N, K)
    rng = np.random.default_rng(21)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, N, K)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32))
    A, B, bias_d = mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias)
    dbg = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    dbg_u = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    out_dbg = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=dbg)
    out = lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_GELU_MXFP6)
    lib.mx_gemm(A, B, bias_d, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=dbg_u, split=False)
    assert torch.equal(out.codes, out_dbg.codes) and torch.equal(out.scales, out_dbg.scales)
    g, gu = dbg.cpu().numpy(), dbg_u.cpu().numpy()
    assert np.isfinite(g).all()
    mask = _split_mask(M, N, split)
    assert np.array_equal(g[~mask], gu[~mask])
    assert_gemm_close(g, O.up_projection(a, sa, b, sb, bias), "split gelu pre-quant")
    codes, scales = mx_to_host(out)
    rc, rs = O.quantize_f32(g)
    assert_codes_equal(codes, rc, scales, rs, "split requant")


def test_split_swiglu(lib):
    M, F, K = 5000, 512, 4096
    _plan(lib, M, 2 * F, K)
    import torch

    rng = np.random.default_rng(22)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, 2 * F, K)
    bias = synth.bf16_round(rng.standard_normal(2 * F).astype(np.float32))
    dbg = torch.full((M, F), float("nan"), dtype=torch.float32, device="cuda")
    out = lib.mx_gemm(mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias), lib.MX_EPI_BIAS_SWIGLU_MXFP6,
                      debug_prequant=dbg)
    h = dbg.cpu().numpy()
    assert np.isfinite(h).all()
    assert_swiglu_close(h, O.gemm(a, sa, b, sb, bias), "split swiglu")
    codes, scales = mx_to_host(out)
    rc, rs = O.quantize_f32(h)
    assert_codes_equal(codes, rc, scales, rs, "split swiglu requant")


def test_split_gate_residual_in_place(lib):
    M, N, K = 5000, 1024, 4096
    _, split = _plan(lib, M, N, K)
    rng = np.random.default_rng(23)
    a, sa = _random_mx(rng, M, K)
    b, sb = _random_mx(rng, N, K)
    bias = synth.bf16_round(rng.standard_normal(N).astype(np.float32))
    gate = synth.bf16_round(rng.standard_normal(N).astype(np.float32))
    res = synth.bf16_round(rng.standard_normal((M, N)).astype(np.float32) * 4)
    r = bf16_to_device(res)
    lib.mx_gemm_gate_residual(mx_upload(a, sa), mx_upload(b, sb), bf16_to_device(bias), bf16_to_device(gate), r,
                              out=r)
    c = O.gemm(a, sa, b, sb, bias)
    g64 = f32_from_bf16_bits(gate).astype(np.float64)
    ref = f32_from_bf16_bits(res).astype(np.float64) + g64 * c
    got = _bf16(r)
    rms = np.sqrt(np.mean(c * c))
    bound = np.abs(g64) * (2.0 ** -7 * np.abs(c) + 1e-3 * rms) + 2.0 ** -8 * np.abs(ref) + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{int(bad.sum())} outside; split tiles {split}"


def test_split_workspace_counters_return_to_zero(lib):
    """A workspace whose counters are zero and whose partial slots hold garbage gives
    the same result as a fresh one, and every launch leaves the counters zero."""
    import torch

    M, N, K = 5000, 1024, 4096
    _plan(lib, M, N, K)
    rng = np.random.default_rng(24)
    A, B = mx_upload(*_random_mx(rng, M, K)), mx_upload(*_random_mx(rng, N, K))
    ws = torch.full((lib.mx_gemm_workspace_bytes(M, N, K),), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:lib.MX_GEMM_WORKSPACE_COUNTER_BYTES] = 0
    clean = lib.mx_gemm(A, B, None, lib.MX_EPI_BIAS_BF16)
    for _ in range(3):
        got = lib.mx_gemm(A, B, None, lib.MX_EPI_BIAS_BF16, workspace=ws)
        assert torch.equal(clean, got)
        assert int(ws[:lib.MX_GEMM_WORKSPACE_COUNTER_BYTES].count_nonzero()) == 0
    assert lib.mx_device_error() == 0


def test_mlp_split_tail(lib):
    """mx_mlp with its full workspace (split tail) against a workspace that holds only
    MXFP6 x and h (no split), and with a garbage-filled workspace (the quantizer
    zeroes the counters): identical results, and the split MLP close to the unsplit one."""
    import torch

    M, d, ff = 5000, 4096, 4096
    _plan(lib, M, ff, d)
    _plan(lib, M, d, ff)
    rng = np.random.default_rng(25)
    x = bf16_to_device(synth.bf16_round(rng.standard_normal((M, d)).astype(np.float32)))
    w1 = lib.mx_quantize(bf16_to_device(synth.bf16_round(rng.standard_normal((ff, d)).astype(np.float32) * 0.02)))
    w2 = lib.mx_quantize(bf16_to_device(synth.bf16_round(rng.standard_normal((d, ff)).astype(np.float32) * 0.02)))
    b1 = bf16_to_device(synth.bf16_round(rng.standard_normal(ff).astype(np.float32) * 0.01))
    b2 = bf16_to_device(synth.bf16_round(rng.standard_normal(d).astype(np.float32) * 0.01))
    full = lib.mx_mlp_workspace_bytes(M, d, ff)
    base = sum(-(-n // 256) * 256 for n in (lib.mx_codes_bytes(M, d), lib.mx_scales_bytes(M, d),
                                            lib.mx_codes_bytes(M, ff), lib.mx_scales_bytes(M, ff),
                                            4 * (-(-M // 128))))   # + a counter word per 128 rows
    assert full > base
    y = lib.mx_mlp(x, w1, b1, w2, b2)
    ws = torch.full((full,), 0xFF, dtype=torch.uint8, device="cuda")
    y_dirty = lib.mx_mlp(x, w1, b1, w2, b2, workspace=ws)
    y_again = lib.mx_mlp(x, w1, b1, w2, b2, workspace=ws)
    assert torch.equal(y, y_dirty) and torch.equal(y, y_again)
    y_unsplit = lib.mx_mlp(x, w1, b1, w2, b2, workspace=torch.empty(base, dtype=torch.uint8, device="cuda"))
    # The same two GEMMs one by one, split and unsplit, with the GELU values the
    # requantization rounded: each MLP equals its stages bit for bit.
    xq = lib.mx_quantize(x)
    g_s = torch.empty((M, ff), dtype=torch.float32, device="cuda")
    g_u = torch.empty((M, ff), dtype=torch.float32, device="cuda")
    hq_s = lib.mx_gemm(xq, w1, b1, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=g_s)
    hq_u = lib.mx_gemm(xq, w1, b1, lib.MX_EPI_BIAS_GELU_MXFP6, debug_prequant=g_u, split=False)
    assert torch.equal(y, lib.mx_gemm(hq_s, w2, b2, lib.MX_EPI_BIAS_BF16))
    assert torch.equal(y_unsplit, lib.mx_gemm(hq_u, w2, b2, lib.MX_EPI_BIAS_BF16, split=False))
    # The two fp32 up-projections differ only in summation order. Their codes may
    # differ only where the two values straddle a rounding boundary: within the
    # values' own difference of one. On sampled rows, each output then stays within
    # the GEMM tolerance of the oracle given its own intermediate, and the two
    # oracle outputs differ exactly by the differing codes' contribution.
    rows = sample_rows(M, n_random=64)
    idx = torch.as_tensor(rows, device="cuda")
    gs, gu = g_s[idx].cpu().numpy(), g_u[idx].cpu().numpy()
    cs, ss = mx_rows_to_host(hq_s, rows)
    cu, su = mx_rows_to_host(hq_u, rows)
    diff = np.abs(gs.astype(np.float64) - gu.astype(np.float64))
    flips, _ = requant_flip_report(cs, ss, cu, su, gu, diff + 1e-30)
    w2c, w2s = mx_to_host(w2)
    ref_s = O.down_projection(cs, ss, w2c, w2s, bf16_from_device(b2))
    ref_u = O.down_projection(cu, su, w2c, w2s, bf16_from_device(b2))
    ys, yu = _bf16(y[idx]), _bf16(y_unsplit[idx])
    assert_gemm_close(ys, ref_s, "split MLP")
    assert_gemm_close(yu, ref_u, "unsplit MLP")
    tol = lambda r: REL_TOL * np.abs(r) + RMS_TOL * np.sqrt(np.mean(r ** 2))  # noqa: E731
    bound = tol(ref_s) + tol(ref_u) + np.abs(ref_s - ref_u)
    assert not (np.abs(ys - yu) > bound).any(), flips
    assert lib.mx_device_error() == 0


def test_split_mlp_graph_replay(lib):
    """mx_mlp with both GEMMs split, captured once and replayed on fresh inputs:
    each replay equals an eager call bit for bit (the first kernel zeroes the
    counters inside the graph too)."""
    import torch

    M, d, ff = 5000, 4096, 4096
    _plan(lib, M, ff, d)
    _plan(lib, M, d, ff)
    rng = np.random.default_rng(26)

    def bf16(shape, sd):
        return bf16_to_device(synth.bf16_round(rng.standard_normal(shape).astype(np.float32) * sd))

    w1, w2 = lib.mx_quantize(bf16((ff, d), 0.02)), lib.mx_quantize(bf16((d, ff), 0.02))
    b1, b2 = bf16(ff, 0.01), bf16(d, 0.01)
    ws = torch.empty(lib.mx_mlp_workspace_bytes(M, d, ff), dtype=torch.uint8, device="cuda")
    x = bf16((M, d), 1.0)
    y = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")

    def run(xi, yi):
        lib.mx_mlp(xi, w1, b1, w2, b2, y=yi, workspace=ws)

    graph_replays_match(lib, run, lambda s: bf16((M, d), 1.0), x, y, n=3)
