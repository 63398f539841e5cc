"""Shared helpers of the GPU parity tests: moving synthetic inputs to the device,
reading MXFP6 results back into the oracle's plain layout, and the GEMM tolerance.

The tolerance is the library's contract for every GEMM output:
    |gpu - oracle| <= 2^-7 * |oracle| + 1e-3 * rms(oracle)
where rms is taken over the compared elements.
"""

from __future__ import annotations

import numpy as np

import oracle as O

REL_TOL = 2.0 ** -7
RMS_TOL = 1e-3
SILU_LIP = 1.1      # max |silu'(v)| is 1.0998


def bf16_to_device(bits: np.ndarray):
    import torch

    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def bf16_from_device(t) -> np.ndarray:
    import torch

    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_from_bf16_bits(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def mx_to_host(mxt, rows=None):
    """MxTensor -> (codes uint8 [rows][K], plain scales uint8 [rows][K/32]) via the oracle's layout code."""
    codes_packed = mxt.codes.cpu().numpy().reshape(mxt.rows, -1)
    tiled = mxt.scales.cpu().numpy()
    codes = O.unpack_codes(codes_packed, mxt.k)
    plain = O.scales_tiled_to_plain(tiled, mxt.rows, mxt.k)
    if rows is not None:
        return codes[rows], plain[rows]
    return codes, plain


def mx_rows_to_host(mxt, rows):
    """Only the listed rows (cheaper for big tensors)."""
    import torch

    idx = torch.as_tensor(np.asarray(rows), device=mxt.codes.device)
    packed = mxt.codes.index_select(0, idx).cpu().numpy()
    tiled = mxt.scales.cpu().numpy()
    codes = O.unpack_codes(packed, mxt.k)
    plain_all = O.scales_tiled_to_plain(tiled, mxt.rows, mxt.k)
    return codes, plain_all[np.asarray(rows)]


def mx_upload(codes: np.ndarray, plain_scales: np.ndarray):
    """Oracle-made MXFP6 matrix (plain layout) -> device MxTensor in the library layout."""
    import torch

    import microscaled_precision_gemm_gb300 as mx

    rows, k = codes.shape
    packed = O.pack_codes(codes)
    tiled = O.scales_plain_to_tiled(plain_scales, rows, k, pad_value=0)
    return mx.MxTensor(torch.from_numpy(packed).cuda(), torch.from_numpy(tiled).cuda(), rows, k)


def sample_rows(m: int, n_random: int = 192, seed: int = 0) -> np.ndarray:
    """First and last row of every 128-row tile, plus seeded random rows."""
    tiles = (m + 127) // 128
    edge = np.concatenate([np.arange(tiles) * 128, np.minimum(np.arange(tiles) * 128 + 127, m - 1)])
    rnd = np.random.default_rng(seed).integers(0, m, size=n_random)
    return np.unique(np.concatenate([edge, rnd]))


def gemm_tolerance_report(gpu: np.ndarray, ref: np.ndarray) -> dict:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    bound = REL_TOL * np.abs(ref) + RMS_TOL * rms
    err = np.abs(gpu - ref)
    bad = err > bound
    return {"rms": rms, "max_err": float(err.max()) if err.size else 0.0,
            "n_bad": int(bad.sum()), "frac_ok": float(1 - bad.mean()) if err.size else 1.0,
            "worst": float((err / np.maximum(bound, 1e-300)).max()) if err.size else 0.0}


def assert_gemm_close(gpu, ref, what=""):
    r = gemm_tolerance_report(gpu, ref)
    assert r["n_bad"] == 0, f"{what}: {r}"
    return r


def assert_codes_equal(gpu_codes, ref_codes, gpu_scales, ref_scales, what=""):
    gs, rs = np.asarray(gpu_scales), np.asarray(ref_scales)
    if not np.array_equal(gs, rs):
        idx = np.argwhere(gs != rs)[:8]
        raise AssertionError(f"{what}: scales differ at {idx.tolist()}: gpu {gs[tuple(idx.T)].tolist()} "
                             f"oracle {rs[tuple(idx.T)].tolist()}")
    gc, rc = np.asarray(gpu_codes), np.asarray(ref_codes)
    if not np.array_equal(gc, rc):
        idx = np.argwhere(gc != rc)[:8]
        raise AssertionError(f"{what}: {int((gc != rc).sum())} codes differ, first at {idx.tolist()}: "
                             f"gpu {[hex(v) for v in gc[tuple(idx.T)].tolist()]} "
                             f"oracle {[hex(v) for v in rc[tuple(idx.T)].tolist()]}")


def swiglu_bound(c_ref):
    """The bound on |h_gpu - silu(g) u| that follows from the GEMM tolerance on the
    stacked accumulators c_ref = [g | u] [M][2F] (bias included)."""
    f = c_ref.shape[1] // 2
    g, u = c_ref[:, :f], c_ref[:, f:]
    tg = REL_TOL * np.abs(g) + RMS_TOL * np.sqrt(np.mean(g * g))
    tu = REL_TOL * np.abs(u) + RMS_TOL * np.sqrt(np.mean(u * u))
    ref = O.silu(g) * u
    return SILU_LIP * tg * (np.abs(u) + tu) + np.abs(O.silu(g)) * tu + 1e-6 * np.abs(ref) + 1e-30


def assert_swiglu_close(h_gpu, c_ref, what):
    """h_gpu [M][F] against the oracle's stacked accumulators c_ref [M][2F] (bias included)."""
    f = c_ref.shape[1] // 2
    ref = O.silu(c_ref[:, :f]) * c_ref[:, f:]
    bound = swiglu_bound(c_ref)
    err = np.abs(np.asarray(h_gpu, np.float64) - ref)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (f"{what}: {len(bad)} of {err.size} outside, first {bad[:4].tolist()}, "
                           f"worst ratio {float((err / bound).max()):.3g}")
    return float((err / bound).max())


def graph_capture(fn):
    """Capture fn() into a CUDA graph (after one warm-up run on the capture stream)."""
    import torch

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()   # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    return g


def graph_replays_match(lib, fn_into, make_input, x_buf, y_buf, n=3):
    """fn_into(x, y) runs the path from x into y; compares graph replays with eager calls."""
    import torch

    g = graph_capture(lambda: fn_into(x_buf, y_buf))
    for i in range(n):
        x_new = make_input(100 + i)
        x_buf.copy_(x_new)
        g.replay()
        torch.cuda.synchronize()
        y_eager = torch.empty_like(y_buf)
        fn_into(x_new, y_eager)
        torch.cuda.synchronize()
        assert torch.equal(y_buf, y_eager), f"replay {i} differs from the eager call"
    assert lib.mx_device_error() == 0


def near_rounding_boundary(v, tol) -> np.ndarray:
    """Per element of v (fp32 values about to be MXFP6-encoded, [rows][K]): True where
    some value within `tol` (same shape, >= 0) of v could encode differently -- a
    rounding boundary between two E2M3 codes (the midpoint of adjacent magnitudes at
    the block's scale, or zero, where the sign bit changes) lies within tol, or the
    block's amax could fall on the other side of a power of two (the shared exponent
    could change, moving every code of the block). Two encoders whose inputs differ
    by at most tol can only disagree on such elements, which bounds the number of
    legitimate code differences."""
    v = np.asarray(v, dtype=np.float64)
    tol = np.broadcast_to(np.asarray(tol, dtype=np.float64), v.shape)
    rows, k = v.shape
    vb = np.abs(v).reshape(rows, k // O.BLOCK, O.BLOCK)
    tb = tol.reshape(rows, k // O.BLOCK, O.BLOCK)
    amax = vb.max(axis=-1)
    # the other encoder's amax lies in [max(|v| - t), max(|v| + t)]
    lo = np.maximum((vb - tb).max(axis=-1), np.finfo(np.float64).tiny)
    hi = (vb + tb).max(axis=-1)
    near_scale = np.floor(np.log2(lo)) != np.floor(np.log2(hi))
    s = O.shared_exponent(amax).astype(np.float64)
    t = vb * np.exp2(-s)[..., None]
    tt = tb * np.exp2(-s)[..., None]
    mags = np.unique(np.abs(np.asarray(O.E2M3_TABLE, dtype=np.float64)))
    mids = (mags[:-1] + mags[1:]) / 2.0
    j = np.clip(np.searchsorted(mids, t), 1, len(mids) - 1)
    dist = np.minimum(np.minimum(np.abs(t - mids[j - 1]), np.abs(t - mids[j])), t)
    near = (dist <= tt) | near_scale[..., None]
    return near.reshape(rows, k)


def requant_flip_report(gpu_codes, gpu_scales, ref_codes, ref_scales, ref_values, tol) -> dict:
    """Differences between the GPU's MXFP6 encoding and an independent oracle's of
    the same rows: differing codes (elements of blocks whose scales differ count as
    differing), rows touched, and the derived bound -- the number of elements near a
    rounding boundary of the oracle's values within the tolerance that the two
    pre-quantization values were held to. Asserts the differences stay within it."""
    gc, rc = np.asarray(gpu_codes), np.asarray(ref_codes)
    gs, rs = np.asarray(gpu_scales), np.asarray(ref_scales)
    scale_diff = np.repeat(gs != rs, O.BLOCK, axis=1)
    differ = (gc != rc) | scale_diff
    # the oracle encodes its fp64 values rounded to fp32: half an fp32 ulp more
    ref = np.asarray(ref_values, dtype=np.float64)
    near = near_rounding_boundary(ref, np.asarray(tol, dtype=np.float64) + 2.0 ** -24 * np.abs(ref))
    rep = {"elements": int(differ.size), "differing": int(differ.sum()), "near_boundary": int(near.sum()),
           "differing_not_near": int((differ & ~near).sum()), "rows_touched": int(differ.any(axis=1).sum()),
           "rows": int(differ.shape[0])}
    assert rep["differing_not_near"] == 0, f"codes differ away from any rounding boundary: {rep}"
    return rep, differ
