"""Python binding of the GB300 MXFP6 MLP library (C ABI: include/mx.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. The library is
loaded from this package's ``_lib/libmxfp6.so`` (built by ``_build.build()``);
if it is missing, every call raises -- there is no fallback.

Entry points keep the C names:

* ``mx_quantize(x)`` -- BF16 [rows][K] -> (codes uint8 [rows][3K/4], tiled scales uint8)
* ``mx_gemm(a, b, bias, epilogue)`` -- block-scaled MXFP6 GEMM with a fused epilogue
* ``mx_mlp(x, w1, b1, w2, b2)`` -- quantize -> up-proj + GELU + requant -> down-proj
* ``mx_gated_mlp(x, wgu, bgu, w2, b2)`` -- the same with a SwiGLU up-projection on the
  stacked [W_g; W_u] weight (``mx_quantize_stacked`` builds it)
* ``mx_gemm_gate_residual(a, b, bias, gate, residual)`` -- residual + gate * (A B^T + bias)
* ``mx_scales_to_plain`` / ``mx_scales_from_plain`` -- host-side scale layout helpers
"""

from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np

from . import _build

__all__ = [
    "MxError",
    "MX_EPI_BIAS_BF16",
    "MX_EPI_BIAS_GELU_MXFP6",
    "MX_EPI_BIAS_SWIGLU_MXFP6",
    "MX_EPI_GATE_RESIDUAL_BF16",
    "MxTensor",
    "load",
    "library_path",
    "mx_codes_bytes",
    "mx_scales_bytes",
    "mx_mlp_workspace_bytes",
    "mx_gemm_workspace_bytes",
    "mx_gemm_launch_plan",
    "mx_gemm_workspace",
    "MX_GEMM_WORKSPACE_COUNTER_BYTES",
    "mx_quantize",
    "mx_quantize_rmsnorm_modulate",
    "mx_quantize_stacked",
    "mx_gemm",
    "mx_gemm_gate_residual",
    "mx_quantize_gemm",
    "mx_quantize_gemm_workspace_bytes",
    "mx_quantize_gemm_xq",
    "mx_mlp",
    "mx_mlp_noalloc",
    "mx_gated_mlp",
    "mx_dit_mlp_block",
    "MX_ACT_GELU_TANH",
    "MX_ACT_SWIGLU",
    "mx_status_string",
    "mx_scales_to_plain",
    "mx_scales_from_plain",
    "mx_device_error",
    "mx_selftest_wait_timeout",
    "mx_version",
    "EXPORTED_SYMBOLS",
]

MX_EPI_BIAS_BF16 = 0
MX_EPI_BIAS_GELU_MXFP6 = 1
MX_EPI_BIAS_SWIGLU_MXFP6 = 2
MX_EPI_GATE_RESIDUAL_BF16 = 3
MX_ACT_GELU_TANH = 0
MX_ACT_SWIGLU = 1
MX_GEMM_WORKSPACE_COUNTER_BYTES = 10240

EXPORTED_SYMBOLS = (
    "mx_codes_bytes",
    "mx_scales_bytes",
    "mx_quantize",
    "mx_gemm",
    "mx_mlp_workspace_bytes",
    "mx_mlp",
    "mx_status_string",
    "mx_scales_to_plain",
    "mx_scales_from_plain",
    "mx_device_error",
    "mx_selftest_wait_timeout",
    "mx_version",
    "mx_mlp_noalloc",
    "mx_gemm_gate_residual",
    "mx_gated_mlp",
    "mx_quantize_rmsnorm_modulate",
    "mx_dit_mlp_block",
    "mx_gemm_workspace_bytes",
    "mx_gemm_launch_plan",
    "mx_quantize_stacked",
    "mx_quantize_gemm_workspace_bytes",
    "mx_quantize_gemm",
)

_lib = None
_lock = threading.Lock()


class MxError(RuntimeError):
    """A library call returned a status other than MX_OK."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {mx_status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load libmxfp6.so and declare its signatures. Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the MXFP6 CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()'); there is no CPU fallback")
        lib = ctypes.CDLL(path)
        vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        sigs = {
            "mx_codes_bytes": (sz, [i64, i64]),
            "mx_scales_bytes": (sz, [i64, i64]),
            "mx_quantize": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, vp]),
            "mx_quantize_stacked": (ctypes.c_int, [ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64),
                                                   ctypes.c_int, i64, vp, vp, vp]),
            "mx_gemm": (ctypes.c_int, [vp, vp, vp, vp, vp, i64, i64, i64, ctypes.c_int, vp, vp, vp, vp, sz, vp]),
            "mx_gemm_workspace_bytes": (sz, [i64, i64, i64]),
            "mx_gemm_launch_plan": (ctypes.c_int, [i64, i64, i64, sz, ctypes.POINTER(ctypes.c_int),
                                                   ctypes.POINTER(ctypes.c_int)]),
            "mx_mlp_workspace_bytes": (sz, [i64, i64, i64]),
            "mx_mlp": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "mx_mlp_noalloc": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp]),
            "mx_gated_mlp": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
            "mx_gemm_gate_residual": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp, vp, sz, vp]),
            "mx_quantize_gemm_workspace_bytes": (sz, [i64, i64]),
            "mx_quantize_gemm": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, vp, i64, ctypes.c_int, vp, vp, vp, vp,
                                                vp, sz, vp]),
            "mx_quantize_rmsnorm_modulate": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, ctypes.c_float, vp, vp, vp,
                                                            vp]),
            "mx_dit_mlp_block": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, vp, ctypes.c_float, ctypes.c_int, vp, vp,
                                                vp, vp, vp, vp, vp, vp, sz, vp]),
            "mx_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "mx_scales_to_plain": (ctypes.c_int, [vp, vp, i64, i64]),
            "mx_scales_from_plain": (ctypes.c_int, [vp, vp, i64, i64]),
            "mx_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint), ctypes.c_int]),
            "mx_selftest_wait_timeout": (ctypes.c_int, [vp]),
            "mx_version": (ctypes.c_int, []),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, where: str) -> None:
    if status != 0:
        raise MxError(status, where)


def mx_status_string(status: int) -> str:
    return load().mx_status_string(int(status)).decode()


def mx_version() -> int:
    return load().mx_version()


def mx_codes_bytes(rows: int, k: int) -> int:
    return load().mx_codes_bytes(rows, k)


def mx_scales_bytes(rows: int, k: int) -> int:
    return load().mx_scales_bytes(rows, k)


def mx_mlp_workspace_bytes(m: int, d: int, ff: int) -> int:
    return load().mx_mlp_workspace_bytes(m, d, ff)


def mx_gemm_workspace_bytes(m: int, n: int, k: int) -> int:
    """Bytes of the split-tail workspace of an [m][k] x [n][k]^T GEMM (0: it never splits)."""
    return load().mx_gemm_workspace_bytes(m, n, k)


def mx_gemm_launch_plan(m: int, n: int, k: int, workspace_bytes: int | None = None) -> tuple[int, int]:
    """(CTA pairs launched, leading tiles divided along K) for this GEMM shape on the
    current device, given a workspace of ``workspace_bytes`` (default: the full size)."""
    lib = load()
    if workspace_bytes is None:
        workspace_bytes = lib.mx_gemm_workspace_bytes(m, n, k)
    pairs, split = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib.mx_gemm_launch_plan(m, n, k, int(workspace_bytes), ctypes.byref(pairs), ctypes.byref(split)),
           "mx_gemm_launch_plan")
    return pairs.value, split.value


def mx_gemm_workspace(m: int, n: int, k: int, device=None, stream=None):
    """A split-tail workspace for [m][k] x [n][k]^T GEMMs, its arrival counters zeroed
    on ``stream`` (reusable: every GEMM leaves them zero again), or None when the
    shape never splits."""
    torch = _torch()
    need = load().mx_gemm_workspace_bytes(m, n, k)
    if need == 0:
        return None
    dev = device if device is not None else "cuda"
    if stream is None:
        return torch.zeros(int(need), dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):   # allocated and zeroed in the order of the GEMM's stream
        return torch.zeros(int(need), dtype=torch.uint8, device=dev)


def _split_workspace(workspace, split: bool, m: int, n: int, k: int, device, stream):
    """(workspace tensor or None, pointer, bytes): the caller's, a new one, or none."""
    if workspace is not None:
        _on(workspace, device, "workspace", _torch().uint8)
        return workspace, _ptr(workspace), workspace.numel()
    if not split:
        return None, None, 0
    ws = mx_gemm_workspace(m, n, k, device, stream if hasattr(stream, "cuda_stream") else None)
    if ws is None:
        return None, None, 0
    return ws, _ptr(ws), ws.numel()


def _torch():
    import torch

    return torch


def _stream_handle(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


@dataclass
class MxTensor:
    """An MXFP6 matrix on the device: packed codes [rows][3K/4] and tiled scales."""

    codes: "object"   # torch.uint8 [rows, 3K/4]
    scales: "object"  # torch.uint8 [mx_scales_bytes(rows, K)]
    rows: int
    k: int


def _empty_u8(n: int, device):
    return _torch().empty(int(n), dtype=_torch().uint8, device=device)


def _cuda_device(t, name: str):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.device


def _on(t, dev, name: str, dtype, numel: int | None = None, exact: bool = False):
    """Refuse a tensor that is not a contiguous CUDA tensor of ``dtype`` on ``dev``
    holding at least (``exact``: exactly) ``numel`` elements. The library takes raw
    pointers and sizes, so a short, misplaced or strided buffer would be read or
    written out of bounds on the device; it is refused here instead."""
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.device != dev:
        raise ValueError(f"{name} must be a CUDA tensor on {dev}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, not {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and (t.numel() != numel if exact else t.numel() < numel):
        raise ValueError(f"{name} holds {t.numel()} elements; {'exactly ' if exact else ''}{numel} needed")
    return t


def _vec(t, dev, name: str, n: int):
    """An optional BF16 vector of exactly n elements on dev."""
    return None if t is None else _on(t, dev, name, _torch().bfloat16, n, exact=True)


def _mx_on(t, dev, name: str, rows: int, k: int):
    """An MxTensor of [rows][k] whose codes and scales are uint8 buffers on dev of
    at least the library's sizes."""
    lib = load()
    if not isinstance(t, MxTensor) or t.rows != rows or t.k != k:
        raise ValueError(f"{name} must be an MxTensor of [{rows}][{k}]")
    _on(t.codes, dev, f"{name}.codes", _torch().uint8, lib.mx_codes_bytes(rows, k))
    _on(t.scales, dev, f"{name}.scales", _torch().uint8, lib.mx_scales_bytes(rows, k))
    return t


def _bf16_matrix(x, name: str, dev=None):
    """A contiguous CUDA bfloat16 [rows][K] tensor (on dev when given)."""
    torch = _torch()
    if not isinstance(x, torch.Tensor) or x.dim() != 2:
        raise ValueError(f"{name} must be a bfloat16 [rows][K] CUDA tensor")
    return _on(x, dev if dev is not None else _cuda_device(x, name), name, torch.bfloat16)


def mx_quantize(x, out: MxTensor | None = None, stream=None) -> MxTensor:
    """K1: quantize a BF16 [rows][K] CUDA tensor (row stride may exceed K) to MXFP6."""
    torch = _torch()
    lib = load()
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("mx_quantize wants a CUDA bfloat16 [rows][K] tensor with unit column stride")
    rows, k = x.shape
    if out is None:
        codes = _empty_u8(lib.mx_codes_bytes(rows, k), x.device).view(rows, -1) if rows else \
            _empty_u8(0, x.device).view(0, k // 4 * 3)
        out = MxTensor(codes, _empty_u8(lib.mx_scales_bytes(rows, k), x.device), rows, k)
    _mx_on(out, x.device, "out", rows, k)
    st = lib.mx_quantize(_ptr(x), rows, k, x.stride(0), _ptr(out.codes), _ptr(out.scales), _stream_handle(stream))
    _check(st, "mx_quantize")
    return out


def mx_quantize_rmsnorm_modulate(x, shift=None, scale=None, eps: float = 1e-6, out: MxTensor | None = None,
                                 debug_y=None, stream=None) -> MxTensor:
    """RMSNorm + modulation + K1: MXFP6(x / rms(x) * (1 + scale) + shift) of a BF16 [rows][K] tensor."""
    torch = _torch()
    lib = load()
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError("mx_quantize_rmsnorm_modulate wants a CUDA bfloat16 [rows][K] tensor")
    rows, k = x.shape
    _vec(shift, x.device, "shift", k)
    _vec(scale, x.device, "scale", k)
    if debug_y is not None:
        _on(debug_y, x.device, "debug_y", torch.float32, rows * k)
    if out is None:
        codes = _empty_u8(lib.mx_codes_bytes(rows, k), x.device).view(rows, -1) if rows else \
            _empty_u8(0, x.device).view(0, k // 4 * 3)
        out = MxTensor(codes, _empty_u8(lib.mx_scales_bytes(rows, k), x.device), rows, k)
    _mx_on(out, x.device, "out", rows, k)
    st = lib.mx_quantize_rmsnorm_modulate(_ptr(x), rows, k, x.stride(0), _ptr(shift), _ptr(scale), float(eps),
                                          _ptr(out.codes), _ptr(out.scales), _ptr(debug_y), _stream_handle(stream))
    _check(st, "mx_quantize_rmsnorm_modulate")
    return out


def mx_quantize_stacked(parts, stream=None) -> MxTensor:
    """Quantize BF16 matrices [R_i][K] into one stacked MXFP6 tensor [sum R_i][K]
    (the C entry point mx_quantize_stacked).

    Rows are quantized independently, so the result is the concatenation of the
    parts' MXFP6 forms; every part but the last needs R_i % 128 == 0 (its tiled
    scales then end on an atom boundary). Builds the [W_g; W_u] weight of
    mx_gated_mlp and the stacked query/key/value/gate weight of one projection.
    """
    torch = _torch()
    lib = load()
    if not parts:
        raise ValueError("mx_quantize_stacked needs at least one part")
    dev = parts[0].device
    for i, p in enumerate(parts):
        if p.dtype != torch.bfloat16 or p.dim() != 2 or not p.is_cuda or p.stride(1) != 1 or p.device != dev:
            raise ValueError(f"part {i} must be a CUDA bfloat16 [rows][K] tensor with unit column stride on {dev}")
    k = parts[0].shape[1]
    rows = sum(int(p.shape[0]) for p in parts)
    if any(p.shape[1] != k for p in parts):
        raise ValueError("parts need equal K")
    codes = _empty_u8(lib.mx_codes_bytes(rows, k), dev).view(rows, -1)
    scales = _empty_u8(lib.mx_scales_bytes(rows, k), dev)
    n = len(parts)
    ptrs = (ctypes.c_void_p * n)(*[_ptr(p) for p in parts])
    prow = (ctypes.c_int64 * n)(*[int(p.shape[0]) for p in parts])
    lds = (ctypes.c_int64 * n)(*[int(p.stride(0)) for p in parts])
    st = lib.mx_quantize_stacked(ptrs, prow, lds, n, k, _ptr(codes), _ptr(scales), _stream_handle(stream))
    _check(st, "mx_quantize_stacked")
    return MxTensor(codes, scales, rows, k)


def mx_gemm(a: MxTensor, b: MxTensor, bias=None, epilogue: int = MX_EPI_BIAS_BF16, out=None,
            debug_prequant=None, stream=None, workspace=None, split: bool = True):
    """K2/K3: a [M][K] x b [N][K]^T on MXFP6 with the fused epilogue.

    Returns a BF16 [M][N] tensor (MX_EPI_BIAS_BF16) or an MxTensor of [M][W]
    (W = N for MX_EPI_BIAS_GELU_MXFP6, N/2 for MX_EPI_BIAS_SWIGLU_MXFP6, where b
    is the stacked [W_g; W_u]). ``debug_prequant`` (fp32 [M][W]) receives the
    activation output the requantization rounds. ``workspace`` (from
    mx_gemm_workspace, or uint8 with its first MX_GEMM_WORKSPACE_COUNTER_BYTES zero)
    is the split-tail scratch; without one, a new one is taken unless ``split`` is
    False (no split tail).
    """
    torch = _torch()
    lib = load()
    if a.k != b.k:
        raise ValueError("inner dimensions differ")
    m, n, k = a.rows, b.rows, a.k
    dev = _cuda_device(a.codes, "a.codes")
    _mx_on(a, dev, "a", m, k)
    _mx_on(b, dev, "b", n, k)
    _vec(bias, dev, "bias", n)
    if epilogue == MX_EPI_BIAS_BF16:
        if out is None:
            out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        _on(out, dev, "out", torch.bfloat16, m * n)
        out_ptr, out_sc = _ptr(out), None
    else:
        w = n // 2 if epilogue == MX_EPI_BIAS_SWIGLU_MXFP6 else n
        if out is None:
            out = MxTensor(_empty_u8(lib.mx_codes_bytes(m, w), dev).view(m, -1) if m else
                           _empty_u8(0, dev).view(0, w // 4 * 3),
                           _empty_u8(lib.mx_scales_bytes(m, w), dev), m, w)
        _mx_on(out, dev, "out", m, w)
        if debug_prequant is not None:
            _on(debug_prequant, dev, "debug_prequant", torch.float32, m * w)
        out_ptr, out_sc = _ptr(out.codes), _ptr(out.scales)
    ws, ws_ptr, ws_bytes = _split_workspace(workspace, split, m, n, k, dev, stream)
    st = lib.mx_gemm(_ptr(a.codes), _ptr(a.scales), _ptr(b.codes), _ptr(b.scales), _ptr(bias), m, n, k,
                     int(epilogue), out_ptr, out_sc, _ptr(debug_prequant), ws_ptr, ws_bytes, _stream_handle(stream))
    _check(st, "mx_gemm")
    return out


def mx_mlp(x, w1: MxTensor, b1, w2: MxTensor, b2, y=None, workspace=None, stream=None):
    """K1 + K3 + K2: y = bf16(MXFP6(gelu(MXFP6(x) W1^T + b1)) W2^T + b2)."""
    torch = _torch()
    lib = load()
    dev = _bf16_matrix(x, "x").device
    m, d = x.shape
    ff = w1.rows
    if w1.k != d or w2.rows != d or w2.k != ff:
        raise ValueError("weight shapes do not match x")
    _mx_on(w1, dev, "w1", ff, d)
    _mx_on(w2, dev, "w2", d, ff)
    _vec(b1, dev, "b1", ff)
    _vec(b2, dev, "b2", d)
    if y is None:
        y = torch.empty((m, d), dtype=torch.bfloat16, device=x.device)
    _on(y, dev, "y", torch.bfloat16, m * d)
    need = lib.mx_mlp_workspace_bytes(m, d, ff)
    if workspace is None:
        workspace = _empty_u8(max(need, 256), x.device)
    _on(workspace, dev, "workspace", torch.uint8)
    st = lib.mx_mlp(_ptr(x), m, d, ff, _ptr(w1.codes), _ptr(w1.scales), _ptr(b1), _ptr(w2.codes),
                    _ptr(w2.scales), _ptr(b2), _ptr(y), _ptr(workspace), workspace.numel(),
                    _stream_handle(stream))
    _check(st, "mx_mlp")
    return y


def mx_mlp_noalloc(x, w1: MxTensor, b1, w2: MxTensor, b2, y=None, stream=None):
    """mx_mlp through the library's static scratch (mx_mlp_noalloc): no workspace is
    allocated for the call. For callers that must not allocate device memory; sizes
    beyond the scratch raise MxError(MX_ERR_WORKSPACE_TOO_SMALL). Calls that overlap
    on the GPU share the scratch and race: order them on one stream."""
    torch = _torch()
    lib = load()
    dev = _bf16_matrix(x, "x").device
    m, d = x.shape
    ff = w1.rows
    if w1.k != d or w2.rows != d or w2.k != ff:
        raise ValueError("weight shapes do not match x")
    _mx_on(w1, dev, "w1", ff, d)
    _mx_on(w2, dev, "w2", d, ff)
    _vec(b1, dev, "b1", ff)
    _vec(b2, dev, "b2", d)
    if y is None:
        y = torch.empty((m, d), dtype=torch.bfloat16, device=x.device)
    _on(y, dev, "y", torch.bfloat16, m * d)
    st = lib.mx_mlp_noalloc(_ptr(x), m, d, ff, _ptr(w1.codes), _ptr(w1.scales), _ptr(b1), _ptr(w2.codes),
                            _ptr(w2.scales), _ptr(b2), _ptr(y), _stream_handle(stream))
    _check(st, "mx_mlp_noalloc")
    return y


def mx_gemm_gate_residual(a: MxTensor, b: MxTensor, bias, gate, residual, out=None, stream=None, workspace=None,
                          split: bool = True):
    """out = bf16(residual + gate * (a b^T + bias)); out may be residual (in place).
    ``workspace`` / ``split``: the split-tail scratch, as mx_gemm."""
    torch = _torch()
    lib = load()
    if a.k != b.k:
        raise ValueError("inner dimensions differ")
    m, n, k = a.rows, b.rows, a.k
    dev = _cuda_device(residual, "residual")
    if tuple(residual.shape) != (m, n):
        raise ValueError("residual must be a contiguous bfloat16 [M][N] tensor")
    _on(residual, dev, "residual", torch.bfloat16, m * n)
    _mx_on(a, dev, "a", m, k)
    _mx_on(b, dev, "b", n, k)
    _vec(bias, dev, "bias", n)
    _vec(gate, dev, "gate", n)
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=residual.device)
    _on(out, dev, "out", torch.bfloat16, m * n)
    ws, ws_ptr, ws_bytes = _split_workspace(workspace, split, m, n, k, residual.device, stream)
    st = lib.mx_gemm_gate_residual(_ptr(a.codes), _ptr(a.scales), _ptr(b.codes), _ptr(b.scales), _ptr(bias),
                                   _ptr(gate), _ptr(residual), m, n, k, _ptr(out), ws_ptr, ws_bytes,
                                   _stream_handle(stream))
    _check(st, "mx_gemm_gate_residual")
    return out


def mx_quantize_gemm_workspace_bytes(m: int, k: int) -> int:
    return load().mx_quantize_gemm_workspace_bytes(m, k)


def mx_quantize_gemm(x, b: MxTensor, bias=None, epilogue: int = MX_EPI_BIAS_BF16, gate=None, residual=None,
                     out=None, workspace=None, stream=None):
    """mx_quantize(x) and the GEMM on it in one pass: the GEMM quantizes most rows of
    the BF16 activations itself while its main loop runs. ``epilogue`` as mx_gemm, or
    MX_EPI_GATE_RESIDUAL_BF16 with ``gate`` / ``residual`` as mx_gemm_gate_residual
    (out may be residual). Returns out (BF16 tensor or MxTensor); ``workspace`` (uint8,
    mx_quantize_gemm_workspace_bytes) then holds MXFP6(x): see mx_quantize_gemm_xq."""
    torch = _torch()
    lib = load()
    dev = _cuda_device(x, "x")
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a CUDA bfloat16 [M][K] tensor with unit column stride")
    m, k = x.shape
    n = b.rows
    if b.k != k:
        raise ValueError("inner dimensions differ")
    _mx_on(b, dev, "b", n, k)
    _vec(bias, dev, "bias", n)
    out_scales = None
    if epilogue == MX_EPI_GATE_RESIDUAL_BF16:
        if residual is None or tuple(residual.shape) != (m, n):
            raise ValueError("residual must be a contiguous bfloat16 [M][N] tensor")
        _on(residual, dev, "residual", torch.bfloat16, m * n)
        _vec(gate, dev, "gate", n)
    if epilogue in (MX_EPI_BIAS_BF16, MX_EPI_GATE_RESIDUAL_BF16):
        if out is None:
            out = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
        _on(out, dev, "out", torch.bfloat16, m * n)
        out_ptr = _ptr(out)
    else:
        w = n // 2 if epilogue == MX_EPI_BIAS_SWIGLU_MXFP6 else n
        if out is None:
            out = MxTensor(_empty_u8(lib.mx_codes_bytes(m, w), dev).view(m, -1) if m else
                           _empty_u8(0, dev).view(0, w // 4 * 3),
                           _empty_u8(lib.mx_scales_bytes(m, w), dev), m, w)
        _mx_on(out, dev, "out", m, w)
        out_ptr, out_scales = _ptr(out.codes), _ptr(out.scales)
    if workspace is None:
        workspace = _empty_u8(max(lib.mx_quantize_gemm_workspace_bytes(m, k), 256), dev)
    _on(workspace, dev, "workspace", torch.uint8)
    st = lib.mx_quantize_gemm(_ptr(x), m, k, x.stride(0), _ptr(b.codes), _ptr(b.scales), _ptr(bias), n,
                              int(epilogue), _ptr(gate), _ptr(residual), out_ptr, out_scales, _ptr(workspace),
                              workspace.numel(), _stream_handle(stream))
    _check(st, "mx_quantize_gemm")
    return out


def mx_quantize_gemm_xq(workspace, m: int, k: int) -> MxTensor:
    """The MXFP6(x) that mx_quantize_gemm left in its workspace, as views of it."""
    lib = load()
    cb, sb = lib.mx_codes_bytes(m, k), lib.mx_scales_bytes(m, k)
    off = -(-cb // 256) * 256
    return MxTensor(workspace[:cb].view(m, -1) if m else workspace[:0].view(0, k // 4 * 3),
                    workspace[off:off + sb], m, k)


def mx_gated_mlp(x, wgu: MxTensor, bgu, w2: MxTensor, b2, y=None, workspace=None, stream=None):
    """K1 + SwiGLU up-projection + K2: y = bf16(MXFP6(silu(g) * u) W2^T + b2),
    [g | u] = MXFP6(x) [W_g; W_u]^T + [b_g; b_u]."""
    torch = _torch()
    lib = load()
    dev = _bf16_matrix(x, "x").device
    m, d = x.shape
    ff = wgu.rows // 2
    if wgu.k != d or wgu.rows != 2 * ff or w2.rows != d or w2.k != ff:
        raise ValueError("weight shapes do not match x")
    _mx_on(wgu, dev, "wgu", 2 * ff, d)
    _mx_on(w2, dev, "w2", d, ff)
    _vec(bgu, dev, "bgu", 2 * ff)
    _vec(b2, dev, "b2", d)
    if y is None:
        y = torch.empty((m, d), dtype=torch.bfloat16, device=x.device)
    _on(y, dev, "y", torch.bfloat16, m * d)
    need = lib.mx_mlp_workspace_bytes(m, d, ff)
    if workspace is None:
        workspace = _empty_u8(max(need, 256), x.device)
    _on(workspace, dev, "workspace", torch.uint8)
    st = lib.mx_gated_mlp(_ptr(x), m, d, ff, _ptr(wgu.codes), _ptr(wgu.scales), _ptr(bgu), _ptr(w2.codes),
                          _ptr(w2.scales), _ptr(b2), _ptr(y), _ptr(workspace), workspace.numel(),
                          _stream_handle(stream))
    _check(st, "mx_gated_mlp")
    return y


def mx_dit_mlp_block(x, shift, scale, gate, w_up: MxTensor, b_up, w2: MxTensor, b2, eps: float = 1e-6,
                     activation: int = MX_ACT_GELU_TANH, y=None, workspace=None, stream=None):
    """y = x + gate * MLP(MXFP6(rmsnorm(x) * (1 + scale) + shift)); y may be x (in place)."""
    torch = _torch()
    lib = load()
    dev = _bf16_matrix(x, "x").device
    m, d = x.shape
    ff = w2.k
    rows_up = 2 * ff if activation == MX_ACT_SWIGLU else ff
    if w_up.k != d or w_up.rows != rows_up or w2.rows != d:
        raise ValueError("weight shapes do not match x")
    _mx_on(w_up, dev, "w_up", rows_up, d)
    _mx_on(w2, dev, "w2", d, ff)
    for name, v, n in (("shift", shift, d), ("scale", scale, d), ("gate", gate, d), ("b_up", b_up, rows_up),
                       ("b2", b2, d)):
        _vec(v, dev, name, n)
    if y is None:
        y = torch.empty((m, d), dtype=torch.bfloat16, device=x.device)
    _on(y, dev, "y", torch.bfloat16, m * d)
    need = lib.mx_mlp_workspace_bytes(m, d, ff)
    if workspace is None:
        workspace = _empty_u8(max(need, 256), x.device)
    _on(workspace, dev, "workspace", torch.uint8)
    st = lib.mx_dit_mlp_block(_ptr(x), m, d, ff, _ptr(shift), _ptr(scale), _ptr(gate), float(eps), int(activation),
                              _ptr(w_up.codes), _ptr(w_up.scales), _ptr(b_up), _ptr(w2.codes), _ptr(w2.scales),
                              _ptr(b2), _ptr(y), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st, "mx_dit_mlp_block")
    return y


def mx_scales_to_plain(tiled, rows: int, k: int) -> np.ndarray:
    """Host: tiled scale bytes -> plain uint8 [rows][K/32]."""
    lib = load()
    t = np.ascontiguousarray(np.asarray(tiled, dtype=np.uint8).reshape(-1))
    if t.size < lib.mx_scales_bytes(rows, k):
        raise ValueError("tiled scale buffer too small")
    out = np.empty((rows, k // 32), dtype=np.uint8)
    _check(lib.mx_scales_to_plain(t.ctypes.data, out.ctypes.data, rows, k), "mx_scales_to_plain")
    return out


def mx_scales_from_plain(plain, rows: int, k: int) -> np.ndarray:
    """Host: plain uint8 [rows][K/32] -> tiled scale bytes (padding rows zero)."""
    lib = load()
    p = np.ascontiguousarray(np.asarray(plain, dtype=np.uint8).reshape(rows, k // 32))
    out = np.empty(lib.mx_scales_bytes(rows, k), dtype=np.uint8)
    _check(lib.mx_scales_from_plain(p.ctypes.data, out.ctypes.data, rows, k), "mx_scales_from_plain")
    return out


def mx_selftest_wait_timeout(stream=None) -> None:
    """Launch the failure-detection self test (a bounded wait that must run out)."""
    _check(load().mx_selftest_wait_timeout(_stream_handle(stream)), "mx_selftest_wait_timeout")


def mx_device_error(clear: bool = True) -> int:
    """Synchronize and read the kernels' device error word (0 = no wait ran out)."""
    flags = ctypes.c_uint(0)
    _check(load().mx_device_error(ctypes.byref(flags), int(clear)), "mx_device_error")
    return flags.value
