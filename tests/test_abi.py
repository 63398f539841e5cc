"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, rejects bad arguments on the host before any launch, and its host-side
scale-layout helpers agree with the oracle's independent layout code."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mx.h")

OK, INVALID, SHAPE, MISALIGNED, WS_SMALL, DEVICE, CUDA = range(7)
BF16, GELU, SWIGLU = 0, 1, 2
A32 = 0x10000   # fake, 32-byte aligned device addresses: never dereferenced by validation
A32b = 0x20000
A32c = 0x30000
A32d = 0x40000
A32e = 0x50000


@pytest.fixture(scope="module")
def mx():
    import microscaled_precision_gemm_gb300 as pkg
    from microscaled_precision_gemm_gb300 import _build

    _build.build()
    pkg.load()
    return pkg


@pytest.fixture(scope="module")
def lib(mx):
    return mx.load()


def test_exports_every_declared_symbol(lib, mx):
    text = open(HEADER).read()
    declared = set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(mx_\w+)\s*\(", text, flags=re.M))
    assert declared == set(mx.EXPORTED_SYMBOLS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version_and_status_strings(mx):
    assert mx.mx_version() == 100
    for s in range(7):
        assert mx.mx_status_string(s).startswith("MX_")
    assert mx.mx_status_string(99) == "unknown mx_status"


def test_size_queries(lib):
    assert lib.mx_codes_bytes(128, 256) == 128 * 192
    assert lib.mx_scales_bytes(128, 256) == 128 * 8
    assert lib.mx_scales_bytes(300, 256) == 384 * 8       # rows padded to 128
    assert lib.mx_scales_bytes(0, 256) == 0
    assert lib.mx_codes_bytes(-1, 256) == 0
    ws = lib.mx_mlp_workspace_bytes(20480, 3072, 12288)
    # MXFP6 x and h, then one counter word per 128 rows (160 words, 640 -> 768 bytes)
    need = 20480 * 3072 * 3 // 4 + 20480 * 96 + 20480 * 12288 * 3 // 4 + 20480 * 384 + 768
    assert _mlp_base(lib, 20480, 3072, 12288) == need
    # plus the split-tail region the larger of the two GEMMs needs (here the
    # down-projection; the up-projection's 24 K-steps never split)
    up, down = lib.mx_gemm_workspace_bytes(20480, 2 * 12288, 3072), lib.mx_gemm_workspace_bytes(20480, 3072, 12288)
    assert up == 0 and down > 0
    assert ws == need + max(up, down)


def _mlp_base(lib, M, d, ff):
    """Smallest MLP workspace: MXFP6 x and h and the row-block counters (a 32-bit
    word per 128 rows), each part 256-byte aligned."""
    return sum(-(-n // 256) * 256 for n in (lib.mx_codes_bytes(M, d), lib.mx_scales_bytes(M, d),
                                            lib.mx_codes_bytes(M, ff), lib.mx_scales_bytes(M, ff),
                                            4 * (-(-M // 128))))


def _q(lib, x=A32, rows=128, k=256, ld=256, codes=A32b, scales=A32c):
    return lib.mx_quantize(x, rows, k, ld, codes, scales, None)


def test_quantize_rejects_bad_arguments(lib):
    assert _q(lib, rows=-1) == INVALID
    assert _q(lib, ld=128) == INVALID                  # ld_x < K
    assert _q(lib, k=100, ld=100) == SHAPE             # K % 128
    assert _q(lib, k=0, ld=0) == SHAPE
    assert _q(lib, ld=260) == MISALIGNED               # ld_x % 8
    assert _q(lib, x=None) == INVALID
    assert _q(lib, codes=None) == INVALID
    assert _q(lib, x=A32 + 8) == MISALIGNED
    assert _q(lib, codes=A32b + 16) == MISALIGNED      # codes want 32 bytes
    assert _q(lib, scales=A32c + 4) == MISALIGNED
    assert _q(lib, rows=0, x=None, codes=None, scales=None) == OK   # empty input: no-op


def _g(lib, a=A32, sa=A32b, b=A32c, sb=A32d, bias=None, M=128, N=512, K=256, epi=BF16, out=A32e,
       out_sc=A32, dbg=None, ws=None, wsb=0):
    return lib.mx_gemm(a, sa, b, sb, bias, M, N, K, epi, out, out_sc, dbg, ws, wsb, None)


def test_gemm_rejects_bad_arguments(lib):
    assert _g(lib, epi=7) == INVALID
    assert _g(lib, M=-1) == INVALID
    assert _g(lib, N=384) == SHAPE                     # N % 256
    assert _g(lib, K=96) == SHAPE                      # K % 128
    assert _g(lib, K=0) == SHAPE
    assert _g(lib, M=1 << 31) == SHAPE
    assert _g(lib, a=None) == INVALID
    assert _g(lib, out=None) == INVALID
    assert _g(lib, epi=GELU, out_sc=None) == INVALID
    assert _g(lib, a=A32 + 16) == MISALIGNED
    assert _g(lib, sb=A32d + 8) == MISALIGNED
    assert _g(lib, bias=A32 + 2) == MISALIGNED
    assert _g(lib, epi=GELU, out=A32e + 16) == MISALIGNED
    assert _g(lib, epi=GELU, dbg=A32 + 4) == MISALIGNED
    assert _g(lib, ws=0x100000 + 64, wsb=1 << 26) == MISALIGNED   # the split workspace wants 256 bytes
    assert _g(lib, M=0, a=None, sa=None, b=None, sb=None, out=None) == OK   # empty: no-op
    assert _g(lib, N=0, a=None, sa=None, b=None, sb=None, out=None) == OK


def test_mlp_rejects_bad_arguments(lib):
    args = dict(x=A32, M=256, d=512, ff=1024, w1=A32b, w1s=A32c, b1=None, w2=A32d, w2s=A32e, b2=None,
                y=A32, ws=0x100000, wsb=1 << 30)

    def call(**kw):
        a = dict(args, **kw)
        return lib.mx_mlp(a["x"], a["M"], a["d"], a["ff"], a["w1"], a["w1s"], a["b1"], a["w2"], a["w2s"],
                          a["b2"], a["y"], a["ws"], a["wsb"], None)

    assert call(M=-1) == INVALID
    assert call(d=384) == SHAPE
    assert call(ff=640) == SHAPE
    assert call(x=None) == INVALID
    assert call(ws=0x100000 + 128) == MISALIGNED
    # the smallest workspace holds MXFP6 x and h; the split-tail region after them is optional
    base = _mlp_base(lib, 256, 512, 1024)
    assert lib.mx_mlp_workspace_bytes(256, 512, 1024) == base      # K <= 1024: no split region
    assert lib.mx_mlp_workspace_bytes(256, 4096, 4096) > _mlp_base(lib, 256, 4096, 4096)
    assert call(wsb=base - 1) == WS_SMALL
    assert call(wsb=base) not in (OK, WS_SMALL, INVALID, SHAPE, MISALIGNED)   # valid: stops at the device
    assert call(M=0, x=None, y=None, ws=None) == OK


def test_swiglu_gemm_arguments(lib):
    assert _g(lib, epi=SWIGLU, out_sc=None) == INVALID
    assert _g(lib, epi=SWIGLU, N=384) == SHAPE         # stacked N = 2F needs N % 256
    assert _g(lib, epi=SWIGLU, out=A32e + 16) == MISALIGNED
    assert _g(lib, epi=SWIGLU, dbg=A32 + 4) == MISALIGNED
    assert _g(lib, epi=3) == INVALID                   # the gate/residual epilogue has its own entry point


def _gr(lib, bias=None, gate=None, res=0x200000, M=128, N=512, K=256, out=0x400000):
    return lib.mx_gemm_gate_residual(A32, A32b, A32c, A32d, bias, gate, res, M, N, K, out, None, 0, None)


def test_gate_residual_rejects_bad_arguments(lib):
    assert _gr(lib, res=None) == INVALID
    assert _gr(lib, N=384) == SHAPE
    assert _gr(lib, gate=A32 + 2) == MISALIGNED
    assert _gr(lib, res=0x200000 + 8) == MISALIGNED
    assert _gr(lib, out=0x200000 + 1024) == INVALID    # partial overlap with the residual
    assert _gr(lib, M=0, res=None, out=None) == OK


def test_quantize_gemm_rejects_bad_arguments(lib):
    """mx_quantize_gemm: the quantizer's and the GEMM's rules on the workspace's
    parts, the workspace size, the gate/residual rules, and no overlap of x with
    the output or the workspace -- all on the host, before the device is touched."""
    X, OUT, WS = 0x1000000, 0x2000000, 0x4000000
    need = lib.mx_quantize_gemm_workspace_bytes(128, 256)
    # codes, scales (both 256-aligned), then a counter word per 128 rows
    assert need == 128 * 192 + 128 * 8 + 256

    def call(x=X, M=128, K=256, ld=256, b=A32b, bs=A32c, bias=None, N=512, epi=BF16, gate=None, res=None,
             out=OUT, out_sc=None, ws=WS, wsb=need):
        return lib.mx_quantize_gemm(x, M, K, ld, b, bs, bias, N, epi, gate, res, out, out_sc, ws, wsb, None)

    assert call(epi=4) == INVALID
    assert call(epi=-1) == INVALID
    assert call(M=-1) == INVALID
    assert call(ld=128) == INVALID                   # ld_x < K
    assert call(K=96, ld=96) == SHAPE
    assert call(N=384) == SHAPE
    assert call(ld=260) == MISALIGNED                # row stride % 8
    assert call(x=None) == INVALID
    assert call(x=X + 2) == MISALIGNED
    assert call(b=None) == INVALID
    assert call(out=None) == INVALID
    assert call(epi=GELU) == INVALID                 # MXFP6 output needs its scales
    assert call(ws=None) == INVALID
    assert call(ws=WS + 64) == MISALIGNED
    assert call(wsb=need - 1) == WS_SMALL
    assert call(epi=3) == INVALID                    # the gate/residual epilogue needs a residual
    assert call(epi=3, res=OUT + 8) == MISALIGNED
    assert call(epi=3, res=OUT + 1024) == INVALID    # partial overlap with the output
    assert call(out=X + 4096) == INVALID             # x overlaps the output
    assert call(ws=X - 256) == INVALID               # x overlaps the workspace
    assert call(epi=3, res=WS + 1024, out=WS + 1024 + (1 << 20)) == INVALID   # residual inside the workspace
    assert call(M=0, x=None, b=None, out=None, ws=None) == OK
    assert call(N=0, x=None, b=None, out=None, ws=None) == OK
    for ok in (call(), call(epi=3, res=OUT), call(epi=GELU, out_sc=0x3000000)):
        assert ok not in (OK, WS_SMALL, INVALID, SHAPE, MISALIGNED)   # valid: stops at the device


def test_gated_mlp_rejects_bad_arguments(lib):
    def call(M=256, d=512, ff=1024, ws=0x100000, wsb=1 << 30, x=A32):
        return lib.mx_gated_mlp(x, M, d, ff, A32b, A32c, None, A32d, A32e, None, A32, ws, wsb, None)

    assert call(M=-1) == INVALID
    assert call(d=384) == SHAPE
    assert call(ff=192) == SHAPE                       # ff % 128
    assert call(x=None) == INVALID
    assert call(wsb=_mlp_base(lib, 256, 512, 1024) - 1) == WS_SMALL
    assert call(M=0, x=None) == OK


def _nq(lib, x=A32, rows=128, k=256, ld=256, shift=None, scale=None, eps=1e-6, codes=A32b, scales=A32c, dbg=None):
    return lib.mx_quantize_rmsnorm_modulate(x, rows, k, ld, shift, scale, eps, codes, scales, dbg, None)


def test_norm_quantize_rejects_bad_arguments(lib):
    assert _nq(lib, eps=-1.0) == INVALID
    assert _nq(lib, eps=float("nan")) == INVALID
    assert _nq(lib, eps=float("inf")) == INVALID
    assert _nq(lib, k=8320, ld=8320) == SHAPE          # above the 8192 columns one CTA holds
    assert _nq(lib, k=100, ld=100) == SHAPE
    assert _nq(lib, shift=A32 + 8) == MISALIGNED
    assert _nq(lib, scale=A32 + 2) == MISALIGNED
    assert _nq(lib, dbg=A32 + 4) == MISALIGNED
    assert _nq(lib, x=None) == INVALID
    assert _nq(lib, rows=0, x=None, codes=None, scales=None) == OK


def test_dit_block_rejects_bad_arguments(lib):
    def call(M=256, d=512, ff=1024, act=0, x=A32, y=0x800000, ws=0x100000, wsb=1 << 30, eps=1e-6, gate=None):
        return lib.mx_dit_mlp_block(x, M, d, ff, None, None, gate, eps, act, A32b, A32c, None, A32d, A32e, None, y,
                                    ws, wsb, None)

    assert call(act=2) == INVALID
    assert call(M=-1) == INVALID
    assert call(d=384) == SHAPE
    assert call(ff=384, act=0) == SHAPE                # GELU: ff is N of the up-projection
    assert call(d=8448) == SHAPE                       # fused quantizer holds at most 8192 columns
    assert call(eps=-1.0) == INVALID
    assert call(y=A32 + 512) == INVALID                # partial overlap of y and x
    assert call(gate=A32 + 2) == MISALIGNED
    assert call(wsb=_mlp_base(lib, 256, 512, 1024) - 1) == WS_SMALL
    assert call(M=0, x=None, y=None) == OK


def test_valid_call_without_gpu_fails_loudly(lib):
    """A well-formed call must reach the device check and fail there: no CPU fallback."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _q(lib) in (CUDA, DEVICE)
    assert _g(lib) in (CUDA, DEVICE)
    assert _g(lib, epi=SWIGLU) in (CUDA, DEVICE)
    assert _gr(lib) in (CUDA, DEVICE)
    assert _nq(lib) in (CUDA, DEVICE)


def test_host_scale_layout_matches_oracle(mx):
    rng = np.random.default_rng(11)
    for rows, k in [(128, 256), (300, 384), (1, 128), (256, 1024)]:
        plain = rng.integers(0, 256, size=(rows, k // 32)).astype(np.uint8)
        tiled = mx.mx_scales_from_plain(plain, rows, k)
        assert np.array_equal(tiled, O.scales_plain_to_tiled(plain, rows, k, pad_value=0))
        assert np.array_equal(mx.mx_scales_to_plain(tiled, rows, k), plain)


def test_binding_refuses_to_run_without_library(monkeypatch, tmp_path):
    import microscaled_precision_gemm_gb300 as pkg

    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg._build, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        pkg.load()


def test_c_caller_compiles_links_and_runs(mx, tmp_path):
    """include/mx.h is valid C11; a C program links the library and gets the same answers."""
    import shutil
    import subprocess

    cc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if cc is None or not os.path.isdir(cuda_inc):
        pytest.skip("gcc or the CUDA headers are not available")
    src = os.path.join(ROOT, "tests", "helpers", "c_abi_probe.c")
    exe = str(tmp_path / "c_abi_probe")
    lib_dir = os.path.dirname(mx.library_path())
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, src,
                    "-o", exe, "-L", lib_dir, "-lmxfp6", "-Wl,-rpath," + lib_dir], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout
    got = dict(line.split(" ", 1) for line in out.strip().splitlines())
    assert got["version"] == "100"
    assert int(got["codes_bytes"]) == 128 * 192
    assert int(got["scales_bytes"]) == 384 * 8
    assert int(got["workspace_bytes"]) == mx.mx_mlp_workspace_bytes(256, 512, 1024)
    assert int(got["bad_shape"]) == SHAPE
    assert int(got["null_ptr"]) == INVALID
    assert int(got["gemm_workspace_bytes"]) == mx.mx_gemm_workspace_bytes(20480, 3072, 12288)
    assert got["status_ok"] == "MX_OK"
    assert got["layout_round_trip"] == "1"


def test_gemm_workspace_bytes(lib):
    """Split-tail workspace: 10 KB of arrival counters plus two 256 KB slots per CTA
    pair, for at most 80 pairs and at most one pair fewer than the tiles; none for
    tiles shorter than 32 K-steps."""
    slot, counters = 2 * 128 * 256 * 4, 10240
    assert lib.mx_gemm_workspace_bytes(20480, 3072, 12288) == counters + 2 * 80 * slot
    assert lib.mx_gemm_workspace_bytes(20480, 12288, 4096) == counters + 2 * 80 * slot
    assert lib.mx_gemm_workspace_bytes(20480, 12288, 3072) == 0     # 24 K-steps
    assert lib.mx_gemm_workspace_bytes(1024, 1280, 4096) == counters + 2 * 19 * slot   # 4 x 5 tiles
    assert lib.mx_gemm_workspace_bytes(4096, 3072, 3968) == 0     # 31 K-steps: never splits
    assert lib.mx_gemm_workspace_bytes(256, 256, 8192) == 0       # one tile
    assert lib.mx_gemm_workspace_bytes(256, 384, 8192) == 0       # unsupported N
    assert lib.mx_gemm_workspace_bytes(0, 256, 8192) == 0


def test_noalloc_checks_shape_then_capacity_on_the_host(lib):
    """mx_mlp_noalloc answers in mx_mlp's order, all before any device call: a bad
    shape as mx_mlp does (also with M = 0), then the capacity of its 64 MiB static
    scratch, then null pointers. At d = 3072, ff = 12288 the MXFP6 x and h of 5590
    tokens fit (the call gets as far as the null-pointer check) and of 5591 do not."""
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fn = ctypes.CFUNCTYPE(ctypes.c_int, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp)(
        ("mx_mlp_noalloc", lib))

    def call(M, d=3072, ff=12288, x=None):
        return fn(x, M, d, ff, None, None, None, None, None, None, None, None)

    cap = 64 << 20
    assert _mlp_base(lib, 5590, 3072, 12288) <= cap < _mlp_base(lib, 5591, 3072, 12288)
    assert call(5590) == INVALID
    assert call(5591) == WS_SMALL
    assert call(-1) == INVALID
    assert call(0, d=100) == SHAPE                 # mx_mlp's answer for d % 256, even with M = 0
    assert call(1 << 20, d=100) == SHAPE           # a bad shape is not reported as a capacity problem
    assert call(8, ff=640) == SHAPE                # GELU up-projection width % 256
    assert call(1 << 31) == SHAPE
    assert call(0) == OK
    assert lib.mx_mlp(None, 0, 100, 12288, None, None, None, None, None, None, None, None, 0, None) == SHAPE


def test_quantize_stacked_rejects_bad_arguments(lib):
    """Every part is checked on the host before the first launch."""
    def call(rows, k=256, lds=None, ptrs=None, codes=A32b, scales=A32c, n=None):
        n = len(rows) if n is None else n
        p = (ctypes.c_void_p * max(1, len(rows)))(*(ptrs or [A32 + 0x100000 * i for i in range(len(rows))]))
        r = (ctypes.c_int64 * max(1, len(rows)))(*rows)
        ld = None if lds is None else (ctypes.c_int64 * len(lds))(*lds)
        return lib.mx_quantize_stacked(p, r, ld, n, k, codes, scales, None)

    assert call([128, 64], n=0) == INVALID
    assert lib.mx_quantize_stacked(None, None, None, 1, 256, A32b, A32c, None) == INVALID
    assert call([100, 64]) == SHAPE                    # a part before the last not a multiple of 128 rows
    assert call([128, -1]) == INVALID
    assert call([128, 64], k=100) == SHAPE
    assert call([128, 64], lds=[256, 128]) == INVALID  # ld_x < K
    assert call([128, 64], lds=[256, 260]) == MISALIGNED
    assert call([128, 64], ptrs=[A32, A32 + 8]) == MISALIGNED
    assert call([128, 64], ptrs=[A32, 0]) == INVALID
    assert call([128, 64], codes=A32b + 16) == MISALIGNED
    assert call([128, 1 << 31]) == SHAPE
    assert call([0, 0], ptrs=[0, 0], codes=0, scales=0) == OK   # nothing to quantize
    # an empty first part may have a null pointer; the call then goes on to the device
    assert call([0, 64], ptrs=[0, A32]) not in (OK, INVALID, SHAPE, MISALIGNED)
    assert call([1 << 23, 1 << 23], k=8192) == SHAPE          # each part fits the size limit, the stack does not


def test_c_hot_path_program_compiles_and_links(mx, tmp_path):
    """The C program the GPU test runs (tests/helpers/c_hot_path.c) is valid C11 against
    include/mx.h and links against the library and the CUDA runtime."""
    import shutil
    import subprocess

    cc = shutil.which("gcc")
    cuda = "/usr/local/cuda"
    cuda_lib = next((p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                     if os.path.exists(os.path.join(p, "libcudart.so"))), None)
    if cc is None or cuda_lib is None:
        pytest.skip("gcc or the CUDA runtime is not available")
    lib_dir = os.path.dirname(mx.library_path())
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "helpers", "c_hot_path.c"), "-o",
                    str(tmp_path / "c_hot_path"), "-L", lib_dir, "-lmxfp6", "-L", cuda_lib, "-lcudart",
                    "-Wl,-rpath," + lib_dir], check=True)
