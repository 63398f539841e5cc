"""A C11 program runs the hot path on the GPU through include/mx.h alone.

tests/helpers/c_hot_path.c allocates its own device buffers with the CUDA runtime,
copies seeded host inputs in, quantizes the weights (mx_quantize, and
mx_quantize_stacked for the stacked [W_g; W_u] of a SwiGLU MLP), runs mx_mlp and
mx_gated_mlp and copies the results back. Its outputs must be bit-identical to the
Python binding's calls on the same inputs (the same kernels and launch plans), and
its stacked weight bit-identical to mx_quantize of the concatenated matrix.
"""

import os
import shutil
import subprocess

import numpy as np
import pytest

import synth
from mxutil import bf16_to_device

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _compile(mx, out_dir):
    cc = shutil.which("gcc")
    cuda = "/usr/local/cuda"
    if cc is None or not os.path.isdir(os.path.join(cuda, "include")):
        pytest.skip("gcc or the CUDA toolkit is not available")
    lib_dir = os.path.dirname(mx.library_path())
    cuda_lib = next((p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                 os.path.join(cuda, "targets", "sbsa-linux", "lib"))
                     if os.path.exists(os.path.join(p, "libcudart.so"))), None)
    if cuda_lib is None:
        pytest.skip("libcudart.so not found")
    exe = os.path.join(out_dir, "c_hot_path")
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I",
                    os.path.join(cuda, "include"), os.path.join(ROOT, "tests", "helpers", "c_hot_path.c"), "-o", exe,
                    "-L", lib_dir, "-lmxfp6", "-L", cuda_lib, "-lcudart", "-Wl,-rpath," + lib_dir,
                    "-Wl,-rpath," + cuda_lib], check=True)
    return exe


def test_c_program_runs_the_hot_path(lib, tmp_path):
    import torch

    exe = _compile(lib, str(tmp_path))
    M, d, ff, ffg = 300, 256, 512, 384
    w = synth.full_mlp(M=M, d=d, ff=ff)
    g = synth.gated_mlp(M=M, d=d, ff=ffg)
    files = {"x": w["x"], "w1": w["w1"], "b1": w["b1"], "w2": w["w2"], "b2": w["b2"],
             "wg": g["wgu"][:ffg], "wu": g["wgu"][ffg:], "bgu": g["bgu"], "w2g": g["w2"]}
    for name, bits in files.items():
        np.ascontiguousarray(bits, dtype=np.uint16).tofile(str(tmp_path / f"{name}.bin"))
    res = subprocess.run([exe, str(tmp_path), str(M), str(d), str(ff), str(ffg)], capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == "ok"

    def load_bf16(name, shape):
        return torch.from_numpy(np.fromfile(str(tmp_path / name), dtype=np.int16).reshape(shape)).view(
            torch.bfloat16).cuda()

    x = bf16_to_device(w["x"])
    y_py = lib.mx_mlp(x, lib.mx_quantize(bf16_to_device(w["w1"])), bf16_to_device(w["b1"]),
                      lib.mx_quantize(bf16_to_device(w["w2"])), bf16_to_device(w["b2"]))
    assert torch.equal(load_bf16("y.bin", (M, d)), y_py), "mx_mlp from C differs from the binding's call"

    wgu = lib.mx_quantize(bf16_to_device(g["wgu"]))   # the concatenated matrix, quantized whole
    stacked = lib.mx_quantize_stacked([bf16_to_device(files["wg"]), bf16_to_device(files["wu"])])
    c_codes = np.fromfile(str(tmp_path / "wgu_codes.bin"), dtype=np.uint8)
    c_scales = np.fromfile(str(tmp_path / "wgu_scales.bin"), dtype=np.uint8)
    assert np.array_equal(c_codes, wgu.codes.cpu().numpy().ravel())
    assert np.array_equal(c_scales, wgu.scales.cpu().numpy())
    assert torch.equal(stacked.codes, wgu.codes) and torch.equal(stacked.scales, wgu.scales)
    yg_py = lib.mx_gated_mlp(x, wgu, bf16_to_device(g["bgu"]), lib.mx_quantize(bf16_to_device(g["w2"])),
                             bf16_to_device(w["b2"]))
    assert torch.equal(load_bf16("yg.bin", (M, d)), yg_py), "mx_gated_mlp from C differs from the binding's call"
    assert lib.mx_device_error() == 0
