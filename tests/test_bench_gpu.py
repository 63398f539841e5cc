"""The bench's JSON line on a GPU, on the smallest workload: one line on stdout
with the contract's keys (value, e2e with its copy sizes, roofline, cpu_baseline,
clocks, the sustained leg and the launch count), and the reference arm's line."""

import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                         timeout=900, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_bench_line_contract(lib):
    d = _run("--config", "pr1", "--steps", "4", "--warmup", "3", "--sustain-s", "0.3", "--cpu-budget", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "clocks", "e2e",
                "gpu_launches", "sustained"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 4 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    # pr1's step is one stage, the quantizer fused into the GEMM: two launches
    assert list(d["stages"]) == ["K1 lead rows + GEMM (in-kernel quantizer)+bias+BF16"]
    assert d["gpu_launches"] == 4 * 2 and d["config"]["quantizer_in_gemm"] is True
    assert d["quantize_isolated"]["gbs"] > 0 and d["quantize_gbs"] == d["quantize_isolated"]["gbs"]
    assert d["config"]["workload"].startswith("single MXFP6 GEMM")
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] == 128 * 256 * 2 and e2e["d2h_bytes_per_step"] == 128 * 512 * 2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["extrapolated"] is False
    assert set(d["roofline"]) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert d["sustained"]["steps"] >= 1 and d["sustained"]["ms_per_step"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    iso = d["gemms_isolated"]["K1 lead rows + GEMM (in-kernel quantizer)+bias+BF16"]
    assert iso["us"] > 0 and iso["launches"] == 20 and iso["gemm_alone"]["us"] > 0


def test_bench_unfused_stages(lib):
    """--unfused: the quantizer in its own stage before the GEMM."""
    d = _run("--config", "pr1", "--steps", "4", "--warmup", "3", "--sustain-s", "0", "--no-cpu-baseline",
             "--unfused")
    assert list(d["stages"]) == ["K1 quantize", "K2 GEMM+bias+BF16"]
    assert d["gpu_launches"] == 4 * 2 and d["config"]["quantizer_in_gemm"] is False


def test_reference_arm_line(lib):
    d = _run("--impl", "reference", "--config", "pr1", "--steps", "3", "--warmup", "3", "--cpu-budget", "1")
    assert d["impl"] == "reference" and d["value"] > 0 and d["dtype"] == "f64"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
