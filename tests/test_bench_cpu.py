"""Host logic of bench.py that needs no GPU: the per-workload GEMM shapes of the
BF16 context against the algorithmic work the roofline uses, and the clock
record's restriction to the samples taken inside the timed region."""

import datetime
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", sorted(bench.CONFIGS))
def test_bf16_context_shapes_carry_the_step_flops(name, fused):
    """The BF16 context times the same contractions the step's MXFP6 GEMM stages do,
    with the quantizer in its own stage or inside the GEMM's; a fused stage carries
    the quantizer's bytes, so the step's algorithmic bytes do not change."""
    cfg = bench.CONFIGS[name]
    M = cfg["M"]
    shapes = bench.gemm_shapes(cfg, M)
    work = bench.stage_work(cfg, M, fused=fused)
    gemm_flops = sum(w["flops"] for w in work.values())
    assert shapes, name
    assert sum(2.0 * m * n * k for m, n, k in shapes) == pytest.approx(gemm_flops, rel=1e-12)
    assert all(m == M for m, _, _ in shapes)
    plain = bench.stage_work(cfg, M)
    assert sum(w["bytes"] for w in work.values()) == pytest.approx(sum(w["bytes"] for w in plain.values()))
    if fused and bench.S_K1 in plain:
        assert bench.S_K1 not in work and any(n in bench.FUSED_STAGES for n in work)


class _FakeSmi:
    """Stands in for the nvidia-smi process: ten samples 25 ms apart starting at t0."""

    def __init__(self, t0: float, cap_at: int):
        self.t0, self.cap_at = t0, cap_at

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        lines = []
        for i in range(10):
            ts = datetime.datetime.fromtimestamp(self.t0 + 0.025 * i).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            cap = "Active" if i == self.cap_at else "Not Active"
            lines.append(f"{ts}, {1400 + 10 * i}, 2070, {500 + i}.0, Not Active, Not Active, Not Active, {cap}")
        return "\n".join(lines) + "\n", ""


def _sampler(fake):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = fake
    return s


def test_clock_record_keeps_only_the_timed_region():
    t0 = 1_700_000_000.0
    clk = _sampler(_FakeSmi(t0, cap_at=5)).stop(window=(t0 + 0.06, t0 + 0.16))
    # samples 3, 4, 5, 6 (at +75, +100, +125, +150 ms) fall inside
    assert clk["window"] == "timed region"
    assert clk["samples"] == 4
    assert clk["sm_mhz"] == pytest.approx((1440 + 1450) / 2)
    assert clk["reasons"] == ["sw_power_cap"]
    assert clk["power_w_max"] == pytest.approx(506.0)


def test_clock_record_outside_the_window_ignores_its_reasons():
    t0 = 1_700_000_000.0
    clk = _sampler(_FakeSmi(t0, cap_at=9)).stop(window=(t0, t0 + 0.1))
    assert clk["samples"] == 5 and clk["reasons"] == []


def test_clock_record_of_a_short_region_extends_only_forward():
    t0 = 1_700_000_000.0
    # region between samples 4 and 5 (+100, +125 ms): no sample inside; the samples
    # after it (5, 6, 7) are taken, never the ones before it (the GPU idled then)
    clk = _sampler(_FakeSmi(t0, cap_at=3)).stop(window=(t0 + 0.105, t0 + 0.12))
    assert clk["samples"] == 3 and clk["reasons"] == []
    assert clk["sm_mhz"] == pytest.approx(1460)
    assert clk["window"].startswith("timed region and the 75 ms after it")


class _FakeSmiNoPower(_FakeSmi):
    """As _FakeSmi, on a board that reports no power draw ("[N/A]")."""

    def communicate(self, timeout=None):
        out, err = super().communicate(timeout)
        lines = []
        for ln in out.strip().splitlines():
            p = ln.split(", ")
            p[3] = "[N/A]"
            lines.append(", ".join(p))
        return "\n".join(lines) + "\n", err


def test_clock_record_without_power_readings():
    t0 = 1_700_000_000.0
    clk = _sampler(_FakeSmiNoPower(t0, cap_at=5)).stop(window=(t0 + 0.06, t0 + 0.16))
    assert clk["samples"] == 4 and clk["power_w_max"] is None
    assert clk["sm_mhz"] == pytest.approx((1440 + 1450) / 2)


def test_clock_record_without_samples_in_the_window_falls_back_to_all():
    t0 = 1_700_000_000.0
    clk = _sampler(_FakeSmi(t0, cap_at=2)).stop(window=(t0 + 10.0, t0 + 11.0))
    assert clk["window"] == "whole sampling run"
    assert clk["samples"] == 10 and clk["reasons"] == ["sw_power_cap"]


def test_cpu_model_names_the_host():
    import platform

    name = bench._cpu_model()
    assert isinstance(name, str) and name
    assert platform.machine() in name


def test_reference_arm_prints_one_contract_line(capsys):
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON line
    with the contract's keys, a cpu_baseline describing the run and a zero-copy e2e."""
    import json

    bench.main(["--impl", "reference", "--config", "pr1", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.2"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == bench.CONFIGS["pr1"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
