#!/usr/bin/env python3
"""Throughput of the MXFP6 MLP hot path on GB300, one JSON line on stdout.

Default workload (N=1): the full DiT MLP block, M=20480 tokens (16384 output +
4096 reference), d=3072, ff=12288 -- one step is the whole hot path over one
batch: K1 quantize x -> K3 up-projection + bias + GELU + MXFP6 requant -> K2
down-projection + bias + BF16 store. The weights are quantized once, before
timing (they are inference weights). `value` is MLP GEMM TFLOP/s over the whole
step (2*M*d*ff*2 flops per step, quantizer time included).

Other --config values measure the smaller single-GEMM workloads (pr1, dit_up,
dit_down), the outlier-heavy wide MLP, and the neighbouring fusions: the SwiGLU
MLP (gated_mlp), the stacked query/key/value/gate projection (qkv_proj), the
MLP half of a DiT block with the fused RMSNorm quantizer and the gate/residual
epilogue (dit_block, dit_block_swiglu), and the attention's input (fused RMSNorm
quantizer -> stacked Q/K/V/gate projection: attn_in) and output projection with
its gate and residual (attn_out).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Timing: CUDA events on the launching stream around exactly K steps, after W
warm-up steps, with a synchronize (and, under torchrun, a barrier) on both sides;
the maximum over ranks is reported. Per-kernel events (the roofline's kernel
times) are recorded inside the same timed region on every fourth step. Between steps the inputs rotate over two
independent copies (weights, activations, outputs: 2 x 556 MB > 129 MB L2), so no
step reads operands another step left in L2. nvidia-smi clocks are sampled during
the timed region.
"""

from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MXFP6 MLP GEMM TFLOPS (% of GB300 FP6 peak); ms per DiT MLP; quantize GB/s"
FP6_SPEC_PEAK_TFLOPS = 5000.0   # NVIDIA GB300 NVL72: 720 PF FP8/FP6 with sparsity / 72 GPUs / 2
FP6_PER_BF16 = 2.0              # dense FP8/FP6 tensor rate = 2 x BF16 (4.5 vs 2.25 PF nominal)

CONFIGS = {
    "full_mlp": dict(kind="mlp", M=20480, d=3072, ff=12288,
                     workload="full DiT MLP block (M=20480 tokens = 16384 output + 4096 reference, d=3072, ff=12288)"),
    "outlier_mlp": dict(kind="mlp", M=20480, d=4096, ff=16384,
                        workload="outlier-heavy wide MLP (M=20480, d=4096, ff=16384, Student-t(3), 1% hot channels x100, 1% zero blocks)"),
    "dit_up": dict(kind="up", M=4096, d=3072, ff=12288,
                   workload="DiT MLP up-projection (M=4096, K=3072, N=12288, bias+GELU+MXFP6 requant)"),
    "dit_down": dict(kind="down", M=16384, d=3072, ff=12288,
                     workload="DiT MLP down-projection (M=16384, K=12288, N=3072, bias+BF16 store)"),
    "pr1": dict(kind="gemm", M=128, d=256, ff=512,
                workload="single MXFP6 GEMM (M=128, K=256, N=512, bias+BF16)"),
    "gated_mlp": dict(kind="gated_mlp", M=20480, d=3072, ff=8192,
                      workload="SwiGLU DiT MLP (M=20480, d=3072, ff=8192: stacked gate/up GEMM N=16384 + "
                               "silu(g)*u + MXFP6 requant, down-projection K=8192)"),
    "qkv_proj": dict(kind="qkv", M=20480, d=3072, ff=4 * 3072,
                     workload="stacked query/key/value/gate projection (M=20480, K=3072, N=4*3072, bias+BF16)"),
    "dit_block": dict(kind="block", M=20480, d=3072, ff=12288, activation="gelu",
                      workload="DiT MLP sub-block (M=20480, d=3072, ff=12288: RMSNorm+modulation+MXFP6 quantize "
                               "-> up+GELU+requant -> down + gate x output + residual)"),
    "dit_block_swiglu": dict(kind="block", M=20480, d=3072, ff=8192, activation="swiglu",
                             workload="DiT MLP sub-block, SwiGLU (M=20480, d=3072, ff=8192: RMSNorm+modulation+"
                                      "MXFP6 quantize -> stacked gate/up+SwiGLU+requant -> down + gate + residual)"),
    "attn_in": dict(kind="attn_in", M=20480, d=3072, ff=4 * 3072,
                    workload="DiT attention input (M=20480, d=3072: RMSNorm+modulation+MXFP6 quantize -> stacked "
                             "query/key/value/gate projection N=4*3072, bias+BF16)"),
    "attn_out": dict(kind="attn_out", M=20480, d=3072, ff=3072,
                     workload="DiT attention output projection (M=20480, K=N=3072: MXFP6 quantize of the attention "
                              "output -> projection + bias + gate + residual, BF16)"),
}

# names of the launches of one step
S_K1 = "K1 quantize"
S_K1N = "K1 RMSNorm+modulate+quantize"
S_UP = "K3 up GEMM+GELU+requant"
S_GU = "K3 gate/up GEMM+SwiGLU+requant"
S_DOWN = "K2 down GEMM+bias+BF16"
S_DOWNR = "K2 down GEMM+bias+gate+residual"
S_GEMM = "K2 GEMM+bias+BF16"
S_QKV = "QKV+gate GEMM+bias+BF16"
S_OUT = "out-proj GEMM+bias+gate+residual"
# the quantizer fused into the GEMM (mx_quantize_gemm: the quantize kernel encodes the
# rows of the first round of tiles, the GEMM the rest while it runs): two launches
S_QUP = "K1 lead rows + K3 up GEMM (in-kernel quantizer)+GELU+requant"
S_QGU = "K1 lead rows + K3 gate/up GEMM (in-kernel quantizer)+SwiGLU+requant"
S_QGEMM = "K1 lead rows + GEMM (in-kernel quantizer)+bias+BF16"
S_QQKV = "K1 lead rows + QKV+gate GEMM (in-kernel quantizer)+bias+BF16"
S_QOUT = "K1 lead rows + out-proj GEMM (in-kernel quantizer)+bias+gate+residual"
FUSED_STAGES = (S_QUP, S_QGU, S_QGEMM, S_QQKV, S_QOUT)

# Per-launch DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the current kernels, keyed by (config, stage); None where no
# capture of the current kernel exists. A stage of two launches (the quantize
# kernel on the leading rows, then the GEMM that quantizes the rest) carries both
# launches' traffic. Copied by hand from the ncu traffic captures of the full DiT
# MLP block and of the M = 4096 up-projection (the steps with the quantizer inside
# the up-projection; the full block's three-kernel step) and of the SwiGLU DiT
# sub-block.
NCU_TRAFFIC_BYTES: dict = {
    ("full_mlp", S_QUP): 3172352 + 0 + 154721280 + 206835968,
    ("full_mlp", "K1 quantize"): 125857280 + 22170112,
    ("full_mlp", "K3 up GEMM+GELU+requant"): 80503296 + 152273408,
    ("full_mlp", "K2 down GEMM+bias+BF16"): 246828800 + 107906560,
    ("dit_up", S_QUP): 3168256 + 4608 + 52893952 + 11980288,
    ("dit_block_swiglu", "K1 RMSNorm+modulate+quantize"): 125882112 + 24203264,
    ("dit_block_swiglu", "K3 gate/up GEMM+SwiGLU+requant"): 89456640 + 105300224,
    ("dit_block_swiglu", "K2 down GEMM+bias+gate+residual"): 281890048 + 105528064,
}


# sm__pipe_tensor_cycles_active as a fraction of elapsed cycles, from one ncu capture
# of the current kernel (a full-set or a traffic capture; for a stage of two
# launches, its GEMM's); None where no capture of the current kernel exists.
NCU_TENSOR_PIPE_ACTIVE: dict = {
    ("full_mlp", S_QUP): 0.786,
    ("dit_up", S_QUP): 0.662,
    ("full_mlp", "K3 up GEMM+GELU+requant"): 0.816,
    ("full_mlp", "K2 down GEMM+bias+BF16"): 0.858,
    ("dit_block_swiglu", "K3 gate/up GEMM+SwiGLU+requant"): 0.837,
    ("dit_block_swiglu", "K2 down GEMM+bias+gate+residual"): 0.800,
    ("attn_out", "out-proj GEMM+bias+gate+residual"): 0.682,
    ("attn_out", S_QOUT): 0.682,
}


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sustained": p["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_rows(m_per_rank: int, world: int, rank: int) -> tuple[int, int]:
    """Weak scaling: every rank owns its own batch of m_per_rank tokens (rows
    [rank*m, (rank+1)*m) of the job's token set); the MLP is token-local, so no
    rank needs another's rows and no collective sits on the data path."""
    return rank * m_per_rank, (rank + 1) * m_per_rank


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "25"]
        self.rows = []
        bus = _pci_bus_id(device_index)
        if bus:
            cmd += ["-i", bus]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def stop(self, window: tuple[float, float] | None = None) -> dict:
        """Ends the sampling; returns the summary of `window` (see summary())."""
        self.rows = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            for line in out.strip().splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    t = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    clk = (float(parts[1]), float(parts[2]))
                except ValueError:
                    continue
                try:
                    power = float(parts[3])
                except ValueError:   # "[N/A]" where the board does not report it
                    power = None
                vals = (clk[0], clk[1], power)
                active = {name for name, val in zip(self.NAMES, parts[4:8]) if val.lower().startswith("active")}
                self.rows.append((t, vals, active))
        return self.summary(window)

    def summary(self, window: tuple[float, float] | None, min_samples: int = 3, max_pad_s: float = 0.1) -> dict:
        """Median SM clock, maximum clock and power, and throttle reasons of the samples
        taken inside `window` (wall-clock seconds). A window shorter than the sampling
        interval may hold fewer than `min_samples`: its end is then moved later in 25 ms
        steps, up to `max_pad_s` (into the back-to-back steps that follow the timed
        region; never earlier, where the GPU idled before it), and the record says by
        how much. Without any sample near the window, all samples are summarised
        ("whole sampling run")."""
        rows = getattr(self, "rows", [])
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "no samples"}
        use, label = [], "whole sampling run"
        if window is not None:
            pad = 0.0
            while True:
                use = [r for r in rows if window[0] <= r[0] <= window[1] + pad]
                if len(use) >= min_samples or pad >= max_pad_s - 1e-9:
                    break
                pad += 0.025
            if use:
                label = "timed region" if pad == 0.0 else (
                    f"timed region and the {pad * 1e3:.0f} ms after it (the region is shorter than the sampling "
                    f"interval; the samples after it are of the same steps, continued back to back)")
        if not use:
            use, label = rows, "whole sampling run"
        sm = [r[1][0] for r in use]
        smax = [r[1][1] for r in use]
        power = [r[1][2] for r in use if r[1][2] is not None]
        reasons = set().union(*(r[2] for r in use))
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power) if power else None, "window": label}


def _pci_bus_id(device_index: int) -> str | None:
    try:
        import torch

        p = torch.cuda.get_device_properties(device_index)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return None


# ------------------------------------------------------------------ GPU arm

def _bf16_dev(bits, dev):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


class Workload:
    """Device-resident inputs and outputs of one copy of the configuration."""

    def __init__(self, mx, cfg: dict, seed: int, dev, m_rows: int, split: bool = True, fused: bool = True):
        import torch

        self.cfg = cfg
        self.fused = fused
        kind = cfg["kind"]
        M, d, ff = m_rows, cfg["d"], cfg["ff"]
        self.M, self.d, self.ff = M, d, ff

        def mx_empty(rows, k):
            return mx.MxTensor(torch.empty((rows, k * 3 // 4), dtype=torch.uint8, device=dev),
                               torch.empty(mx.mx_scales_bytes(rows, k), dtype=torch.uint8, device=dev), rows, k)

        if kind in ("mlp", "gated_mlp", "block"):
            if kind == "mlp":
                gen = synth.outlier_mlp if cfg is CONFIGS["outlier_mlp"] else synth.full_mlp
                w = gen(seed=seed, M=M, d=d, ff=ff)
                w_up, b_up = w["w1"], w["b1"]
            elif kind == "gated_mlp":
                w = synth.gated_mlp(seed=seed, M=M, d=d, ff=ff)
                w_up, b_up = w["wgu"], w["bgu"]
            else:
                w = synth.dit_block(seed=seed, M=M, d=d, ff=ff, activation=cfg["activation"])
                w_up, b_up = w["w_up"], w["b_up"]
                self.shift, self.scale, self.gate = (_bf16_dev(w[k], dev) for k in ("shift", "scale", "gate"))
                self.eps = w["eps"]
            self.x = _bf16_dev(w["x"], dev)
            self.w1 = mx.mx_quantize(_bf16_dev(w_up, dev))
            self.w2 = mx.mx_quantize(_bf16_dev(w["w2"], dev))
            self.b1 = _bf16_dev(b_up, dev)
            self.b2 = _bf16_dev(w["b2"], dev)
            self.xq = mx_empty(M, d)
            self.hq = mx_empty(M, ff)
            self.y = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
            self.host = w
        elif kind in ("up", "gemm", "qkv"):
            if kind == "up":
                w = synth.dit_up(seed=seed, M=M, d=d, ff=ff)
            elif kind == "qkv":
                w = synth.qkv_proj(seed=seed, M=M, d=d, stack=ff // d)
            else:
                w = synth.pr1(seed=seed, M=M, K=d, N=ff)
            self.x = _bf16_dev(w["x"], dev)
            self.w1 = mx.mx_quantize(_bf16_dev(w["w"], dev))
            self.b1 = _bf16_dev(w["b"], dev)
            self.xq = mx_empty(M, d)
            if kind == "up":
                self.hq = mx_empty(M, ff)
            else:
                self.y = torch.empty((M, ff), dtype=torch.bfloat16, device=dev)
            self.host = w
        elif kind == "attn_in":
            w = synth.attn_in(seed=seed, M=M, d=d)
            self.x = _bf16_dev(w["x"], dev)
            self.shift, self.scale = _bf16_dev(w["shift"], dev), _bf16_dev(w["scale"], dev)
            self.eps = w["eps"]
            self.w1 = mx.mx_quantize(_bf16_dev(w["w"], dev))
            self.b1 = _bf16_dev(w["b"], dev)
            self.xq = mx_empty(M, d)
            self.y = torch.empty((M, ff), dtype=torch.bfloat16, device=dev)
            self.host = w
        elif kind == "attn_out":
            w = synth.attn_out(seed=seed, M=M, d=d)
            self.a = _bf16_dev(w["a"], dev)
            self.x = _bf16_dev(w["x"], dev)
            self.w2 = mx.mx_quantize(_bf16_dev(w["w"], dev))
            self.b2 = _bf16_dev(w["b"], dev)
            self.gate = _bf16_dev(w["gate"], dev)
            self.xq = mx_empty(M, d)
            self.y = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
            self.host = w
        elif kind == "down":
            w = synth.dit_down(seed=seed, M=M, ff=ff, d=d)
            z = torch.from_numpy(w["z"]).to(dev)
            h = torch.nn.functional.gelu(z, approximate="tanh").to(torch.bfloat16)
            del z
            self.hq = mx.mx_quantize(h)
            del h
            self.w2 = mx.mx_quantize(_bf16_dev(w["w"], dev))
            self.b2 = _bf16_dev(w["b"], dev)
            self.y = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
            self.host = {"w": w["w"], "b": w["b"]}
        # one split-tail workspace (arrival counters zeroed once; every GEMM leaves
        # them zero) shared by the step's GEMMs, which run one after the other
        shapes = {"mlp": [(M, ff, d), (M, d, ff)], "gated_mlp": [(M, 2 * ff, d), (M, d, ff)],
                  "block": [(M, 2 * ff, d), (M, d, ff)], "up": [(M, ff, d)], "gemm": [(M, ff, d)],
                  "qkv": [(M, ff, d)], "attn_in": [(M, ff, d)], "attn_out": [(M, d, d)], "down": [(M, d, ff)]}
        need = max(mx.mx_gemm_workspace_bytes(*s) for s in shapes[kind]) if split else 0
        # (a workspace smaller than mx_gemm_workspace_bytes runs the GEMMs unsplit)
        self.ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        self.split = split
        # mx_quantize_gemm's workspace (MXFP6 activations + row-block counters)
        self.qws = None
        if kind in ("mlp", "gated_mlp", "up", "gemm", "qkv", "attn_out"):
            self.qws = torch.empty(max(256, mx.mx_quantize_gemm_workspace_bytes(M, d)), dtype=torch.uint8,
                                   device=dev)
        torch.cuda.synchronize()

    def gemm_alone(self, mx):
        """{fused stage name: callable}: the stage's GEMM on activations already in MXFP6
        (xq, filled here once by the quantize kernel), without the quantizer."""
        kind = self.cfg["kind"]
        if not self.fused or kind not in ("mlp", "gated_mlp", "up", "gemm", "qkv", "attn_out"):
            return {}
        src = self.a if kind == "attn_out" else self.x
        mx.mx_quantize(src, out=self.xq)
        swiglu = kind == "gated_mlp"
        if kind in ("mlp", "gated_mlp", "up"):
            epi = mx.MX_EPI_BIAS_SWIGLU_MXFP6 if swiglu else mx.MX_EPI_BIAS_GELU_MXFP6
            return {S_QGU if swiglu else S_QUP: lambda: mx.mx_gemm(self.xq, self.w1, self.b1, epi, out=self.hq,
                                                                    workspace=self.ws)}
        if kind in ("gemm", "qkv"):
            return {S_QQKV if kind == "qkv" else S_QGEMM: lambda: mx.mx_gemm(self.xq, self.w1, self.b1,
                                                                          mx.MX_EPI_BIAS_BF16, out=self.y,
                                                                          workspace=self.ws)}
        return {S_QOUT: lambda: mx.mx_gemm_gate_residual(self.xq, self.w2, self.b2, self.gate, self.x, out=self.y,
                                                         workspace=self.ws)}

    def quantizer(self, mx):
        """(name, callable) of the step's whole quantizer, launched on its own."""
        kind = self.cfg["kind"]
        if kind in ("block", "attn_in"):
            return S_K1N, lambda: mx.mx_quantize_rmsnorm_modulate(self.x, self.shift, self.scale, self.eps,
                                                                  out=self.xq)
        if kind == "down":
            return None, None
        src = self.a if kind == "attn_out" else self.x
        return S_K1, lambda: mx.mx_quantize(src, out=self.xq)

    def stages(self, mx):
        """The step's launches as (name, callable) in stream order."""
        kind = self.cfg["kind"]
        swiglu = kind == "gated_mlp" or (kind == "block" and self.cfg["activation"] == "swiglu")
        epi_up = mx.MX_EPI_BIAS_SWIGLU_MXFP6 if swiglu else mx.MX_EPI_BIAS_GELU_MXFP6
        out = []
        if self.fused and kind in ("mlp", "gated_mlp", "up"):
            out.append((S_QGU if swiglu else S_QUP,
                        lambda: mx.mx_quantize_gemm(self.x, self.w1, self.b1, epi_up, out=self.hq, workspace=self.qws)))
        elif self.fused and kind in ("gemm", "qkv"):
            out.append((S_QQKV if kind == "qkv" else S_QGEMM,
                        lambda: mx.mx_quantize_gemm(self.x, self.w1, self.b1, mx.MX_EPI_BIAS_BF16, out=self.y,
                                                    workspace=self.qws)))
        elif self.fused and kind == "attn_out":
            out.append((S_QOUT, lambda: mx.mx_quantize_gemm(self.a, self.w2, self.b2, mx.MX_EPI_GATE_RESIDUAL_BF16,
                                                            gate=self.gate, residual=self.x, out=self.y,
                                                            workspace=self.qws)))
        else:
            if kind in ("mlp", "gated_mlp", "up", "gemm", "qkv"):
                out.append((S_K1, lambda: mx.mx_quantize(self.x, out=self.xq)))
            if kind == "attn_out":
                out.append((S_K1, lambda: mx.mx_quantize(self.a, out=self.xq)))
                out.append((S_OUT, lambda: mx.mx_gemm_gate_residual(self.xq, self.w2, self.b2, self.gate, self.x,
                                                                    out=self.y, workspace=self.ws)))
            if kind in ("mlp", "gated_mlp", "up"):
                out.append((S_GU if swiglu else S_UP, lambda: mx.mx_gemm(self.xq, self.w1, self.b1, epi_up,
                                                                             out=self.hq, workspace=self.ws)))
            if kind in ("gemm", "qkv"):
                out.append((S_QKV if kind == "qkv" else S_GEMM,
                            lambda: mx.mx_gemm(self.xq, self.w1, self.b1, mx.MX_EPI_BIAS_BF16, out=self.y,
                                               workspace=self.ws)))
        if kind in ("block", "attn_in"):
            out.append((S_K1N, lambda: mx.mx_quantize_rmsnorm_modulate(self.x, self.shift, self.scale, self.eps,
                                                                       out=self.xq)))
        if kind == "attn_in":
            out.append((S_QKV, lambda: mx.mx_gemm(self.xq, self.w1, self.b1, mx.MX_EPI_BIAS_BF16, out=self.y,
                                                     workspace=self.ws)))
        if kind == "block":
            out.append((S_GU if swiglu else S_UP, lambda: mx.mx_gemm(self.xq, self.w1, self.b1, epi_up, out=self.hq,
                                                                         workspace=self.ws)))
        if kind in ("mlp", "gated_mlp", "down"):
            out.append((S_DOWN, lambda: mx.mx_gemm(self.hq, self.w2, self.b2, mx.MX_EPI_BIAS_BF16, out=self.y,
                                                     workspace=self.ws)))
        if kind == "block":
            out.append((S_DOWNR, lambda: mx.mx_gemm_gate_residual(self.hq, self.w2, self.b2, self.gate, self.x,
                                                                  out=self.y, workspace=self.ws)))
        return out


def gemm_shapes(cfg: dict, M: int) -> list:
    """(m, n, k) of the step's GEMMs, in BF16 terms (the SwiGLU gate/up GEMM is one 2 ff wide matmul)."""
    d, ff, kind = cfg["d"], cfg["ff"], cfg["kind"]
    swiglu = kind == "gated_mlp" or (kind == "block" and cfg.get("activation") == "swiglu")
    if kind in ("mlp", "gated_mlp", "block"):
        return [(M, 2 * ff if swiglu else ff, d), (M, d, ff)]
    if kind in ("up", "gemm", "qkv", "attn_in"):
        return [(M, ff, d)]
    if kind == "down":
        return [(M, d, ff)]
    if kind == "attn_out":
        return [(M, d, d)]
    return []


def bf16_context(shapes: list, dev, iters: int = 20) -> dict | None:
    """torch.matmul in BF16 (cuBLAS) on each shape, back to back after warm-up, CUDA events."""
    import torch

    if not shapes:
        return None
    gen = torch.Generator(device=dev).manual_seed(0)
    per, total = [], 0.0
    for (m, n, k) in shapes:
        a = torch.randn((m, k), device=dev, dtype=torch.bfloat16, generator=gen)
        b = torch.randn((n, k), device=dev, dtype=torch.bfloat16, generator=gen)
        out = torch.empty((m, n), device=dev, dtype=torch.bfloat16)
        for _ in range(3):
            torch.matmul(a, b.t(), out=out)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            torch.matmul(a, b.t(), out=out)
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        per.append({"m": m, "n": n, "k": k, "ms": ms, "tflops": 2 * m * n * k / (ms * 1e-3) / 1e12})
        total += ms
        del a, b, out
    return {"kernel": "torch.matmul BF16 (cuBLAS), the step's GEMM shapes, back to back, outside the timed region",
            "ms": total, "gemms": per}


def mlp_min_workspace_bytes(mx, M: int, d: int, ff: int) -> int:
    """MLP workspace without the split-tail region: MXFP6 x and h and a counter word
    per 128 rows, 256-byte aligned parts."""
    parts = (mx.mx_codes_bytes(M, d), mx.mx_scales_bytes(M, d), mx.mx_codes_bytes(M, ff), mx.mx_scales_bytes(M, ff),
             4 * (-(-M // 128)))
    return sum(-(-n // 256) * 256 for n in parts)


def quantizer_bytes(cfg: dict, M: int) -> float:
    """Algorithmic bytes of quantizing the step's activations: BF16 in, MXFP6 out."""
    return M * cfg["d"] * (2 + 0.78125)


def stage_work(cfg: dict, M: int, fused: bool = False) -> dict:
    """Algorithmic flops / bytes per launch of each stage of the step (0.78125 = 0.75
    code + 1/32 scale bytes per MXFP6 element). fused: the quantizer runs inside the
    GEMM that reads its output (Workload.stages with fused=True), and that stage does
    both one's work."""
    d, ff = cfg["d"], cfg["ff"]
    kind = cfg["kind"]
    swiglu = kind == "gated_mlp" or (kind == "block" and cfg.get("activation") == "swiglu")
    q = 0.78125
    out = {}
    if kind in ("mlp", "gated_mlp", "up", "gemm", "qkv"):
        out[S_K1] = {"bytes": M * d * (2 + q), "flops": 0.0}
    if kind in ("block", "attn_in"):
        out[S_K1N] = {"bytes": M * d * (2 + q), "flops": 0.0}
    if kind == "attn_in":
        out[S_QKV] = {"flops": 2.0 * M * d * ff, "bytes": (M + ff) * d * q + M * ff * 2}
    if kind == "attn_out":
        out[S_K1] = {"bytes": M * d * (2 + q), "flops": 0.0}
        out[S_OUT] = {"flops": 2.0 * M * d * ff, "bytes": M * d * q + ff * d * q + M * ff * 4}
    if kind in ("mlp", "up", "block") and not swiglu:
        out[S_UP] = {"flops": 2.0 * M * d * ff, "bytes": M * d * q + ff * d * q + M * ff * q}
    if swiglu:
        out[S_GU] = {"flops": 2.0 * M * d * 2 * ff, "bytes": M * d * q + 2 * ff * d * q + M * ff * q}
    if kind == "gemm":
        out[S_GEMM] = {"flops": 2.0 * M * d * ff, "bytes": (M + ff) * d * q + M * ff * 2}
    if kind == "qkv":
        out[S_QKV] = {"flops": 2.0 * M * d * ff, "bytes": (M + ff) * d * q + M * ff * 2}
    if kind in ("mlp", "gated_mlp", "down"):
        out[S_DOWN] = {"flops": 2.0 * M * d * ff, "bytes": M * ff * q + d * ff * q + M * d * 2}
    if kind == "block":
        out[S_DOWNR] = {"flops": 2.0 * M * d * ff, "bytes": M * ff * q + d * ff * q + M * d * 4}
    if fused and kind in ("mlp", "gated_mlp", "up", "gemm", "qkv", "attn_out"):
        # the quantizer stage folds into the GEMM stage that reads its output
        k1 = out.pop(S_K1)
        for merged, gemm in ((S_QUP, S_UP), (S_QGU, S_GU), (S_QGEMM, S_GEMM), (S_QQKV, S_QKV), (S_QOUT, S_OUT)):
            if gemm in out:
                g = out.pop(gemm)
                out[merged] = {"flops": g["flops"], "bytes": g["bytes"] + k1["bytes"]}
    return out


def run_gpu(args) -> dict | None:
    import torch

    import microscaled_precision_gemm_gb300 as mx

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    mx.load()
    cfg = CONFIGS[args.config]
    M = cfg["M"]
    lo, hi = shard_rows(M, world, rank)
    # two independent copies; copy i uses seed (2*rank + i) so every rank's batch is its own
    copies = [Workload(mx, cfg, seed=2 * rank + i, dev=dev, m_rows=hi - lo, split=not args.no_split,
                       fused=not args.unfused)
              for i in range(args.copies)]
    stream = torch.cuda.current_stream()
    stage_names = [n for n, _ in copies[0].stages(mx)]
    launches = [c.stages(mx) for c in copies]

    for i in range(args.warmup):
        for _, fn in launches[i % len(launches)]:
            fn()
    torch.cuda.synchronize()
    if mx.mx_device_error() != 0:
        raise RuntimeError("a kernel reported a device-side wait timeout during warm-up")

    n_st = len(stage_names)
    # per-kernel events on every fourth timed step: an event recorded between two
    # kernels ends the programmatic overlap of the second one's launch with the
    # first one's tail, so the uninstrumented steps keep it
    probe = [i for i in range(args.steps) if i % 4 == 3] or [0]
    ev = {i: [torch.cuda.Event(enable_timing=True) for _ in range(n_st + 1)] for i in probe}
    clocks = ClockSampler(dev.index or 0)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    t_region0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        e = ev.get(i)
        if e is not None:
            e[0].record(stream)
        for j, (_, fn) in enumerate(launches[i % len(launches)]):
            fn()
            if e is not None:
                e[j + 1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    t_region1 = time.time()
    barrier(world)
    total_ms = max_over_ranks(start.elapsed_time(stop), world)

    per_stage = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in probe) / len(probe) for j in range(n_st)]
    if mx.mx_device_error() != 0:
        raise RuntimeError("a kernel reported a device-side wait timeout in the timed region")

    ms_step = total_ms / args.steps
    work = stage_work(cfg, hi - lo, fused=not args.unfused)
    step_flops = sum(w["flops"] for w in work.values()) * world
    value = step_flops / (ms_step * 1e-3) / 1e12
    # the quantizer alone, back to back over the copies with no event between launches
    # (inside a step its event window also holds the launch gap after the previous kernel)
    k1_isolated = None
    k1_name = copies[0].quantizer(mx)[0]
    if k1_name is not None:
        k1_fns = [c.quantizer(mx)[1] for c in copies]
        for i in range(4):
            k1_fns[i % len(k1_fns)]()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        n_iso = 50
        a.record(stream)
        for i in range(n_iso):
            k1_fns[i % len(k1_fns)]()
        b.record(stream)
        torch.cuda.synchronize()
        iso_ms = a.elapsed_time(b) / n_iso
        k1_isolated = {"kernel": k1_name, "us": iso_ms * 1e3,
                       "gbs": quantizer_bytes(cfg, hi - lo) / (iso_ms * 1e-3) / 1e9,
                       "launches": n_iso, "note": "back-to-back launches over the input copies, outside the timed region"}

    # every GEMM stage alone, back to back over the copies (its launches overlap one
    # another's prologue and tail as consecutive launches of one kernel do), outside
    # the timed region: the kernel's own rate, without the step's other kernels
    gemms_isolated = {}
    for name in stage_names:
        if not work[name]["flops"]:
            continue
        fns = [dict(c.stages(mx))[name] for c in copies]
        for i in range(3):
            fns[i % len(fns)]()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        n_iso = 20
        a.record(stream)
        for i in range(n_iso):
            fns[i % len(fns)]()
        b.record(stream)
        torch.cuda.synchronize()
        g_ms = a.elapsed_time(b) / n_iso
        tf = work[name]["flops"] / (g_ms * 1e-3) / 1e12
        gemms_isolated[name] = {"us": g_ms * 1e3, "tflops": tf, "frac_fp6_peak_spec": tf / FP6_SPEC_PEAK_TFLOPS,
                                "launches": n_iso}
        # a fused stage's GEMM alone, on activations already quantized (the GEMM's own rate)
        alone = [c.gemm_alone(mx).get(name) for c in copies]
        if alone[0] is not None:
            for i in range(3):
                alone[i % len(alone)]()
            torch.cuda.synchronize()
            a.record(stream)
            for i in range(n_iso):
                alone[i % len(alone)]()
            b.record(stream)
            torch.cuda.synchronize()
            g_ms = a.elapsed_time(b) / n_iso
            tf = work[name]["flops"] / (g_ms * 1e-3) / 1e12
            gemms_isolated[name]["gemm_alone"] = {"us": g_ms * 1e3, "tflops": tf,
                                                  "frac_fp6_peak_spec": tf / FP6_SPEC_PEAK_TFLOPS,
                                                  "note": "the same GEMM on activations already in MXFP6"}

    # sustained leg: the same rotation of steps, back to back for a few seconds after
    # the timed region (and after the quantizer's isolated timing, which would
    # otherwise run at the power-capped clock the leg leaves behind), so the power
    # cap has settled and the clock sampler (every 25 ms) has many samples inside
    # its window
    sustained = None
    if args.sustain_s > 0:
        n_sus = max(1, int(args.sustain_s / max(total_ms / args.steps * 1e-3, 1e-6)))
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        barrier(world)
        t_sus0 = time.time()
        s0.record(stream)
        for i in range(n_sus):
            for _, fn in launches[i % len(launches)]:
                fn()
        s1.record(stream)
        torch.cuda.synchronize()
        t_sus1 = time.time()
        barrier(world)
        sustained = {"steps": n_sus, "ms_per_step": max_over_ranks(s0.elapsed_time(s1), world) / n_sus,
                     "seconds": t_sus1 - t_sus0, "window": (t_sus0, t_sus1)}
    clk = clocks.stop(window=(t_region0, t_region1))
    peaks = load_peaks()
    # The driver measured cuBLAS bf16 both as a burst and as a seconds-long loop under
    # the power cap; take the sustained figure when the power cap acted in our timed
    # region, the burst figure otherwise.
    capped = "sw_power_cap" in (clk.get("reasons") or [])
    bf16_basis = peaks["bf16_sustained"] if capped else peaks["bf16"]
    basis_name = "sustained" if capped else "burst"
    fp6_peak = FP6_PER_BF16 * bf16_basis
    stage_report = {}
    for name, ms in zip(stage_names, per_stage):
        w = work[name]
        rep = {"ms": ms}
        if w["flops"]:
            rep["tflops"] = w["flops"] / (ms * 1e-3) / 1e12
            rep["frac_fp6_peak_measured"] = rep["tflops"] / fp6_peak
            rep["frac_fp6_peak_spec"] = rep["tflops"] / FP6_SPEC_PEAK_TFLOPS
        rep["gbs"] = w["bytes"] / (ms * 1e-3) / 1e9
        stage_report[name] = rep
    # dominant kernel = largest share of the step
    dom = max(stage_names, key=lambda n: stage_report[n]["ms"])
    dw = work[dom]
    if dw["flops"]:
        roof = {"kernel": dom, "bound": "tensor", "achieved": stage_report[dom]["tflops"], "peak": fp6_peak,
                "unit": "TFLOP/s", "frac": stage_report[dom]["tflops"] / fp6_peak,
                "peak_basis": f"2 x {peaks['source']} {basis_name} bf16 cuBLAS ({bf16_basis} TFLOP/s): "
                              f"dense FP6/FP8 rate = 2 x BF16 (of {peaks['source']})",
                "traffic": NCU_TRAFFIC_BYTES.get((args.config, dom)),
                "frac_spec_5pf": stage_report[dom]["tflops"] / FP6_SPEC_PEAK_TFLOPS,
                "tensor_pipe_active_ncu": NCU_TENSOR_PIPE_ACTIVE.get((args.config, dom))}
    else:
        roof = {"kernel": dom, "bound": "hbm", "achieved": stage_report[dom]["gbs"], "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": stage_report[dom]["gbs"] / peaks["hbm_gbs"],
                "traffic": NCU_TRAFFIC_BYTES.get((args.config, dom))}


    # end to end through the public API with host buffers (rank 0's view; all ranks run it)
    e2e = run_e2e(mx, copies, cfg, args, world)

    # context: the default BF16 GEMM (torch.matmul, cuBLAS) on the step's GEMM shapes,
    # against this step's MXFP6 GEMM stages (the comparison the source pages make)
    bf16_ctx = bf16_context(gemm_shapes(cfg, hi - lo), dev)
    if bf16_ctx is not None:
        ours = sum(stage_report[n]["ms"] for n in stage_names if work[n]["flops"])
        bf16_ctx["mxfp6_gemm_ms"] = ours
        bf16_ctx["mxfp6_speedup"] = bf16_ctx["ms"] / ours if ours > 0 else None

    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp6_e2m3 (fp32 accumulate)",
        "data": "synthetic (seeded numpy PCG64, BF16 RNE; random-init weights)",
        "config": {"workload": cfg["workload"], "M_per_gpu": hi - lo, "d": cfg["d"], "ff": cfg["ff"],
                   "l2": f"inputs, weights and outputs rotate over {args.copies} independent copies per step; "
                         "each step's working set exceeds the 129 MB L2, so no step reads operands the "
                         "previous step left in L2" if args.copies > 1 else "single copy (profiling run)",
                   "parallelism": f"token-sharded x{world}, weights replicated, no collective",
                   "split_tail": not args.no_split,
                   "quantizer_in_gemm": not args.unfused},
        "ms_per_mlp": ms_step if cfg["kind"] in ("mlp", "gated_mlp", "block") else None,
        "stages": stage_report,
        "roofline": roof,
        "pct_fp6_peak_spec_5pf": value / FP6_SPEC_PEAK_TFLOPS,
        # a fused stage is two launches (the quantize kernel, then the GEMM)
        "gpu_launches": args.steps * sum(2 if n in FUSED_STAGES else 1 for n in stage_names),
        "clocks": clk,
        "gpu": {"name": torch.cuda.get_device_name(dev),
                "sms": torch.cuda.get_device_properties(dev).multi_processor_count},
        "e2e": e2e,
    }
    k1 = S_K1 if S_K1 in stage_report else (S_K1N if S_K1N in stage_report else None)
    if k1 is not None:
        line["quantize_gbs"] = stage_report[k1]["gbs"]
        line["quantize_frac_hbm"] = stage_report[k1]["gbs"] / peaks["hbm_gbs"]
    elif k1_isolated is not None:
        # the step quantizes inside the GEMM: the standalone quantizer's rate, launched alone
        line["quantize_gbs"] = k1_isolated["gbs"]
        line["quantize_frac_hbm"] = k1_isolated["gbs"] / peaks["hbm_gbs"]
        line["quantize_note"] = ("the timed step quantizes the activations inside the GEMM (the quantize kernel "
                                 "encodes only the rows of the first round of tiles); quantize_gbs is the "
                                 "standalone quantizer over all rows, launched alone")
    if k1_isolated is not None:
        k1_isolated["frac_hbm"] = k1_isolated["gbs"] / peaks["hbm_gbs"]
        line["quantize_isolated"] = k1_isolated
    if gemms_isolated:
        for rep in gemms_isolated.values():
            rep["frac_fp6_peak_measured"] = rep["tflops"] / fp6_peak
            if "gemm_alone" in rep:
                rep["gemm_alone"]["frac_fp6_peak_measured"] = rep["gemm_alone"]["tflops"] / fp6_peak
        line["gemms_isolated"] = gemms_isolated
        line["gemms_isolated_note"] = ("each GEMM stage launched alone 20 times back to back over the input copies, "
                                       "outside the timed region")
    if bf16_ctx is not None:
        line["bf16_context"] = bf16_ctx
    if sustained is not None:
        sclk = clocks.summary(sustained.pop("window"))
        sms = sustained["ms_per_step"]
        sustained.update({
            "value": step_flops / (sms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "pct_fp6_peak_spec_5pf": step_flops / (sms * 1e-3) / 1e12 / FP6_SPEC_PEAK_TFLOPS,
            "clocks": sclk,
            # time x clock: comparable between runs at different SM clocks (us * MHz)
            "time_x_mhz": sms * 1e3 * sclk["sm_mhz"] if sclk.get("sm_mhz") else None,
            "note": "the timed region's rotation of steps, back to back right after it, with no events "
                    "between kernels; clocks from the samples inside this leg's own window"})
        line["sustained"] = sustained
        if sustained["time_x_mhz"]:
            # the clock at which the sustained leg's cycles per step give the timed region's
            # step time: the timed region's effective SM clock, whatever the samples say
            line["sm_mhz_effective"] = sustained["time_x_mhz"] / (ms_step * 1e3)
    if clk.get("sm_mhz"):
        line["time_x_mhz"] = ms_step * 1e3 * clk["sm_mhz"]
        roof["kernel_time_x_mhz"] = stage_report[dom]["ms"] * 1e3 * clk["sm_mhz"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, budget_s=args.cpu_budget)
    return line


def run_e2e(mx, copies, cfg, args, world) -> dict:
    """Same metric through the public API (mx_mlp, or the configuration's calls)
    with pinned host input and output buffers: every step copies its input
    host->device and its result device->host inside the timed region. Steps are
    pipelined on three streams (upload, compute, download) with two device
    buffers, so step i+1's upload and step i-1's download overlap step i's compute."""
    import torch

    kind = cfg["kind"]
    c = copies[0]
    if kind in ("mlp", "gated_mlp", "block"):
        src, dst = c.x, c.y
    elif kind == "down":
        src, dst = c.hq.codes, c.y
    elif kind == "up":
        src, dst = c.x, c.hq.codes
    elif kind == "attn_out":
        src, dst = c.a, c.y
    else:
        src, dst = c.x, c.y
    h_in = torch.empty(src.shape, dtype=src.dtype, pin_memory=True)
    h_in.copy_(src)
    h_out = torch.empty(dst.shape, dtype=dst.dtype, pin_memory=True)
    steps = max(1, min(args.steps, 50))
    dev = src.device
    x_buf = [src, torch.empty_like(src)]
    y_buf = [dst, torch.empty_like(dst)]
    ws = None
    if kind in ("mlp", "gated_mlp", "block"):
        ws_bytes = mx.mx_mlp_workspace_bytes(c.M, c.d, c.ff) if c.split else mlp_min_workspace_bytes(mx, c.M, c.d,
                                                                                                      c.ff)
        ws = torch.empty(max(256, ws_bytes), dtype=torch.uint8, device=dev)
    s_up, s_comp, s_down = (torch.cuda.Stream(device=dev) for _ in range(3))
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731
    up_done = [ev(), ev()]
    comp_done = [ev(), ev()]
    down_done = [ev(), ev()]
    for e in comp_done + down_done:
        e.record(torch.cuda.current_stream())

    def compute(slot):
        if kind == "mlp":
            mx.mx_mlp(x_buf[slot], c.w1, c.b1, c.w2, c.b2, y=y_buf[slot], workspace=ws, stream=s_comp)
        elif kind == "gated_mlp":
            mx.mx_gated_mlp(x_buf[slot], c.w1, c.b1, c.w2, c.b2, y=y_buf[slot], workspace=ws, stream=s_comp)
        elif kind == "block":
            act = mx.MX_ACT_SWIGLU if cfg["activation"] == "swiglu" else mx.MX_ACT_GELU_TANH
            mx.mx_dit_mlp_block(x_buf[slot], c.shift, c.scale, c.gate, c.w1, c.b1, c.w2, c.b2, eps=c.eps,
                                activation=act, y=y_buf[slot], workspace=ws, stream=s_comp)
        elif kind == "attn_in":
            mx.mx_quantize_rmsnorm_modulate(x_buf[slot], c.shift, c.scale, c.eps, out=c.xq, stream=s_comp)
            mx.mx_gemm(c.xq, c.w1, c.b1, mx.MX_EPI_BIAS_BF16, out=y_buf[slot], stream=s_comp, workspace=c.ws)
        elif kind == "attn_out" and c.fused:
            mx.mx_quantize_gemm(x_buf[slot], c.w2, c.b2, mx.MX_EPI_GATE_RESIDUAL_BF16, gate=c.gate, residual=c.x,
                                out=y_buf[slot], workspace=c.qws, stream=s_comp)
        elif kind == "attn_out":
            mx.mx_quantize(x_buf[slot], out=c.xq, stream=s_comp)
            mx.mx_gemm_gate_residual(c.xq, c.w2, c.b2, c.gate, c.x, out=y_buf[slot], stream=s_comp,
                                     workspace=c.ws)
        elif kind == "down":
            mx.mx_gemm(mx.MxTensor(x_buf[slot], c.hq.scales, c.hq.rows, c.hq.k), c.w2, c.b2,
                       mx.MX_EPI_BIAS_BF16, out=y_buf[slot], stream=s_comp, workspace=c.ws)
        elif kind == "up" and c.fused:
            mx.mx_quantize_gemm(x_buf[slot], c.w1, c.b1, mx.MX_EPI_BIAS_GELU_MXFP6,
                                out=mx.MxTensor(y_buf[slot], c.hq.scales, c.hq.rows, c.hq.k), workspace=c.qws,
                                stream=s_comp)
        elif kind == "up":
            mx.mx_quantize(x_buf[slot], out=c.xq, stream=s_comp)
            mx.mx_gemm(c.xq, c.w1, c.b1, mx.MX_EPI_BIAS_GELU_MXFP6,
                       out=mx.MxTensor(y_buf[slot], c.hq.scales, c.hq.rows, c.hq.k), stream=s_comp, workspace=c.ws)
        elif c.fused:
            mx.mx_quantize_gemm(x_buf[slot], c.w1, c.b1, mx.MX_EPI_BIAS_BF16, out=y_buf[slot], workspace=c.qws,
                                stream=s_comp)
        else:
            mx.mx_quantize(x_buf[slot], out=c.xq, stream=s_comp)
            mx.mx_gemm(c.xq, c.w1, c.b1, mx.MX_EPI_BIAS_BF16, out=y_buf[slot], stream=s_comp, workspace=c.ws)

    def step(i):
        slot = i % 2
        s_up.wait_event(comp_done[slot])            # x[slot] no longer read by step i-2
        with torch.cuda.stream(s_up):
            x_buf[slot].copy_(h_in, non_blocking=True)
        up_done[slot].record(s_up)
        s_comp.wait_event(up_done[slot])
        s_comp.wait_event(down_done[slot])           # y[slot] already downloaded by step i-2
        compute(slot)
        comp_done[slot].record(s_comp)
        s_down.wait_event(comp_done[slot])
        with torch.cuda.stream(s_down):
            h_out.copy_(y_buf[slot], non_blocking=True)
        down_done[slot].record(s_down)

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    s_comp.wait_event(a)
    s_down.wait_event(a)
    for i in range(steps):
        step(i)
    s_down.wait_stream(s_comp)
    b.record(s_down)
    torch.cuda.synchronize()
    ms = max_over_ranks(a.elapsed_time(b), world) / steps
    flops = sum(w["flops"] for w in stage_work(cfg, c.M).values()) * world
    return {"value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms, "steps": steps,
            "h2d_bytes_per_step": int(src.numel() * src.element_size()),
            "d2h_bytes_per_step": int(dst.numel() * dst.element_size()),
            "pipelining": "3 streams (upload / compute / download), 2 device buffers"}


# ------------------------------------------------------------------ CPU oracle arm

def _cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _cpu_model() -> str:
    """The host CPU's model name and architecture ("Neoverse-V2 (aarch64)" on a Grace host)."""
    import platform

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return f"{ln.split(':', 1)[1].strip()} ({platform.machine()})"
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine() or "unknown"


class OracleWorkload:
    """The configuration's inputs with oracle-quantized weights (setup, untimed)."""

    def __init__(self, cfg: dict, sample_rows: int):
        import oracle as O

        self.O = O
        self.cfg = cfg
        kind = cfg["kind"]
        M = cfg["M"]
        d, ff = cfg["d"], cfg["ff"]
        if kind in ("mlp", "gated_mlp", "block"):
            if kind == "mlp":
                gen = synth.outlier_mlp if cfg is CONFIGS["outlier_mlp"] else synth.full_mlp
                w = gen(M=M, d=d, ff=ff)
                w_up = w["w1"]
            elif kind == "gated_mlp":
                w = synth.gated_mlp(M=M, d=d, ff=ff)
                w_up = w["wgu"]
            else:
                w = synth.dit_block(M=M, d=d, ff=ff, activation=cfg["activation"])
                w_up = w["w_up"]
            self.w1q, self.w1s = O.quantize_bf16(w_up)
            self.w2q, self.w2s = O.quantize_bf16(w["w2"])
        elif kind in ("attn_in", "attn_out"):
            w = synth.attn_in(M=M, d=d) if kind == "attn_in" else synth.attn_out(M=M, d=d)
            self.w1q, self.w1s = O.quantize_bf16(w["w"])
        elif kind in ("up", "gemm", "qkv"):
            if kind == "up":
                w = synth.dit_up(M=M)
            elif kind == "qkv":
                w = synth.qkv_proj(M=M, d=d, stack=ff // d)
            else:
                w = synth.pr1()
            self.w1q, self.w1s = O.quantize_bf16(w["w"])
        else:
            w = synth.dit_down(M=min(M, sample_rows * 8))
            self.w2q, self.w2s = O.quantize_bf16(w["w"])
            w["x_f32"] = w.pop("z")
        self.w = w

    def step(self, rows: np.ndarray) -> float:
        """One bounded sample of the hot path on `rows`; returns its algorithmic flops."""
        O, w, kind = self.O, self.w, self.cfg["kind"]
        d, ff = self.cfg["d"], self.cfg["ff"]
        if kind == "mlp":
            O.mlp(w["x"][rows], self.w1q, self.w1s, w["b1"], self.w2q, self.w2s, w["b2"])
            return 4.0 * len(rows) * d * ff
        if kind == "gated_mlp":
            O.gated_mlp(w["x"][rows], self.w1q, self.w1s, w["bgu"], self.w2q, self.w2s, w["b2"])
            return 6.0 * len(rows) * d * ff
        if kind == "block":
            O.dit_mlp_block(w["x"][rows], w["shift"], w["scale"], w["gate"], w["eps"], self.w1q, self.w1s,
                            w["b_up"], self.w2q, self.w2s, w["b2"], activation=self.cfg["activation"])
            return (6.0 if self.cfg["activation"] == "swiglu" else 4.0) * len(rows) * d * ff
        if kind == "up":
            xq, xs = O.quantize_bf16(w["x"][rows])
            g = O.up_projection(xq, xs, self.w1q, self.w1s, w["b"])
            O.quantize_f32(g.astype(np.float32))
            return 2.0 * len(rows) * d * ff
        if kind == "attn_in":
            a = O.rms_norm_modulate(w["x"][rows], w["shift"], w["scale"], w["eps"])
            xq, xs = O.quantize_f32(a.astype(np.float32))
            O.gemm(xq, xs, self.w1q, self.w1s, w["b"])
            return 2.0 * len(rows) * d * ff
        if kind == "attn_out":
            xq, xs = O.quantize_bf16(w["a"][rows])
            O.gate_residual(O.gemm(xq, xs, self.w1q, self.w1s, w["b"]), w["gate"], w["x"][rows])
            return 2.0 * len(rows) * d * ff
        if kind in ("gemm", "qkv"):
            xq, xs = O.quantize_bf16(w["x"][rows])
            O.gemm(xq, xs, self.w1q, self.w1s, w["b"])
            return 2.0 * len(rows) * d * ff
        z = w["x_f32"][rows % w["x_f32"].shape[0]]
        hq, hs = O.quantize_f32(O.gelu_tanh(z.astype(np.float64)).astype(np.float32))
        O.down_projection(hq, hs, self.w2q, self.w2s, w["b"])
        return 2.0 * len(rows) * d * ff


def _grow_sample(ow, rng, M: int, target_s: float):
    """Doubles the row sample (from 16) until one oracle step on it takes at least
    target_s / 2 (or covers all M rows); returns (rows, seconds, flops) of that step.
    A step has a fixed cost (the oracle dequantizes its weights every time), so a
    small calibration sample would over-estimate the cost of a row."""
    n = 16
    while True:
        rows = np.sort(rng.choice(M, size=min(n, M), replace=False))
        t0 = time.perf_counter()
        flops = ow.step(rows)
        dt = time.perf_counter() - t0
        if dt >= target_s / 2 or n >= M:
            return rows, dt, flops
        n *= 2


def cpu_baseline(cfg: dict, budget_s: float) -> dict:
    """The oracle, as it stands. The single-GEMM workload and the M = 4096
    up-projection are timed whole; the larger workloads on a bounded row sample,
    whose time is extrapolated linearly in M to the whole workload (the oracle's
    cost per token row is constant once its weights are quantized) and labelled so."""
    ow = OracleWorkload(cfg, sample_rows=64)
    rng = np.random.default_rng(0)
    M = cfg["M"]
    ow.step(rng.integers(0, M, 8))   # warm the thread pools
    whole = cfg["kind"] in ("gemm", "up")
    if whole:
        rows = np.arange(M)
        t0 = time.perf_counter()
        flops = ow.step(rows)
        dt = time.perf_counter() - t0
    else:
        rows, dt, flops = _grow_sample(ow, rng, M, budget_s)
    n = len(rows)
    out = {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": _cores(), "cpu_model": _cpu_model(),
           "kind": "oracle", "seconds": dt,
           "sample": (f"all {M} token rows of the workload" if whole else f"{n} of {M} token rows of the same "
                      f"workload") + " (weights quantized by the oracle beforehand, untimed); fp64 numpy + "
                                     "brute-force E2M3 search",
           "extrapolated": not whole,
           "full_workload_s": dt * M / n}
    if not whole:
        out["rule"] = (f"full_workload_s = seconds x {M} / {n}: linear in the token count M; value is the "
                       f"sample's own rate")
    return out


def run_reference(args) -> dict | None:
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    cfg = CONFIGS[args.config]
    ow = OracleWorkload(cfg, sample_rows=64)
    rng = np.random.default_rng(1)
    M = cfg["M"]
    ow.step(rng.integers(0, M, 4))   # warm the thread pools
    total_budget = args.cpu_budget * 4
    rows_per_step = len(_grow_sample(ow, rng, M, total_budget / max(1, args.steps + args.warmup))[0])
    for _ in range(args.warmup):
        ow.step(rng.integers(0, M, rows_per_step))
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flops += ow.step(rng.integers(0, M, rows_per_step))
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    sample = (f"{rows_per_step} random token rows of {M} per step (weights quantized by the oracle "
              f"beforehand, untimed)")
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded numpy PCG64, BF16 RNE; random-init weights)",
        "config": {"workload": cfg["workload"], "M_per_gpu": M, "d": cfg["d"], "ff": cfg["ff"]},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _cores(), "cpu_model": _cpu_model(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="full_mlp", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle CPU work for the baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="quantize all activations in their own kernel before the GEMM (the timed step's "
                         "single-GEMM stages only; mx_mlp always quantizes inside its up-projection)")
    ap.add_argument("--no-split", action="store_true",
                    help="run the GEMMs without the split tail (the same work, tiles whole; for comparison)")
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back steps after the timed region (the sustained leg; 0: none)")
    ap.add_argument("--copies", type=int, default=2,
                    help="independent input copies rotated between steps (2 keeps L2 cold; 1 for profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if line is not None:
        print(json.dumps(line))
    world, _, _ = dist_env()
    if world > 1 and args.impl != "reference":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
