#!/usr/bin/env python
"""Throughput of the INT4-KV attention hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
quantize-on-append of the new K/V rows, split-KV decode with its fused
in-SRAM dequantization, and the log-sum-exp combine (prefill workload: the
append of all prompt rows, then causal prefill).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   (the float64 oracle on host cores)

Prints ONE JSON line (rank 0).  Inputs are seeded synthetic data resident in
HBM before the timed region; L2 reuse across steps is defeated by rotating
through enough cache copies to exceed 4x the L2 size.  Steps run from CUDA
graphs of the public-API calls; the device time comes from CUDA events on
the launching stream.  `e2e` repeats the measurement through the same calls
with pinned host buffers copied in and the output copied out every step.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "int4-KV decode attn: KV GB/s (% of HBM peak); prefill TFLOP/s (% of peak)"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default="gqa_decode")
    p.add_argument("--splits", type=int, default=-1, help="decode split count (-1: workload default, 0: auto)")
    p.add_argument("--secondary", type=int, default=1, help="also time long_decode and causal_prefill")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU budget of the oracle baseline")
    p.add_argument("--e2e-steps", type=int, default=50)
    return p.parse_args(argv)


# ----------------------------------------------------------------- peaks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


# ------------------------------------------------------------ distributed

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(backend):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def reduce_max(x: float, device=None) -> float:
    """Max of a scalar over ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_per_rank: float, device=None):
    """Whole-job throughput: units summed over ranks / slowest rank's time."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
    t = reduce_max(seconds_per_rank, device)
    if world > 1:
        u = torch.tensor([float(units_per_rank)], dtype=torch.float64, device=device)
        dist.all_reduce(u)
        units = float(u.item())
    else:
        units = float(units_per_rank)
    return units / t, t, world


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(self.NAMES, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------- profile summaries

def source_digest(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "quantized_kv_attention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_file: str, digest: str, units: float):
    """DRAM bytes per launch from a committed ncu summary, scaled to `units`
    (the summary's `units_per_launch`), or None if the kernel changed since."""
    path = os.path.join(ROOT, "profiles", summary_file)
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = dict(re.findall(r"^(\w+)\s*=\s*(\S+)\s*$", text, flags=re.M))
    if fields.get("source_sha") != digest or "dram_bytes_per_launch" not in fields:
        return None
    per = float(fields["dram_bytes_per_launch"])
    base = float(fields.get("units_per_launch", units) or units)
    return per * units / base
