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
    p.add_argument("--workload", default="long_decode")
    p.add_argument("--splits", type=int, default=-1, help="decode split count (-1: workload default, 0: auto)")
    p.add_argument("--secondary", type=int, default=1,
                   help="with the long_decode headline, also time the other workloads as secondary lines")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU budget of the oracle baseline")
    p.add_argument("--e2e-steps", type=int, default=50)
    p.add_argument("--soak", type=float, default=1.0, help="seconds of the step loop before timing (clock samples)")
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


# ----------------------------------------------------------- GPU workloads

def _l2_bytes(torch, device):
    try:
        return int(torch.cuda.get_device_properties(device).L2_cache_size)
    except Exception:
        return 126 * 2**20


def _fill_contiguous(qa, torch, cache, B, Hkv, N, D, seed, device, outliers=None, oscale=10.0):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    for b in range(B):
        sub = qa.KvCache(cache.k_codes[b:b + 1], cache.k_scales[b:b + 1], cache.v_codes[b:b + 1],
                         cache.v_scales[b:b + 1], D, Hkv, capacity=cache.capacity)
        k = torch.randn(1, Hkv, N, D, device=device, generator=g)
        if outliers is not None:
            for h in range(Hkv):
                k[0, h, :, torch.as_tensor(outliers[h], device=device)] *= oscale
        v = torch.randn(1, Hkv, N, D, device=device, generator=g)
        qa.quantize_kv(k, v, sub)
        del k, v


def _graph(torch, fn):
    """Capture fn() (public-API calls) into a CUDA graph after one eager run."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _timed_graphs(torch, steps, enqueue_steps, enqueue_inner, inner_count, gpu_index,
                  period=1, soak_s=1.0, chunk=256):
    """Time exactly `steps` steps, replayed from CUDA graphs of the public-API
    calls (so the host never starves the GPU), between a barrier and a
    synchronize on both sides, with CUDA events on the launching stream.

    enqueue_steps(n) enqueues n consecutive steps starting from rotation slot
    0 (period = rotation length); enqueue_inner(n) enqueues n back-to-back
    launches of the dominant kernel alone, timed the same way to give its mean
    launch duration.  Clocks are sampled over a soak of the same graphs right
    before the timed region and over the region itself."""
    S = min(steps, max(period, chunk // period * period))
    g_main = _graph(torch, lambda: enqueue_steps(S))
    rem = steps % S
    g_rem = _graph(torch, lambda: enqueue_steps(rem)) if rem else None
    g_inner = _graph(torch, lambda: enqueue_inner(inner_count))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    i0, i1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_index)
    with sampler:
        t0 = time.time()
        while time.time() - t0 < soak_s:
            g_main.replay()
            torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        start.record()
        for _ in range(steps // S):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record()
        torch.cuda.synchronize()
        barrier()
        reps = max(1, int(math.ceil(2 * steps / max(1, inner_count))))
        g_inner.replay()
        torch.cuda.synchronize()
        i0.record()
        for _ in range(reps):
            g_inner.replay()
        i1.record()
        torch.cuda.synchronize()
    return start.elapsed_time(end), i0.elapsed_time(i1) / (reps * inner_count), sampler.summary()


def workload_config(name, splits=None, scale=None):
    """The `config` object both arms print for a workload."""
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    D = cfg["D"]
    out = {"workload": name}
    for key in ("B", "Hq", "Hkv", "D", "Nq", "Nk", "len_lo", "len_hi", "page", "outliers", "seed"):
        if key in cfg:
            out[key] = cfg[key]
    out["softmax_scale"] = 1.0 / math.sqrt(D) if scale is None else scale
    if cfg["kind"] == "prefill":
        out["causal"] = True
        out["flops_per_step"] = prefill_flops(cfg["B"], cfg["Hq"], cfg["Nq"], cfg["Nk"], D, True)
        out["l2"] = "inputs larger than L2: Q and O are 134 MB each per step"
    else:
        if splits is None:
            splits = 152 if name == "long_decode" else 0
        out["splits"] = "auto" if splits == 0 else splits
        out["l2"] = ("KV-cache copies rotate but stay L2-resident (17 KB each): a latency figure"
                     if name == "single_head_decode" else "rotating KV-cache copies totalling more than 4x L2")
        if cfg["kind"] == "paged":
            lens, _, _ = wl.paged_layout(cfg["seed"], cfg["B"], cfg["len_lo"], cfg["len_hi"], cfg["page"])
            out["kv_bytes_per_step"] = int(lens.sum()) * cfg["Hkv"] * (D + 4)
        else:
            out["kv_bytes_per_step"] = cfg["B"] * cfg["Hkv"] * cfg["Nk"] * (D + 4)
    out["step"] = ("append all K/V rows (quantize) + causal prefill" if cfg["kind"] == "prefill"
                   else "append one K/V row per sequence + split-KV decode (one fused launch) + merge")
    return out


def run_decode(name, args, device, gpu_index, rank, splits=None, scale=None, e2e=True):
    """One qattn_decode_append step per timed step (append one K/V row per
    sequence, attend, merge).  splits / scale override the workload's split
    count (152 for long_decode, else automatic) and softmax scale 1/sqrt(D)."""
    import torch
    import quantized_kv_attention_gb300 as qa
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    B, Hq, Hkv, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"]
    paged = cfg["kind"] == "paged"
    seed = cfg["seed"] + 1000 * rank
    if splits is None:
        splits = args.splits if args.splits >= 0 else (152 if name == "long_decode" else 0)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    torch.manual_seed(seed)
    if paged:
        lens, table, P = wl.paged_layout(cfg["seed"], B, cfg["len_lo"], cfg["len_hi"], cfg["page"])
        max_len = int(cfg["len_hi"])
        kv_bytes = int(lens.sum()) * Hkv * (D + 4)
    else:
        Nk = cfg["Nk"]
        lens = [Nk] * B
        max_len = Nk
        kv_bytes = B * Hkv * Nk * (D + 4)
    # a 17 KB cache cannot leave L2; 64 copies bound the set-up of a latency figure
    copies = min(max(1, math.ceil(4 * _l2_bytes(torch, device) / kv_bytes)), 64)
    caches = []
    for r in range(copies):
        if paged:
            c = qa.KvCache.paged(P, Hkv, D, torch.from_numpy(table), device=device)
            g = torch.Generator(device=device)
            g.manual_seed(seed * 31 + r)
            for b, n in enumerate(lens):
                sub = qa.KvCache(c.k_codes, c.k_scales, c.v_codes, c.v_scales, D, Hkv,
                                 page_table=c.page_table[b:b + 1], num_pages=P)
                k = torch.randn(1, Hkv, int(n), D, device=device, generator=g)
                v = torch.randn(1, Hkv, int(n), D, device=device, generator=g)
                qa.quantize_kv(k, v, sub)
        else:
            c = qa.KvCache.contiguous(B, Hkv, Nk, D, device=device)
            oc = wl.outlier_channels(cfg["seed"], Hkv, D, cfg["outliers"]) if cfg.get("outliers") else None
            _fill_contiguous(qa, torch, c, B, Hkv, Nk, D, seed * 31 + r, device, oc, cfg.get("outlier_scale", 1.0))
        caches.append(c)
    torch.cuda.synchronize()
    # lengths after the append: the new row of sequence b is token lens[b] - 1
    sl = torch.tensor([int(x) for x in lens], dtype=torch.int32, device=device)
    q = torch.randn(B, Hq, D, device=device).half()
    new_k = torch.randn(B, Hkv, D, device=device)
    new_v = torch.randn(B, Hkv, D, device=device)
    out = torch.empty(B, Hq, D, dtype=torch.float16, device=device)
    ws_bytes = qa.decode_workspace_size(B, Hq, Hkv, D, max_len, splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=device)
    launches = 1 + (1 if ws_bytes > 0 else 0)

    def step(r):  # append + attend, one qattn_decode_append call
        qa.decode_append(q, new_k, new_v, caches[r], sl, max_len, scale, splits, workspace=ws, out=out)

    def enqueue_steps(n):
        for i in range(n):
            step(i % copies)

    enqueue_inner = enqueue_steps

    enqueue_steps(max(args.warmup, 1))
    torch.cuda.synchronize()
    inner_count = max(copies, 64 // copies * copies)
    total_ms, dec_ms, clocks = _timed_graphs(torch, args.steps, enqueue_steps, enqueue_inner, inner_count,
                                             gpu_index, period=copies, soak_s=args.soak)
    value, tmax, world = aggregate(kv_bytes * args.steps / 1e9, total_ms / 1e3, device)

    # e2e: every step copies its inputs (q and the new K/V rows, packed in one
    # pinned host buffer) to the device, makes the public call and copies the
    # output back to pinned host memory; the steps are replayed from a CUDA
    # graph of those three operations, as a serving loop would run them
    def _off(n):
        return (n + 255) // 256 * 256
    q_bytes, kv_row_bytes = q.numel() * 2, new_k.numel() * new_k.element_size()
    k_off = _off(q_bytes)
    v_off = k_off + _off(kv_row_bytes)
    h_in = torch.empty(v_off + kv_row_bytes, dtype=torch.uint8).pin_memory()
    h_in[:q_bytes].copy_(q.cpu().view(torch.uint8).reshape(-1))
    h_in[k_off:k_off + kv_row_bytes].copy_(new_k.cpu().view(torch.uint8).reshape(-1))
    h_in[v_off:v_off + kv_row_bytes].copy_(new_v.cpu().view(torch.uint8).reshape(-1))
    d_in = torch.empty_like(h_in, device=device)
    q_d = d_in[:q_bytes].view(torch.float16).view(q.shape)
    k_d = d_in[k_off:k_off + kv_row_bytes].view(new_k.dtype).view(new_k.shape)
    v_d = d_in[v_off:v_off + kv_row_bytes].view(new_v.dtype).view(new_v.shape)
    out_h = torch.empty(B, Hq, D, dtype=torch.float16).pin_memory()

    def e2e_step(i):
        d_in.copy_(h_in, non_blocking=True)
        qa.decode_append(q_d, k_d, v_d, caches[i % copies], sl, max_len, scale, splits, workspace=ws, out=out)
        out_h.copy_(out, non_blocking=True)

    e2e_val, e2e_done = None, 0
    if args.e2e_steps > 0 and e2e:
        n_graph = copies * max(1, 16 // copies)
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            with torch.cuda.graph(gr, stream=cs):
                for i in range(n_graph):
                    e2e_step(i)
        torch.cuda.synchronize()
        reps = max(1, args.e2e_steps // n_graph)
        gr.replay()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            gr.replay()
        e1.record()
        torch.cuda.synchronize()
        assert torch.equal(out_h.to(device), out)  # the last step's output reached the host
        e2e_done = reps * n_graph
        e2e_val, _, _ = aggregate(kv_bytes * e2e_done / 1e9, e0.elapsed_time(e1) / 1e3, device)
        e2e_val = round(e2e_val, 2)
    h2d = q.numel() * 2 + new_k.numel() * 4 + new_v.numel() * 4
    d2h = out.numel() * 2

    peaks, pk_src = measured_peaks()
    achieved = kv_bytes / (dec_ms / 1e3) / 1e9
    traffic = profiled_traffic(f"decode_{name}_ncu.txt", source_digest("decode.cu", "ptx.cuh", "quant_row.cuh"),
                               kv_bytes)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(tmax * 1e3 / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": workload_config(name, splits, scale),
        "setup": {"cache_copies": copies, "rotation_mib": round(copies * kv_bytes / 2**20),
                  "parallelism": f"replicas x{world}", "timing": "CUDA graphs of the API calls"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": traffic, "kernel": "decode with fused append + merge (one qattn_decode_append call)",
                     "peak_source": pk_src, "us_per_launch": round(dec_ms * 1e3, 3)},
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_done,
                "timing": "CUDA graph of the step: one H2D copy of q and the new K/V rows from pinned host "
                          "memory, the qattn_decode_append call, one D2H copy of the output"},
        "gpu_launches": launches * args.steps,
        "clocks": clocks,
    }
    del caches
    torch.cuda.empty_cache()
    return res


def prefill_flops(B, Hq, Nq, Nk, D, causal=True):
    """4 * D flops per visible (query, key) pair (QK^T and PV)."""
    if causal:
        shift = Nk - Nq
        pairs = sum(min(Nk, i + shift + 1) for i in range(Nq))
    else:
        pairs = Nq * Nk
    return 4.0 * D * B * Hq * pairs


def run_decode_lowbit(name, args, device, gpu_index, rank, bits=3):
    """A contiguous decode workload's shape with an INT3 cache (ten 3-bit
    values per 32-bit word, 52 + 52 + 2 + 2 bytes per (token, kv-head) at
    D = 128) or an INT2 cache (sixteen 2-bit values per word, 32 + 32 + 2 + 2
    bytes).  A step appends one K/V row per sequence (qattn_quantize_kv at
    position seq_lens[b] - 1) and runs one qattn_decode; CUDA graphs of the
    API calls, rotating cache copies larger than 4x L2; the roofline times the
    decode call alone."""
    import torch
    import quantized_kv_attention_gb300 as qa
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    B, Hq, Hkv, D, Nk = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Nk"]
    splits = 152 if name == "long_decode" else 0
    seed = cfg["seed"] + 1000 * rank
    scale = 1.0 / math.sqrt(D)
    tok_bytes = 52 if bits == 3 else D * bits // 8
    row_bytes = 2 * tok_bytes + 4
    kv_bytes = B * Hkv * Nk * row_bytes
    copies = max(1, math.ceil(4 * _l2_bytes(torch, device) / kv_bytes))
    caches = []
    g = torch.Generator(device=device)
    for r in range(copies):
        c = qa.KvCache.contiguous(B, Hkv, Nk, D, device=device, code_bits=bits)
        g.manual_seed(seed * 31 + r)
        for b in range(B):
            sub = qa.KvCache(c.k_codes[b:b + 1], c.k_scales[b:b + 1], c.v_codes[b:b + 1], c.v_scales[b:b + 1], D,
                             Hkv, capacity=c.capacity, code_bits=bits)
            qa.quantize_kv(torch.randn(1, Hkv, Nk, D, device=device, generator=g),
                           torch.randn(1, Hkv, Nk, D, device=device, generator=g), sub)
        caches.append(c)
    torch.cuda.synchronize()
    sl = torch.full((B,), Nk, dtype=torch.int32, device=device)
    start_pos = sl - 1
    q = torch.randn(B, Hq, D, device=device).half()
    new_k = torch.randn(B, Hkv, 1, D, device=device)
    new_v = torch.randn(B, Hkv, 1, D, device=device)
    out = torch.empty(B, Hq, D, dtype=torch.float16, device=device)
    ws = torch.empty(max(qa.decode_workspace_size(B, Hq, Hkv, D, Nk, splits), 16), dtype=torch.uint8, device=device)

    def attend(r):
        qa.decode(q, caches[r], sl, Nk, scale, splits, workspace=ws, out=out)

    def enqueue_steps(n):
        for i in range(n):
            qa.quantize_kv(new_k, new_v, caches[i % copies], start_pos)
            attend(i % copies)

    def enqueue_inner(n):
        for i in range(n):
            attend(i % copies)

    enqueue_steps(max(args.warmup, 1))
    torch.cuda.synchronize()
    inner_count = max(copies, 64 // copies * copies)
    total_ms, dec_ms, clocks = _timed_graphs(torch, args.steps, enqueue_steps, enqueue_inner, inner_count,
                                             gpu_index, period=copies, soak_s=args.soak)
    value, tmax, world = aggregate(kv_bytes * args.steps / 1e9, total_ms / 1e3, device)
    peaks, pk_src = measured_peaks()
    achieved = kv_bytes / (dec_ms / 1e3) / 1e9
    res = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(tmax * 1e3 / args.steps, 5),
        "steps": args.steps,
        "config": {"workload": f"{name}_int{bits}", "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "Nk": Nk, "code_bits": bits,
                   "splits": splits, "seed": cfg["seed"], "softmax_scale": scale, "kv_bytes_per_step": kv_bytes,
                   "l2": "rotating KV-cache copies totalling more than 4x L2",
                   "step": f"append one K/V row per sequence (INT{bits} quantize) + split-KV decode + merge"},
        "setup": {"cache_copies": copies, "parallelism": f"replicas x{world}",
                  "timing": "CUDA graphs of the API calls"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(f"decode_{name}_int{bits}_ncu.txt",
                                                 source_digest("decode.cu", "ptx.cuh", "quant_row.cuh"), kv_bytes),
                     "kernel": f"decode + merge (one qattn_decode call, INT{bits} cache)", "peak_source": pk_src,
                     "us_per_launch": round(dec_ms * 1e3, 3)},
        "clocks": clocks,
    }
    del caches
    torch.cuda.empty_cache()
    return res


def run_decode_flashq(name, args, device, gpu_index, rank):
    """A decode workload's shape with the decode buffer (qattn_flashq_*):
    the INT4 cache holds Nk - 64 rows, and a cycle of 64 steps appends one
    K/V row per (sequence, kv-head) into the int8 buffer, decodes over the
    cached rows, merges the buffered rows in, and finally flushes the buffer
    into the cache (every replay rewrites the same 64 cache rows, so replays
    are identical).  Timed per step over whole cycles, CUDA graphs of the API
    calls, rotating cache copies larger than 4x L2."""
    import torch
    import quantized_kv_attention_gb300 as qa
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    B, Hq, Hkv, D, Nk = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Nk"]
    splits = 152 if name == "long_decode" else 0
    nb = qa.FLASHQ_ROWS
    Lc = Nk - nb
    seed = cfg["seed"] + 1000 * rank
    scale = 1.0 / math.sqrt(D)
    cached_bytes = B * Hkv * Lc * (D + 4)
    buf_bytes = B * Hkv * (nb + 1) / 2 * (2 * D + 4)  # mean rows buffered at a step, int8 K and V
    kv_bytes = cached_bytes + buf_bytes
    copies = max(1, math.ceil(4 * _l2_bytes(torch, device) / cached_bytes))
    caches, bufs = [], []
    lens = torch.full((B,), Lc, dtype=torch.int32, device=device)
    for r in range(copies):
        c = qa.KvCache.contiguous(B, Hkv, Nk, D, device=device)
        oc = wl.outlier_channels(cfg["seed"], Hkv, D, cfg["outliers"]) if cfg.get("outliers") else None
        _fill_contiguous(qa, torch, c, B, Hkv, Lc, D, seed * 31 + r, device, oc, cfg.get("outlier_scale", 1.0))
        f = qa.FlashqBuffer.create(B, Hkv, D, device=device)
        qa.flashq_init(f, c, lens)
        caches.append(c)
        bufs.append(f)
    torch.cuda.synchronize()
    q = torch.randn(B, Hq, D, device=device).half()
    new_k = torch.randn(B, Hkv, D, device=device)
    new_v = torch.randn(B, Hkv, D, device=device)
    out = torch.empty(B, Hq, D, dtype=torch.float16, device=device)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=device)
    ws = torch.empty(max(qa.decode_workspace_size(B, Hq, Hkv, D, Lc, splits), 16), dtype=torch.uint8, device=device)

    def cycle(r):
        for _ in range(nb):
            qa.flashq_append(new_k, new_v, bufs[r])
            qa.decode(q, caches[r], lens, Lc, scale, splits, workspace=ws, out=out, lse=lse)
            qa.flashq_attend(q, bufs[r], scale, out, lse)
        qa.flashq_flush(bufs[r], caches[r], lens)

    for r in range(copies):
        cycle(r)
    torch.cuda.synchronize()
    g = _graph(torch, lambda: [cycle(r) for r in range(copies)])
    reps = max(1, args.steps // (nb * copies))
    sampler = ClockSampler(gpu_index)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with sampler:
        g.replay()
        torch.cuda.synchronize()
        barrier()
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        barrier()
    steps = reps * nb * copies
    value, tmax, world = aggregate(kv_bytes * steps / 1e9, e0.elapsed_time(e1) / 1e3, device)
    res = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(tmax * 1e3 / steps, 5), "steps": steps,
        "config": {"workload": f"{name}_flashq", "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "Nk": Nk,
                   "cached_rows": Lc, "buffer_rows": nb, "seed": cfg["seed"], "softmax_scale": scale,
                   "kv_bytes_per_step": int(kv_bytes),
                   "l2": "rotating KV-cache copies totalling more than 4x L2",
                   "step": "append one K/V row per sequence into the int8 buffer + split-KV decode over the "
                           "cached rows + merge of the buffered rows; a flush into the INT4 cache every 64 steps"},
        "setup": {"cache_copies": copies, "parallelism": f"replicas x{world}",
                  "timing": "CUDA graphs of whole 64-step cycles of the API calls"},
        "clocks": sampler.summary(),
    }
    del caches, bufs
    torch.cuda.empty_cache()
    return res


def run_prefill(name, args, device, gpu_index, rank, steps=None):
    import torch
    import quantized_kv_attention_gb300 as qa
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    B, Hq, Hkv, D, Nq, Nk = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Nq"], cfg["Nk"]
    steps = steps or args.steps
    scale = 1.0 / math.sqrt(D)
    g = torch.Generator(device=device)
    g.manual_seed(cfg["seed"] + 1000 * rank)
    k = torch.randn(B, Hkv, Nk, D, device=device, generator=g)
    v = torch.randn(B, Hkv, Nk, D, device=device, generator=g)
    q = torch.randn(B, Hq, Nq, D, device=device, generator=g).half()
    out = torch.empty_like(q)
    cache = qa.KvCache.contiguous(B, Hkv, Nk, D, device=device)
    flops = prefill_flops(B, Hq, Nq, Nk, D, True)

    def enqueue_steps(n):
        for _ in range(n):
            qa.quantize_kv(k, v, cache)
            qa.prefill(q, cache, Nk, scale, True, out=out)

    def enqueue_inner(n):
        for _ in range(n):
            qa.prefill(q, cache, Nk, scale, True, out=out)

    enqueue_steps(max(args.warmup, 1))
    torch.cuda.synchronize()
    total_ms, pf_ms, clocks = _timed_graphs(torch, steps, enqueue_steps, enqueue_inner, 2, gpu_index,
                                            chunk=8, soak_s=args.soak)
    value, tmax, world = aggregate(flops * steps / 1e12, total_ms / 1e3, device)

    # e2e through the public API with pinned host buffers
    q_h, k_h, v_h = q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory()
    out_h = torch.empty(q.shape, dtype=torch.float16).pin_memory()
    e2e_steps = min(args.e2e_steps, 10)

    def e2e_step():
        q.copy_(q_h, non_blocking=True)
        k.copy_(k_h, non_blocking=True)
        v.copy_(v_h, non_blocking=True)
        qa.quantize_kv(k, v, cache)
        qa.prefill(q, cache, Nk, scale, True, out=out)
        out_h.copy_(out, non_blocking=True)

    e2e_val = None
    if e2e_steps > 0:
        e2e_step()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(e2e_steps):
            e2e_step()
        e1.record()
        torch.cuda.synchronize()
        e2e_val, _, _ = aggregate(flops * e2e_steps / 1e12, e0.elapsed_time(e1) / 1e3, device)
        e2e_val = round(e2e_val, 2)

    peaks, pk_src = measured_peaks()
    achieved = flops / (pf_ms / 1e3) / 1e12
    # the prefill kernel is timed alone in a region of milliseconds: the burst peak applies
    peak = peaks["bf16_tflops"]
    peak_sus = peaks.get("bf16_tflops_sustained", peak)
    traffic = profiled_traffic(f"prefill_{name}_ncu.txt", source_digest("prefill.cu", "ptx.cuh", "umma.cuh"), flops)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(tmax * 1e3 / steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": workload_config(name),
        "setup": {"parallelism": f"replicas x{world}", "timing": "CUDA graphs of the API calls"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "prefill", "peak_source": pk_src + " bf16 burst (fp16 runs at the bf16 rate)",
                     "frac_of_sustained": round(achieved / peak_sus, 4),
                     "ms_per_launch": round(pf_ms, 4)},
        "e2e": {"value": e2e_val, "unit": "TFLOP/s",
                "h2d_bytes_per_step": q.numel() * 2 + k.numel() * 4 + v.numel() * 4,
                "d2h_bytes_per_step": out.numel() * 2, "steps": e2e_steps},
        "gpu_launches": 2 * steps,
        "clocks": clocks,
    }
    del k, v, q, out, cache
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ CPU oracle

def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_step_factory(name, units=None):
    """An oracle step over a bounded sample of `name`; returns (step_fn,
    units of the metric per step, unit, description)."""
    import numpy as np
    from oracle import attention as att
    from oracle import codec
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    D, Hq, Hkv = cfg["D"], cfg["Hq"], cfg["Hkv"]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D)
    if cfg["kind"] == "prefill":
        Nq, Nk = cfg["Nq"], cfg["Nk"]
        rows = units or 256
        k = wl.kv_slice(cfg["seed"], "k", 0, 0, Nk, D).numpy()[None, None]
        v = wl.kv_slice(cfg["seed"], "v", 0, 0, Nk, D).numpy()[None, None]
        q = wl.queries(cfg["seed"], 1, 1, Nq, D).numpy()[:, :, Nq - rows:]
        flops = prefill_flops(1, 1, rows, Nk, D, True)

        def step():
            pk, sk = codec.quantize_pack(k)
            pv, sv = codec.quantize_pack(v)
            att.attention_quantized(q, pk, sk, pv, sv, scale, True)
        desc = f"one head, the last {rows} causal query rows of Nq=Nk={Nk} (append of that head's K/V included)"
        return step, flops / 1e12, "TFLOP/s", desc
    if cfg["kind"] == "paged":
        lens, _, _ = wl.paged_layout(cfg["seed"], cfg["B"], cfg["len_lo"], cfg["len_hi"], cfg["page"])
        N = int(lens[0])
    else:
        N = cfg["Nk"]
    # a bounded sample: whole kv-heads of sequence 0, about 20 MB of cache at most
    heads = units or max(1, min(Hkv, int(20e6 // (N * (D + 4)))))
    oc = wl.outlier_channels(cfg["seed"], Hkv, D, cfg["outliers"]) if cfg.get("outliers") else None
    k = np.stack([wl.kv_slice(cfg["seed"], "k", 0, h, N, D, oc, cfg.get("outlier_scale", 1.0)).numpy()
                  for h in range(heads)])[None]
    v = np.stack([wl.kv_slice(cfg["seed"], "v", 0, h, N, D).numpy() for h in range(heads)])[None]
    pk, sk = codec.quantize_pack(k)
    pv, sv = codec.quantize_pack(v)
    q = wl.queries(cfg["seed"], 1, heads * G, D).numpy()[:, :, None]
    new = k[:, :, -1:].copy()

    def step():
        codec.quantize_pack(new)
        codec.quantize_pack(new)
        att.attention_quantized(q, pk, sk, pv, sv, scale)
    desc = f"sequence 0, {heads} of {Hkv} kv-heads x {N} tokens (append of one row + decode)"
    return step, heads * N * (D + 4) / 1e9, "GB/s", desc


def cpu_baseline(name, budget_s):
    step, units, unit, desc = oracle_step_factory(name)
    step()
    t0 = time.perf_counter()
    n = 0
    while True:
        step()
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(units * n / dt, 4), "unit": unit, "cores": _cores(), "kind": "oracle",
            "sample": f"{desc}; {n} steps in {dt:.1f} s; numpy float64, BLAS threads = all cores"}


def run_reference(args):
    """The float64 oracle on the host cores, as the reference arm."""
    name = args.workload
    kind_prefill = name == "causal_prefill"
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))   # seconds per step
    probe, _, _, _ = oracle_step_factory(name, units=1 if not kind_prefill else 64)
    t0 = time.perf_counter()
    probe()
    t1 = time.perf_counter() - t0
    base = 64 if kind_prefill else 1
    units = max(base, min((8192 if kind_prefill else 8), int(base * budget / max(t1, 1e-6))))
    if kind_prefill:
        units = max(64, units // 64 * 64)
    step, per_step, unit, desc = oracle_step_factory(name, units=units)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt
    return {"metric": METRIC, "value": round(value, 4), "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": workload_config(name, None if args.splits < 0 else args.splits),
            "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": _cores(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def run_quantize(name, args, device, gpu_index, rank):
    """qattn_quantize_kv alone (a1, quantize-on-append) on a prefill workload's
    K and V rows (fp32 in): GB/s of its algorithmic bytes, the fp32 rows read
    plus the INT4 codes and fp16 scales written, per (token, kv-head) row
    D*4 + D/2 + 2 bytes for each of K and V.  Rotating input copies larger
    than 2x L2; CUDA graphs of the API call, CUDA events on the stream."""
    import torch
    import quantized_kv_attention_gb300 as qa
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    B, Hkv, D, N = cfg["B"], cfg["Hkv"], cfg["D"], cfg["Nk"]
    rows = 2 * B * Hkv * N
    step_bytes = rows * (D * 4 + D // 2 + 2)
    in_bytes = rows * D * 4
    copies = max(2, math.ceil(2 * _l2_bytes(torch, device) / in_bytes))
    g = torch.Generator(device=device)
    g.manual_seed(cfg["seed"] + 1000 * rank)
    ks = [torch.randn(B, Hkv, N, D, device=device, generator=g) for _ in range(copies)]
    vs = [torch.randn(B, Hkv, N, D, device=device, generator=g) for _ in range(copies)]
    cache = qa.KvCache.contiguous(B, Hkv, N, D, device=device)

    def enqueue(n):
        for i in range(n):
            qa.quantize_kv(ks[i % copies], vs[i % copies], cache)

    enqueue(max(args.warmup, 1))
    torch.cuda.synchronize()
    steps = min(args.steps, 100)
    total_ms, one_ms, clocks = _timed_graphs(torch, steps, enqueue, enqueue, copies * max(1, 32 // copies),
                                             gpu_index, period=copies, soak_s=min(args.soak, 0.5))
    value, tmax, world = aggregate(step_bytes * steps / 1e9, total_ms / 1e3, device)
    peaks, pk_src = measured_peaks()
    achieved = step_bytes / (one_ms / 1e3) / 1e9
    res = {
        "value": round(value, 1), "unit": "GB/s", "ms_per_step": round(tmax * 1e3 / steps, 5), "steps": steps,
        "config": {"workload": f"{name}_quantize", "B": B, "Hkv": Hkv, "D": D, "rows_per_tensor": N,
                   "x_dtype": "fp32", "bytes_per_step": step_bytes,
                   "l2": "rotating input copies totalling more than 2x L2",
                   "step": "quantize all K and V rows of the prompt into the INT4 cache (one qattn_quantize_kv)"},
        "setup": {"input_copies": copies, "parallelism": f"replicas x{world}", "timing": "CUDA graphs of the API call"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(f"quantize_{name}_quantize_ncu.txt",
                                                 source_digest("quantize.cu", "quant_row.cuh", "ptx.cuh"), step_bytes),
                     "kernel": "quantize_kv",
                     "peak_source": pk_src, "us_per_launch": round(one_ms * 1e3, 3)},
        "clocks": clocks,
    }
    del ks, vs, cache
    torch.cuda.empty_cache()
    return res


def run_decode_pq(name, args, device, gpu_index, rank):
    """A contiguous decode workload's shape over a progressive cache
    (qattn_pq_quantize blocks of 64 tokens, qattn_decode_pq): per (token,
    kv-head) and tensor D/2 code bytes, per 64-token block and tensor a
    2D + 16 byte record.  A step is one qattn_decode_pq call (its blocks are
    appended 64 tokens at a time, not per step); CUDA graphs of the API call,
    rotating cache copies larger than 4x L2."""
    import torch
    import quantized_kv_attention_gb300 as qa
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    B, Hq, Hkv, D, Nk = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["Nk"]
    scale = 1.0 / math.sqrt(D)
    kv_bytes = 2 * B * Hkv * (Nk * D // 2 + (Nk // 64) * (2 * D + 16))
    copies = max(1, math.ceil(4 * _l2_bytes(torch, device) / kv_bytes))
    g = torch.Generator(device=device)
    g.manual_seed(cfg["seed"] + 1000 * rank + 5)
    caches = []
    for _ in range(copies):
        c = qa.PqCache.contiguous(B, Hkv, Nk, D, device=device)
        for b in range(B):
            sub = qa.PqCache(c.k_codes[b:b + 1], c.v_codes[b:b + 1], c.k_params[b:b + 1], c.v_params[b:b + 1], D, Hkv,
                             c.capacity)
            qa.pq_quantize(torch.randn(1, Hkv, Nk, D, device=device, generator=g),
                           torch.randn(1, Hkv, Nk, D, device=device, generator=g), sub)
        caches.append(c)
    torch.cuda.synchronize()
    sl = torch.full((B,), Nk, dtype=torch.int32, device=device)
    q = torch.randn(B, Hq, D, device=device, generator=g).half()
    out = torch.empty(B, Hq, D, dtype=torch.float16, device=device)
    ws = torch.empty(max(qa.decode_pq_workspace_size(B, Hq, Hkv, D, Nk, 0), 16), dtype=torch.uint8, device=device)

    def enqueue(n):
        for i in range(n):
            qa.decode_pq(q, caches[i % copies], sl, Nk, scale, 0, workspace=ws, out=out)

    enqueue(max(args.warmup, 1))
    torch.cuda.synchronize()
    inner = max(copies, 64 // copies * copies)
    total_ms, one_ms, clocks = _timed_graphs(torch, args.steps, enqueue, enqueue, inner, gpu_index, period=copies,
                                             soak_s=min(args.soak, 0.5))
    value, tmax, world = aggregate(kv_bytes * args.steps / 1e9, total_ms / 1e3, device)
    peaks, pk_src = measured_peaks()
    achieved = kv_bytes / (one_ms / 1e3) / 1e9
    res = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(tmax * 1e3 / args.steps, 5), "steps": args.steps,
        "config": {"workload": f"{name}_pq", "B": B, "Hq": Hq, "Hkv": Hkv, "D": D, "Nk": Nk, "softmax_scale": scale,
                   "kv_bytes_per_step": kv_bytes, "l2": "rotating KV-cache copies totalling more than 4x L2",
                   "step": "split-KV decode over progressive INT8 -> INT4 blocks (one qattn_decode_pq call)"},
        "setup": {"cache_copies": copies, "parallelism": f"replicas x{world}", "timing": "CUDA graphs of the API call"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": profiled_traffic(f"decode_pq_{name}_pq_ncu.txt",
                                                 source_digest("pq.cu", "quant_row.cuh", "ptx.cuh"), kv_bytes),
                     "kernel": "decode_pq + combine",
                     "peak_source": pk_src, "us_per_launch": round(one_ms * 1e3, 3)},
        "clocks": clocks,
    }
    del caches
    torch.cuda.empty_cache()
    return res


def run_compare(name, args, device, gpu_index, rank):
    """The comparison arms of "Quantized Cross-Attention ... In-SRAM
    Dequantization" §5.2-§5.3 on a workload's shape: attention over an FP16
    KV cache (qattn_decode_fp16 / qattn_prefill_fp16), and post-
    dequantization (qattn_dequantize_kv of the whole INT4 cache into FP16 in
    HBM, then the same FP16 call).  Returns two lines: the FP16 arm (GB/s of
    its FP16 K/V bytes for decode, TFLOP/s for prefill, with a roofline), and
    the post-dequantization arm (the workload's own metric, INT4 bytes or
    FLOP per step, so it compares with the fused line directly).  CUDA graphs
    of the API calls; FP16 caches rotate through copies larger than 4x L2
    when they fit in 16 GB."""
    import torch
    import quantized_kv_attention_gb300 as qa
    from quantized_kv_attention_gb300 import workloads as wl
    cfg = dict(wl.WORKLOADS[name])
    B, Hq, Hkv, D = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"]
    prefill = cfg["kind"] == "prefill"
    N = cfg["Nk"]
    scale = 1.0 / math.sqrt(D)
    peaks, pk_src = measured_peaks()
    g = torch.Generator(device=device)
    g.manual_seed(cfg["seed"] + 1000 * rank + 77)
    f16_bytes = 2 * B * Hkv * N * D * 2
    copies = max(1, min(math.ceil(4 * _l2_bytes(torch, device) / f16_bytes), int(16e9 // f16_bytes)))
    ks = [torch.randn(B, Hkv, N, D, device=device, generator=g).half() for _ in range(copies)]
    vs = [torch.randn(B, Hkv, N, D, device=device, generator=g).half() for _ in range(copies)]
    # the INT4 cache of the post-dequantization arm, and its FP16 copy
    cache = qa.KvCache.contiguous(B, Hkv, N, D, device=device)
    qa.quantize_kv(torch.randn(B, Hkv, N, D, device=device, generator=g),
                   torch.randn(B, Hkv, N, D, device=device, generator=g), cache)
    k16, v16 = torch.empty_like(ks[0]), torch.empty_like(vs[0])
    if prefill:
        Nq = cfg["Nq"]
        q = torch.randn(B, Hq, Nq, D, device=device, generator=g).half()
        out = torch.empty_like(q)
        work = prefill_flops(B, Hq, Nq, N, D, True)

        def arm16(i):
            qa.prefill_fp16(q, ks[i % copies], vs[i % copies], N, scale, True, out=out)

        def post(i):
            qa.dequantize_kv(cache, B, N, k16, v16)
            qa.prefill_fp16(q, k16, v16, N, scale, True, out=out)
    else:
        q = torch.randn(B, Hq, D, device=device, generator=g).half()
        out = torch.empty(B, Hq, D, dtype=torch.float16, device=device)
        sl = torch.full((B,), N, dtype=torch.int32, device=device)
        ws = torch.empty(max(qa.decode_fp16_workspace_size(B, Hq, Hkv, D, N, 0), 16), dtype=torch.uint8,
                         device=device)
        work = B * Hkv * N * (D + 4)

        def arm16(i):
            qa.decode_fp16(q, ks[i % copies], vs[i % copies], sl, N, scale, 0, workspace=ws, out=out)

        def post(i):
            qa.dequantize_kv(cache, B, N, k16, v16)
            qa.decode_fp16(q, k16, v16, sl, N, scale, 0, workspace=ws, out=out)

    steps = min(args.steps, 20 if prefill else 200)
    res = {}
    for arm, fn, per in (("fp16", arm16, copies), ("postdequant", post, 1)):
        def enqueue(n, fn=fn):
            for i in range(n):
                fn(i)
        enqueue(max(args.warmup, 1))
        torch.cuda.synchronize()
        total_ms, one_ms, clocks = _timed_graphs(torch, steps, enqueue, enqueue, per * max(1, 8 // per), gpu_index,
                                                 period=per, soak_s=min(args.soak, 0.5),
                                                 chunk=8 if prefill else 256)
        value, tmax, world = aggregate((work / 1e12 if prefill else work / 1e9) * steps, total_ms / 1e3, device)
        line = {"value": round(value, 2), "unit": "TFLOP/s" if prefill else "GB/s",
                "ms_per_step": round(tmax * 1e3 / steps, 5), "steps": steps,
                "config": {"workload": f"{name}_{arm}", "kv": "fp16" if arm == "fp16" else
                           "int4 dequantized to fp16 in HBM, then attended",
                           "l2": f"{per} rotating FP16 cache copies" if arm == "fp16" else "FP16 copy rewritten every step"},
                "clocks": clocks}
        if arm == "fp16":
            if prefill:
                ach = work / (one_ms / 1e3) / 1e12
                line["roofline"] = {"bound": "tensor", "achieved": round(ach, 1), "peak": peaks["bf16_tflops"],
                                    "unit": "TFLOP/s", "frac": round(ach / peaks["bf16_tflops"], 4),
                                    "ms_per_launch": round(one_ms, 4), "peak_source": pk_src}
            else:
                ach = f16_bytes / (one_ms / 1e3) / 1e9
                line["value"] = round(f16_bytes * steps / 1e9 / tmax, 2)
                line["roofline"] = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                                    "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                                    "traffic": profiled_traffic(f"decode16_{name}_fp16_ncu.txt",
                                                                source_digest("fp16kv.cu", "ptx.cuh"), f16_bytes),
                                    "us_per_launch": round(one_ms * 1e3, 3), "peak_source": pk_src}
                line["config"]["kv_bytes_per_step"] = f16_bytes
        res[arm] = line
    del ks, vs, cache, k16, v16
    torch.cuda.empty_cache()
    return res


def compact(res):
    """A secondary line's essentials: throughput, step time, roofline, clocks."""
    out = {k: res[k] for k in ("value", "unit", "ms_per_step") if k in res}
    cfg = res.get("config", {})
    out["config"] = {k: cfg[k] for k in ("workload", "splits", "softmax_scale", "kv_bytes_per_step",
                                        "bytes_per_step", "flops_per_step", "code_bits") if k in cfg}
    if "roofline" in res:
        r = res["roofline"]
        out["roofline"] = {k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic",
                                            "frac_of_sustained", "us_per_launch", "ms_per_launch") if k in r}
    if res.get("e2e", {}).get("value") is not None:
        out["e2e"] = {"value": res["e2e"]["value"], "unit": res["e2e"]["unit"]}
    if "clocks" in res:
        out["clocks"] = {k: res["clocks"].get(k) for k in ("sm_mhz", "reasons")}
    if "error" in res:
        out["error"] = res["error"]
    return out


def secondary_lines(args, device, gpu_index, rank):
    """Every other workload of the hot path, each timed like the headline."""
    sec = {}

    def add(key, fn):
        try:  # a secondary number: its failure must not take the others with it
            sec[key] = compact(fn())
        except Exception as e:  # reported, not hidden
            sec[key] = {"error": f"{type(e).__name__}: {e}"}

    add("gqa_decode", lambda: run_decode("gqa_decode", args, device, gpu_index, rank, splits=0))
    add("paged_decode", lambda: run_decode("paged_decode", args, device, gpu_index, rank, splits=0,
                                           e2e=False))
    add("paged_decode_scale1", lambda: run_decode("paged_decode", args, device, gpu_index, rank, splits=0,
                                                  scale=1.0, e2e=False))
    for n in (64, 128, 256):
        add(f"long_decode_splits{n}", lambda n=n: run_decode("long_decode", args, device, gpu_index, rank,
                                                             splits=n, e2e=False))
    add("single_head_decode", lambda: run_decode("single_head_decode", args, device, gpu_index, rank, splits=0,
                                                 e2e=False))
    add("long_decode_flashq", lambda: run_decode_flashq("long_decode", args, device, gpu_index, rank))
    add("long_decode_int3", lambda: run_decode_lowbit("long_decode", args, device, gpu_index, rank, 3))
    add("long_decode_int2", lambda: run_decode_lowbit("long_decode", args, device, gpu_index, rank, 2))
    add("long_decode_pq", lambda: run_decode_pq("long_decode", args, device, gpu_index, rank))
    add("causal_prefill", lambda: run_prefill("causal_prefill", args, device, gpu_index, rank,
                                              steps=min(args.steps, 50)))
    add("causal_prefill_quantize", lambda: run_quantize("causal_prefill", args, device, gpu_index, rank))
    for wname in ("long_decode", "gqa_decode", "causal_prefill"):
        try:
            for arm, line in run_compare(wname, args, device, gpu_index, rank).items():
                sec[f"{wname}_{arm}"] = compact(line)
        except Exception as e:  # reported, not hidden
            sec[f"{wname}_fp16"] = {"error": f"{type(e).__name__}: {e}"}
    return sec


VARIANTS = ("_int3", "_int2", "_flashq", "_quantize", "_fp16", "_postdequant", "_pq")


def run_workload(name, args, device, gpu_index, rank):
    """A workload by name: a base workload (the hot path's step), or a base
    name with a suffix for one secondary line on its shape (_int3, _int2:
    the low-bit caches; _flashq: the decode buffer; _quantize: the append
    kernel alone; _fp16, _postdequant: the comparison arms)."""
    from quantized_kv_attention_gb300 import workloads as wl
    suffix = next((v for v in VARIANTS if name.endswith(v)), "")
    base = name[: len(name) - len(suffix)]
    if base not in wl.WORKLOADS:
        raise SystemExit(f"unknown workload {name}")
    if suffix in ("_int3", "_int2"):
        res = run_decode_lowbit(base, args, device, gpu_index, rank, int(suffix[-1]))
    elif suffix == "_flashq":
        res = run_decode_flashq(base, args, device, gpu_index, rank)
    elif suffix == "_quantize":
        res = run_quantize(base, args, device, gpu_index, rank)
    elif suffix == "_pq":
        res = run_decode_pq(base, args, device, gpu_index, rank)
    elif suffix:
        res = run_compare(base, args, device, gpu_index, rank)[suffix[1:]]
    else:
        kind = wl.WORKLOADS[base]["kind"]
        res = (run_prefill if kind == "prefill" else run_decode)(base, args, device, gpu_index, rank)
    for key, val in (("metric", METRIC), ("n_gpus", 1), ("warmup", args.warmup), ("higher_is_better", True),
                     ("scaling", "weak"), ("vs_baseline", None), ("dtype", "f16"), ("data", "synthetic")):
        res.setdefault(key, val)
    return res


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    import torch
    from quantized_kv_attention_gb300 import build as qbuild
    from quantized_kv_attention_gb300 import workloads as wl
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    rank, world = dist_init("nccl")
    if rank == 0:
        qbuild.build()
    barrier()
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    res = run_workload(args.workload, args, device, gpu_index, rank)
    if args.secondary and world == 1 and args.workload == "long_decode":
        res["secondary"] = secondary_lines(args, device, gpu_index, rank)
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(res), flush=True)
    import torch.distributed as dist
    if dist.is_initialized():
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
