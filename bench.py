"""Benchmark of global attention with decomposed relative-position bias.

One step = one pass of the whole path over one batch: the fused entry
(dera_relpos_fused: projection + biased online-softmax attention, one kernel
launch) on the DeepEncoder global-attention workload (B=1, 12 heads, 64x64
grid, N=4096, head_dim 64, bf16; inputs already in HBM).  The L2 cache is
flushed (256 MiB write) between timed steps, outside each step's events.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU float64
oracle instead (the reference arm of this method), on a bounded sample.
Under torchrun the global batch holds N times the workload's (batch, head)
problems and every rank computes its contiguous range of them (weak scaling;
the path has no exchange step); the slowest rank's time counts.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ms and TFLOP/s of 64×64-grid rel-pos global attention; % of GB300 BF16 peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}
L2_FLUSH_BYTES = 256 << 20


# --------------------------------------------------------------------------- helpers (no GPU needed)
def attention_flops(BH: int, N: int, d: int = 64) -> float:
    """Algorithmic FLOPs of the attention: QK^T and PV, 2*N*N*d each per (batch, head)."""
    return 4.0 * BH * N * N * d


def projection_flops(BH: int, N: int, H: int, W: int, d: int = 64) -> float:
    return 2.0 * BH * N * (H + W) * d


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# The sources each timed kernel is compiled from: stored counters stay valid while these are
# unchanged, whatever happens to the other kernels' files.
KERNEL_SOURCES = {
    "relpos_attn_kernel": ("attention.cuh", "attention_inst.cuh", "attention_w16.cu", "attention_w32.cu",
                           "attention_w40.cu", "attention_w64.cu", "common.cuh", "ptx.cuh", "launch.cuh"),
    "relpos_bwd": ("backward.cu", "backward.cuh", "common.cuh", "ptx.cuh", "launch.cuh"),
}


def source_hash(kernel: str = "relpos_attn_kernel") -> str:
    """Hash of the CUDA sources a kernel is built from, to tell whether stored ncu counters still
    describe it."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "relative_position_bias_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel.split("<")[0]]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None if absent or stale."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            entries = json.load(f)
    except (OSError, ValueError):
        return None
    e = entries.get(f"{kernel}/{workload}")
    if not e or e.get("source_hash") != source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


def aggregate_max(value: float, group=None) -> float:
    """Max over ranks of a per-rank float (the slowest rank sets the job time)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def job_value(flops_per_step: float, steps: int, world: int, slowest_s: float) -> float:
    """Whole-job TFLOP/s: every rank runs `steps` steps of its own replica; the slowest rank's time counts."""
    return flops_per_step * steps * world / slowest_s / 1e12


def percentile(xs: list[float], q: float) -> float:
    s = sorted(xs)
    k = (len(s) - 1) * q
    lo, hi = int(k), min(int(k) + 1, len(s) - 1)
    return s[lo] + (s[hi] - s[lo]) * (k - lo)


class ClockSampler:
    """Samples SM clock and throttle reasons with nvidia-smi while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self) -> dict | None:
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), power=float(parts[3]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], swp=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        smax = max(r["smax"] for r in rows)
        loaded = [r for r in rows if r["power"] > 0.35 * max(x["power"] for x in rows)] or rows
        reasons = set()
        for r in loaded:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(loaded)}


# --------------------------------------------------------------------------- reference arm (CPU oracle)
def oracle_rows_timing(x64: dict, w, rows, head: int) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.fused_rows(x64["q"], x64["k"], x64["v"], x64["rel_pos_h"], x64["rel_pos_w"], head, rows, w.H, w.W,
                      w.scale)
    return time.perf_counter() - t0


def cpu_oracle_throughput(w, budget_s: float, seed: int = 0) -> tuple[float, str, int]:
    """TFLOP/s of the float64 oracle on whole heads of the workload, for about `budget_s` seconds."""
    import numpy as np
    import oracle
    from relative_position_bias_gb300 import inputs as I
    x = I.make_inputs(w, seed=seed)
    q, k, v = (I.to_f64(x[n]) for n in ("q", "k", "v"))
    th, tw = I.to_f64(x["rel_pos_h"]), I.to_f64(x["rel_pos_w"])
    heads = 0
    t0 = time.perf_counter()
    while heads < w.BH and (time.perf_counter() - t0) < budget_s:
        oracle.fused(q[heads:heads + 1], k[heads:heads + 1], v[heads:heads + 1], th, tw, w.H, w.W, w.scale)
        heads += 1
    dt = time.perf_counter() - t0
    flops = attention_flops(heads, w.N)
    del np
    return flops / dt / 1e12, f"{heads} of {w.BH} heads of the workload through oracle.fused ({dt:.1f} s)", heads


def run_reference(args, w) -> dict:
    """The reference arm: the CPU oracle, each step a bounded sample of the workload's rows."""
    import numpy as np
    from relative_position_bias_gb300 import inputs as I
    cores = len(os.sched_getaffinity(0))
    x = I.make_inputs(w, seed=0)
    x64 = {n: I.to_f64(t) for n, t in x.items()}
    total_budget = float(os.environ.get("DERA_REF_BUDGET_S", "90"))
    per_step = total_budget / max(1, args.steps + args.warmup)
    # calibrate rows per step against the per-step budget
    rng = np.random.default_rng(0)
    rows = 64
    dt = oracle_rows_timing(x64, w, np.sort(rng.choice(w.N, rows, replace=False)), 0)
    rows = int(max(1, min(w.N, rows * per_step / max(dt, 1e-6))))
    times = []
    for s in range(args.warmup + args.steps):
        sel = np.sort(rng.choice(w.N, rows, replace=False))
        t = oracle_rows_timing(x64, w, sel, s % w.BH)
        if s >= args.warmup:
            times.append(t)
    flops_step = 4.0 * rows * w.N * w.d
    total = sum(times)
    value = flops_step * len(times) / total / 1e12
    sample = f"{rows} random query rows of one head per step (of {w.BH}x{w.N} rows), oracle.fused_rows in float64"
    return {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, "oracle"), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def workload_config(w, entry: str, world: int = 1) -> dict:
    kind = (f"DeepEncoder windowed attention, B={w.B} windows={w.windows} heads={w.heads} {w.H}x{w.W} window"
            if w.windows > 1 else f"DeepEncoder global attention, B={w.B} heads={w.heads} {w.H}x{w.W} grid")
    return {"workload": f"{w.name}: {kind} (N={w.N}), head_dim {w.d}, {w.dtype}, tables [{2 * w.H - 1},{w.d}] "
                        f"sigma {w.sigma_table}, scale {w.scale:g}",
            "B": w.B, "windows": w.windows, "heads": w.heads, "H": w.H, "W": w.W, "head_dim": w.d, "entry": entry,
            "l2": "flushed between timed steps (256 MiB write outside the step events)",
            "global_BH": world * w.BH,
            "parallelism": (f"dp{world}: contiguous (batch, head) ranges of the global batch, "
                            f"{w.BH} per GPU, no data-path collective") if world > 1 else "single GPU"}


# --------------------------------------------------------------------------- our arm
def run_ours(args, w, rank: int, world: int) -> dict | None:
    import torch
    import torch.distributed as dist
    import relative_position_bias_gb300 as rpb
    from relative_position_bias_gb300 import build as rbuild
    from relative_position_bias_gb300 import inputs as I
    from relative_position_bias_gb300.shard import bh_range

    rbuild.build()
    rpb.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    # weak scaling: the global batch holds world * BH (batch, head) problems and this rank
    # computes the contiguous range bh_range(world * BH, rank, world), drawn with its own seed
    lo, hi = bh_range(world * w.BH, rank, world)
    assert hi - lo == w.BH
    x = I.make_inputs(w, seed=rank)
    d = {k: t.to(dev) for k, t in x.items()}
    out = torch.empty(w.BH, w.N, w.d, dtype=w.torch_dtype, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    fargs = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)

    def step():
        if args.entry == "fused":
            rpb.fused(*fargs, out=out)
        else:
            rh, rw = rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, rel_h=rel_h, rel_w=rel_w)
            rpb.attention(d["q"], d["k"], d["v"], rh, rw, w.H, w.W, w.scale, out=out)

    rel_h = rel_w = None
    if args.entry != "fused":
        rel_h = torch.empty(w.BH, w.N, w.H, device=dev)
        rel_w = torch.empty(w.BH, w.N, w.W, device=dev)
    launches_per_step = 1 if args.entry == "fused" else 2

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clocks:
        t_wall = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_s = aggregate_max(sum(ms) / 1e3)
    flops = attention_flops(w.BH, w.N, w.d)
    # value, ms_per_step and roofline.achieved all use the mean over the timed steps (the summed
    # step time of the slowest rank over the step count); the median is reported beside them
    value = job_value(flops, args.steps, world, total_s)
    ms_mean = 1e3 * total_s / args.steps
    ms_med = statistics.median(ms)

    # end to end through the public API: every step copies its inputs from
    # pinned host memory and reads its result back to pinned host memory.
    # Steps alternate between two device buffer sets, with the input copies
    # and the read-backs on streams of their own, so one step's copies overlap
    # the neighbouring steps' kernels (the copies stay inside the timed region).
    host = {k: t.pin_memory() for k, t in x.items()}
    host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    dbuf = [d, {k: torch.empty_like(t) for k, t in d.items()}]
    obuf = [out, torch.empty_like(out)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    e2e_steps = max(3, min(args.steps, 50))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]

    def step_on(b):
        db = dbuf[b]
        if args.entry == "fused":
            rpb.fused(db["q"], db["k"], db["v"], db["rel_pos_h"], db["rel_pos_w"], w.H, w.W, w.scale, out=obuf[b])
        else:
            rh, rw = rpb.project(db["q"], db["rel_pos_h"], db["rel_pos_w"], w.H, w.W, rel_h=rel_h, rel_w=rel_w)
            rpb.attention(db["q"], db["k"], db["v"], rh, rw, w.H, w.W, w.scale, out=obuf[b])

    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    e0.record(s_in)
    for i in range(e2e_steps):
        b = i & 1
        if i >= 2:
            s_in.wait_event(ev_done[b])  # step i - 2 has finished reading buffer set b
        with torch.cuda.stream(s_in):
            for k in dbuf[b]:
                dbuf[b][k].copy_(host[k], non_blocking=True)
        ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_read[b])  # the result of step i - 2 has been read back
        with torch.cuda.stream(stream):
            step_on(b)
        ev_done[b].record(stream)
        s_out.wait_event(ev_done[b])
        with torch.cuda.stream(s_out):
            host_out[b].copy_(obuf[b], non_blocking=True)
        ev_read[b].record(s_out)
    s_out.wait_event(ev_done[(e2e_steps - 1) & 1])
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_s = aggregate_max(e0.elapsed_time(e1) / 1e3)
    e2e_value = job_value(flops, e2e_steps, world, e2e_s)

    # the other kernels of the path, on the same workload: projection alone
    # (HBM-bound) and the two-step path (projection + compact-bias attention)
    rh = torch.empty(w.BH, w.N, w.H, device=dev)
    rw = torch.empty(w.BH, w.N, w.W, device=dev)
    extra_steps = max(3, min(args.steps, 100))

    def timed(fn):
        evs = []
        for _ in range(3):
            flush.fill_(3)
            fn()
        for _ in range(extra_steps):
            flush.fill_(7)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    proj_ms = timed(lambda: rpb.project(d["q"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, rel_h=rh, rel_w=rw))
    attn_ms = timed(lambda: rpb.attention(d["q"], d["k"], d["v"], rh, rw, w.H, w.W, w.scale, out=out))
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    proj_bytes = (w.BH * w.N * w.d * 2 + w.BH * w.N * (w.H + w.W) * 4 + (2 * w.H - 1 + 2 * w.W - 1) * w.d * 2)
    extra = {
        "projection": {"kernel": "relpos_project_kernel", "ms": proj_ms, "bytes_per_launch": proj_bytes,
                       "gbs": proj_bytes / (proj_ms * 1e-3) / 1e9, "hbm_peak_gbs": hbm,
                       "frac_hbm": proj_bytes / (proj_ms * 1e-3) / 1e9 / hbm},
        "two_step": {"ms": proj_ms + attn_ms, "attention_ms": attn_ms,
                     "attention_tflops": attention_flops(w.BH, w.N, w.d) / (attn_ms * 1e-3) / 1e12},
    }
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms_mean / 1e3) / 1e12
    kernel = "relpos_attn_kernel<64,fused>" if args.entry == "fused" else "relpos_attn_kernel<64,compact>"
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_mean, "statistic": "mean over the timed steps",
        "ms_median": ms_med, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, args.entry, world),
        "ms_p10": percentile(ms, 0.1), "ms_p90": percentile(ms, 0.9),
        "pct_of_bf16_peak": 100.0 * achieved / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": stored_traffic(kernel, w.name),
                     "kernel": kernel, "peak_source": f"bf16_tflops (burst) of {peak_src}",
                     "flops_per_launch": flops},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "overlap": "two device buffer sets; input copies and read-backs on their own streams"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
        "other_kernels": extra,
    }
    if not args.no_cpu_baseline:
        v, sample, _ = cpu_oracle_throughput(w, budget_s=args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
                                "kind": "oracle", "sample": sample}
    return line


def backward_flops(BH: int, N: int, d: int = 64) -> float:
    """Algorithmic FLOPs of the attention backward: dv = P^T dO, dP = dO v^T, dq = dZ k, dk = dZ^T q and
    the recomputation of S = q k^T, 2*N*N*d each per (batch, head) (2.5 times the forward's)."""
    return 10.0 * BH * N * N * d


def run_backward(args, w, rank: int, world: int) -> dict | None:
    """`--entry backward`: one step = dera_relpos_fused_backward (projection, rows, cols and table
    kernels) on the workload, with the training forward's out and lse and a random dout
    already in HBM; gradients in the input dtype."""
    import torch
    import relative_position_bias_gb300 as rpb
    from relative_position_bias_gb300 import build as rbuild
    from relative_position_bias_gb300 import inputs as I

    if w.d != 64:
        raise SystemExit("the backward supports head_dim 64")
    rbuild.build()
    rpb.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    x = I.make_inputs(w, seed=rank)
    d = {k: t.to(dev) for k, t in x.items()}
    g = torch.Generator().manual_seed(1000 + rank)
    dout = torch.randn(w.BH, w.N, w.d, generator=g).to(w.torch_dtype).to(dev)
    fargs = (d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], w.H, w.W, w.scale)
    out, lse = rpb.fused_lse(*fargs)
    ws = torch.empty(rpb.backward_workspace_size(w.BH, w.H, w.W, w.d), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        return rpb.fused_backward(d["q"], d["k"], d["v"], d["rel_pos_h"], d["rel_pos_w"], out, lse, dout, w.H, w.W,
                                  w.scale, grad_dtype=w.torch_dtype, workspace=ws)

    def timed(fn, n):
        for _ in range(args.warmup):
            flush.fill_(1)
            fn()
        torch.cuda.synchronize()
        evs = []
        for i in range(n):
            flush.fill_(i & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    with ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else 0) as clocks:
        ms = timed(step, args.steps)
    fwd_ms = timed(lambda: rpb.fused_lse(*fargs), max(3, min(args.steps, 100)))
    total_s = aggregate_max(sum(ms) / 1e3)
    flops = backward_flops(w.BH, w.N, w.d)
    value = job_value(flops, args.steps, world, total_s)
    if rank != 0:
        return None
    ms_mean = 1e3 * total_s / args.steps
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    achieved = flops / (ms_mean / 1e3) / 1e12
    cfg = workload_config(w, "backward", world)
    return {
        "metric": "TFLOP/s of the attention backward (dq, dk, dv and the table gradients) on the workload",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_mean, "statistic": "mean over the timed steps", "ms_median": statistics.median(ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "the whole backward call (4 kernels)",
                     "peak_source": f"bf16_tflops (burst) of {peak_src}", "flops_per_launch": flops,
                     "flops_executed": 14.0 * w.BH * w.N * w.N * w.d},
        "training_forward": {"ms": statistics.median(fwd_ms),
                             "tflops": attention_flops(w.BH, w.N, w.d) / (statistics.median(fwd_ms) * 1e-3) / 1e12},
        "gpu_launches": 4 * args.steps,
        "clocks": clocks.summary(),
    }


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="global64")
    ap.add_argument("--entry", choices=["fused", "two_step", "backward"], default="fused")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps < 1:
        ap.error("--steps must be >= 1")

    from relative_position_bias_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    line = run_backward(args, w, rank, world) if args.entry == "backward" else run_ours(args, w, rank, world)
    if line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
