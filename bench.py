#!/usr/bin/env python
"""Benchmark: bf16 causal attention fwd+bwd at B4 H8 T8192 d128 on GB300.

One step = one pass of the hot path over one batch of seeded synthetic input:
attn_fwd (O, LSE) then attn_bwd (delta preprocess, dK/dV kernel, dQ kernel;
the deterministic two-pass backward).  FLOPs follow the pages' convention:
fwd = 4 * B * H * Lq * Lkv * d, exactly halved for causal, fwd+bwd = 3.5x.

Prints ONE JSON line (rank 0).  Under torchrun (N > 1) every rank runs its own
independent replica of the step on its own GPU (the units are independent; no
collective on the data path) and the value is the total work of all ranks
divided by the slowest rank's time ("weak" scaling).

``--impl reference`` times the fp64 CPU oracle (the only reference this
project has) on the host cores, one bounded sample of the same workload per
step; under torchrun only rank 0 runs it.

Inputs (256 MiB of q/k/v/dO plus outputs) are larger than the 129 MB L2, so no
L2 flush is done between steps.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time


def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


# The oracle's BLAS runs on every core this process may use: the thread counts
# are read when numpy loads its BLAS, so they are set before anything imports it
# (a value the caller exported is kept and reported).
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_var, str(host_cores()))

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "fwd+bwd TFLOP/s (bf16, B4 H8 T8192 d128 causal) and % of GB300 tensor peak"
UNIT = "TFLOP/s"


# ----------------------------------------------------------------------------
# rank handling (host logic; tested with gloo on CPU)
# ----------------------------------------------------------------------------

def dist_env():
    """(rank, local_rank, world_size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def dist_init(world: int, backend: str):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (x itself when world == 1)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(flops_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """TFLOP/s of all ranks together: every rank does flops_per_step per step."""
    return world * flops_per_step * steps / (max_ms * 1e-3) / 1e12


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

CLOCK_FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
                "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
                "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    """Samples nvidia-smi every 200 ms in the background; keeps the samples
    taken between mark_start() and mark_stop()."""

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.t0 = self.t1 = None
        self.proc = None
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        time.sleep(0.3)
        return self

    def _reader(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.strip().split(",")]
            if len(parts) == len(CLOCK_FIELDS):
                self.samples.append((time.time(), parts))

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()
        time.sleep(0.25)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.samples or self.t0 is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"], "samples": 0}
        t1 = self.t1 if self.t1 is not None else time.time()
        win = [p for (t, p) in self.samples if self.t0 - 0.2 <= t <= t1 + 0.2] or [p for (_, p) in self.samples]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = sorted(v for v in (num(p[1]) for p in win) if v is not None)
        mx = [v for v in (num(p[2]) for p in win) if v is not None]
        names = {5: "hw_slowdown", 6: "hw_thermal_slowdown", 7: "sw_thermal_slowdown", 8: "sw_power_cap"}
        reasons = sorted({names[i] for p in win for i in names if p[i].lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win),
                "power_w_max": max((v for v in (num(p[3]) for p in win) if v is not None), default=None)}


# ----------------------------------------------------------------------------
# measured peaks and the committed ncu traffic summary
# ----------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def source_digest(kernel_file: str) -> str:
    with open(os.path.join(ROOT, "exact_attention_34_gb300", "csrc", kernel_file), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from profiles/ncu_traffic.json, or None
    when absent or when the kernel source changed since the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)[kernel]
        if d["source_sha1"] != source_digest(d["source_file"]):
            return None
        return float(d["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


# ----------------------------------------------------------------------------
# the GPU arm
# ----------------------------------------------------------------------------

KERNEL_FILES = {"fwd": "fwd_sm103.cu", "bwd_dkdv": "bwd_sm103.cu", "bwd_dq": "bwd_sm103.cu",
                "bwd_preprocess": "small_kernels.cu", "decode": "decode_sm103.cu", "combine": "small_kernels.cu"}


def run_gpu(args):
    import torch

    import exact_attention_34_gb300 as ea
    from exact_attention_34_gb300 import build as eb

    rank, local_rank, world = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local_rank)
    dist_init(world, "nccl")
    eb.build()
    dev = torch.device("cuda", local_rank)

    p = W.headline()
    F_fwd = W.fwd_flops(p)
    F_step = 3.5 * F_fwd
    q_h, k_h, v_h, do_h = (t.pin_memory() for t in W.make_inputs(p, seed=0))
    q, k, v, do = (t.to(dev) for t in (q_h, k_h, v_h, do_h))
    o = torch.empty_like(q)
    lse = torch.empty(p.B, p.Hq, p.Lq, device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(ea.attn_bwd_workspace_size(p.B, p.Lq, p.Hq, p.d, True, q.dtype), device=dev,
                     dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def step():
        ea.attn_fwd(q, k, v, o, lse, causal=True, stream=stream)
        ea.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, causal=True, deterministic=True, stream=stream)

    # ---- device-resident timing: EXACTLY `steps` steps between events
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # one event per step boundary: the first-to-last span is the timed region,
    # consecutive pairs give the per-step spread
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    with ClockSampler(local_rank) as clk:
        barrier(world)
        torch.cuda.synchronize()
        clk.mark_start()
        evs[0].record(stream)
        for i in range(args.steps):
            step()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        clk.mark_stop()
        barrier(world)
    local_ms = evs[0].elapsed_time(evs[-1])
    max_ms = max_over_ranks(local_ms, world, dev)
    value = whole_job_value(F_step, args.steps, world, max_ms)
    ms_per_step = max_ms / args.steps
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    quart = [round(per_step[min(len(per_step) - 1, int(f * len(per_step)))], 4) for f in (0.25, 0.5, 0.75)]

    # ---- per-kernel durations (a separate pass with launch events enabled)
    ea.attn_timing_enable(True)
    for _ in range(args.kernel_steps):
        step()
    torch.cuda.synchronize()
    ktimes = {}
    for name in ("fwd", "bwd_preprocess", "bwd_dkdv", "bwd_dq"):
        ms, n = ea.attn_timing_query(name)
        ktimes[name] = {"avg_ms": ms / max(n, 1), "launches": n}
    ea.attn_timing_enable(False)
    # algorithmic work per launch: dK/dV carries 4 of the 5 backward GEMMs
    # (S, dP, dV, dK), dQ carries dS K (its S and dP are recomputation)
    peaks = measured_peaks()
    algo = {"fwd": F_fwd, "bwd_dkdv": 2.0 * F_fwd, "bwd_dq": 0.5 * F_fwd}
    dom = max(("fwd", "bwd_dkdv", "bwd_dq"), key=lambda n: ktimes[n]["avg_ms"])
    achieved = algo[dom] / (ktimes[dom]["avg_ms"] * 1e-3) / 1e12
    # the kernels run inside a timed region of tens to hundreds of ms at the
    # full SM clock (sampled below), so the burst peak is the one that applies;
    # the fraction of the sustained (power-capped, lower-clock) figure is context
    peak = peaks["bf16_tflops"]
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(dom),
                "peak_kind": f"bf16 dense, burst, {peaks['source']}",
                "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                "per_kernel": {n: {"avg_ms": round(ktimes[n]["avg_ms"], 4), "launches": ktimes[n]["launches"],
                                   **({"tflops": round(algo[n] / (ktimes[n]["avg_ms"] * 1e-3) / 1e12, 1)}
                                      if n in algo and ktimes[n]["avg_ms"] > 0 else {})}
                               for n in ktimes}}

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs host -> device and its gradients device -> host; the
    # uploads of step t+1 and the downloads of step t-1 run on two copy streams
    # (one per direction) while step t computes, with two sets of device buffers.
    dq_h, dk_h, dv_h = (torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv))
    host_in, host_out = (q_h, k_h, v_h, do_h), (dq_h, dk_h, dv_h)
    dev_in = [[torch.empty_like(t) for t in (q, k, v, do)] for _ in range(2)]
    dev_out = [[torch.empty_like(t) for t in (dq, dk, dv)] for _ in range(2)]
    dev_ol = [(torch.empty_like(o), torch.empty_like(lse)) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d_done, comp_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def h2d(t):
        bi = t % 2
        with torch.cuda.stream(up):
            if t >= 2:
                up.wait_event(comp_done[bi])  # step t-2 has finished reading these inputs
            for dst, src in zip(dev_in[bi], host_in):
                dst.copy_(src, non_blocking=True)
            h2d_done[bi].record(up)

    def compute(t):
        bi = t % 2
        stream.wait_event(h2d_done[bi])
        if t >= 2:
            stream.wait_event(d2h_done[bi])  # step t-2's gradients have left these buffers
        q2, k2, v2, do2 = dev_in[bi]
        o2, lse2 = dev_ol[bi]
        g = dev_out[bi]
        ea.attn_fwd(q2, k2, v2, o2, lse2, causal=True, stream=stream)
        ea.attn_bwd(q2, k2, v2, o2, lse2, do2, g[0], g[1], g[2], ws, causal=True, deterministic=True, stream=stream)
        comp_done[bi].record(stream)

    def d2h(t):
        bi = t % 2
        with torch.cuda.stream(down):
            down.wait_event(comp_done[bi])
            for dst, src in zip(host_out, dev_out[bi]):
                dst.copy_(src, non_blocking=True)
            d2h_done[bi].record(down)

    def run_pipelined(n):
        h2d(0)
        for t in range(n):
            if t + 1 < n:
                h2d(t + 1)
            compute(t)
            d2h(t)

    e2e_steps = args.steps
    run_pipelined(2)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    run_pipelined(e2e_steps)
    e1.record(down)  # after the last gradients reached the host
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)

    # the same steps with every copy serialised on the compute stream (context)
    def serial_step():
        q2, k2, v2, do2 = dev_in[0]
        for dst, src in zip(dev_in[0], host_in):
            dst.copy_(src, non_blocking=True)
        ea.attn_fwd(q2, k2, v2, o, lse, causal=True, stream=stream)
        ea.attn_bwd(q2, k2, v2, o, lse, do2, dq, dk, dv, ws, causal=True, deterministic=True, stream=stream)
        for dst, src in zip(host_out, (dq, dk, dv)):
            dst.copy_(src, non_blocking=True)

    serial_step()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(e2e_steps):
        serial_step()
    s1.record(stream)
    torch.cuda.synchronize()
    serial_ms = max_over_ranks(s0.elapsed_time(s1), world, dev)
    h2d_b = sum(t.numel() * t.element_size() for t in host_in)
    d2h_b = sum(t.numel() * t.element_size() for t in host_out)
    e2e = {"value": round(whole_job_value(F_step, e2e_steps, world, e2e_ms), 2), "unit": UNIT,
           "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b, "steps": e2e_steps,
           "overlap": "H2D of step t+1 and D2H of step t-1 on two copy streams during step t",
           "serial_value": round(whole_job_value(F_step, e2e_steps, world, serial_ms), 2)}

    st, code, site = ea.attn_device_status()
    if code != 0:
        raise SystemExit(f"device status {code} at site {site}")

    extra = {}
    if rank == 0 and not args.no_extra:
        extra = other_rows(args, dev, peaks)

    result = None
    if rank == 0:
        clocks = clk.summary()
        cpu = None if args.no_cpu_baseline else cpu_baseline_sample(args.cpu_budget_s)
        result = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "ms_per_step_q1_median_q3": quart, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "bf16 causal attention fwd+bwd, B4 H8 T8192 d128 (deterministic two-pass bwd)",
                       "global_batch": p.B * world, "seq_len": p.Lq, "heads": p.Hq, "head_dim": p.d,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (256 MiB q/k/v/dO), no flush",
                       "flops_per_step": F_step},
            "pct_of_peak": {"burst": round(value / world / peaks["bf16_tflops"], 4),
                            "sustained": round(value / world / peaks["bf16_tflops_sustained"], 4),
                            "source": peaks["source"]},
            "roofline": roofline, "e2e": e2e, "gpu_launches": 4 * args.steps, "clocks": clocks,
            "cpu_baseline": cpu, "rows": extra,
        }
    return result


def other_rows(args, dev, peaks):
    """Quick one-shot numbers for the other rows of the path (context, not the headline)."""
    import numpy as np
    import torch

    import exact_attention_34_gb300 as ea

    out = {}

    def timed(fn, n=10):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    g = torch.Generator(device=dev).manual_seed(0)
    # the headline workload with the single-pass backward (atomic dQ)
    p = W.headline()
    q = torch.randn(p.B, p.Lq, p.Hq, p.d, device=dev, generator=g).to(torch.bfloat16)
    k, v, do = torch.randn_like(q), torch.randn_like(q), torch.randn_like(q)

    def sp_step():
        o, lse = ea.forward(q, k, v, causal=True)
        ea.backward(q, k, v, o, lse, do, causal=True, deterministic=False)

    ms = timed(sp_step)
    ea.attn_timing_enable(True)
    for _ in range(5):
        sp_step()
    torch.cuda.synchronize()
    kt = {n: round(ea.attn_timing_query(n)[0] / 5, 4)
          for n in ("fwd", "bwd_preprocess", "bwd_dkdv_atomic", "dq_convert")}
    ea.attn_timing_enable(False)
    out["single_pass_fwd_bwd"] = {"ms": round(ms, 4), "tflops": round(3.5 * W.fwd_flops(p) / ms / 1e9, 1),
                                  "kernel_ms": kt, "note": "same workload, atomic-dQ backward (not bitwise reproducible)"}

    # the single pass with dQ added in key-tile order (bitwise reproducible)
    def ordered_step():
        o, lse = ea.forward(q, k, v, causal=True)
        ea.backward(q, k, v, o, lse, do, causal=True, deterministic=2)

    ms = timed(ordered_step)
    ea.attn_timing_enable(True)
    for _ in range(5):
        ordered_step()
    torch.cuda.synchronize()
    kt = {n: round(ea.attn_timing_query(n)[0] / 5, 4)
          for n in ("fwd", "bwd_preprocess", "bwd_dkdv_ordered", "dq_convert")}
    ea.attn_timing_enable(False)
    out["single_pass_deterministic"] = {
        "ms": round(ms, 4), "tflops": round(3.5 * W.fwd_flops(p) / ms / 1e9, 1), "kernel_ms": kt,
        "note": "same workload, single-pass backward with each query tile's dQ added in key-tile order "
                "(bitwise reproducible; deterministic=2)"}
    del q, k, v, do
    # local-window mask on the headline shapes: a 1024-key causal sliding
    # window (flops over the valid (row, key) pairs)
    p = W.headline()
    win = (1024, 0)
    q = torch.randn(p.B, p.Lq, p.Hq, p.d, device=dev, generator=g).to(torch.bfloat16)
    k, v, do = torch.randn_like(q), torch.randn_like(q), torch.randn_like(q)

    def win_step():
        o, lse = ea.forward(q, k, v, window=win)
        ea.backward(q, k, v, o, lse, do, window=win)

    ms = timed(win_step)
    pairs = sum(min(i + 1, win[0] + 1) for i in range(p.Lq))
    f_win = 4.0 * p.B * p.Hq * p.d * pairs
    out["window_fwd_bwd"] = {"ms": round(ms, 4), "tflops": round(3.5 * f_win / ms / 1e9, 1),
                             "window": list(win), "note": "B4 H8 T8192 d128 bf16, keys within 1024 before the row"}
    del q, k, v, do
    # segment (document) masks on the headline shapes, causal within each
    # document (flops over the valid pairs): packed documents of 1024 tokens,
    # and documents of seeded random lengths 1..2047 (boundaries off the tile
    # grid).  A step computes the ids' block summary once, then fwd + bwd.
    p = W.headline()
    q = torch.randn(p.B, p.Lq, p.Hq, p.d, device=dev, generator=g).to(torch.bfloat16)
    k, v, do = torch.randn_like(q), torch.randn_like(q), torch.randn_like(q)
    rng = np.random.default_rng(11)
    ragged = []
    for _ in range(p.B):
        lens, tot = [], 0
        while tot < p.Lq:
            n = min(int(rng.integers(1, 2048)), p.Lq - tot)
            lens.append(n)
            tot += n
        ragged.append(lens)
    layouts = {
        "segments_fwd_bwd": [[1024] * (p.Lq // 1024)] * p.B,
        "segments_ragged_fwd_bwd": ragged,
    }
    for name, lens in layouts.items():
        seg = torch.tensor(np.stack([np.repeat(np.arange(len(ls), dtype=np.int32), ls) for ls in lens]),
                           device=dev)

        def seg_step():
            segs = (seg, seg, ea.segment_info(seg, seg))
            o, lse = ea.forward(q, k, v, causal=True, segments=segs)
            ea.backward(q, k, v, o, lse, do, causal=True, segments=segs)

        ms = timed(seg_step)
        pairs = sum(n * (n + 1) // 2 for ls in lens for n in ls)  # over all batch elements
        f_seg = 4.0 * p.Hq * p.d * pairs
        kind = "packed 1024-token documents" if name == "segments_fwd_bwd" else \
            f"{sum(len(ls) for ls in lens)} documents of seeded random lengths 1..2047"
        out[name] = {"ms": round(ms, 4), "tflops": round(3.5 * f_seg / ms / 1e9, 1),
                     "note": f"B4 H8 T8192 d128 bf16, causal within {kind}; the block summary drops tiles "
                             "across documents and runs single-document tiles unmasked"}
    del q, k, v, do
    # head_dim 256 (its own kernels): the headline shapes at d = 256
    q = torch.randn(p.B, p.Lq, p.Hq, 256, device=dev, generator=g).to(torch.bfloat16)
    k, v, do = torch.randn_like(q), torch.randn_like(q), torch.randn_like(q)

    def d256_step():
        o, lse = ea.forward(q, k, v, causal=True)
        ea.backward(q, k, v, o, lse, do, causal=True)

    ms = timed(d256_step)
    f256 = 4.0 * p.B * p.Hq * p.Lq * p.Lq * 256 / 2
    out["d256_fwd_bwd"] = {"ms": round(ms, 4), "tflops": round(3.5 * f256 / ms / 1e9, 1),
                           "note": "B4 H8 T8192 d256 bf16 causal, deterministic backward (dV, dK, dQ kernels)"}
    del q, k, v, do
    # KVLenMask + GQA + Lq != Lkv fwd+bwd (flops over valid keys)
    p = W.kvlen_gqa()
    q = torch.randn(p.B, p.Lq, p.Hq, p.d, device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn(p.B, p.Lkv, p.Hkv, p.d, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn_like(k)
    do = torch.randn_like(q)
    kl = torch.tensor(p.kv_lens, dtype=torch.int32, device=dev)

    def kv_step(splits):
        o, lse = ea.forward(q, k, v, kv_lens=kl, num_splits=splits)
        ea.backward(q, k, v, o, lse, do, kv_lens=kl)

    ms = timed(lambda: kv_step(0))
    ms1 = timed(lambda: kv_step(1))
    n_split = ea.attn_fwd_num_splits(p.B, p.Lq, p.Lkv, p.Hq, p.d, True, q.dtype)
    out["kvlen_gqa_fwd_bwd"] = {
        "ms": round(ms, 4), "tflops": round(3.5 * W.fwd_flops(p) / ms / 1e9, 1),
        "forward_pieces": n_split, "unsplit_ms": round(ms1, 4),
        "unsplit_tflops": round(3.5 * W.fwd_flops(p) / ms1 / 1e9, 1),
        "note": "B4 Hq8 Hkv2 Lq2048 Lkv16384 d128 bf16, KV lengths (13350, 236, 1, 0); the forward cuts each "
                "query-tile pair's key range into the library's number of pieces (num_splits=0)"}
    del q, k, v, do
    # split-KV decode (HBM-bound): bytes of valid K/V + q + partials + o
    for Lq, causal in ((1, False), (16, True)):
        out[f"decode_Lq{Lq}"] = decode_row(dev, g, peaks, timed, Lq, causal)
    torch.cuda.empty_cache()
    out["grid"] = grid_rows(dev, peaks)
    return out


# Cells of the attention grid timed by the default run: the longest sequences
# at both head sizes, a ragged length, and float32 (the rest: --sweep).
GRID_ROWS = [(8192, 64, False, "bf16"), (8192, 64, True, "bf16"), (8192, 128, False, "bf16"),
             (8192, 128, True, "bf16"), (3000, 128, True, "bf16"), (3000, 64, True, "bf16"),
             (2048, 128, False, "fp32"), (2048, 128, True, "fp32")]


def grid_rows(dev, peaks):
    """fwd+bwd of each GRID_ROWS cell (B4 H8, deterministic backward, eager
    calls): median and quartiles of five repeats, each repeat enough
    back-to-back steps for ~25 ms, and the fraction of the burst bf16 peak
    (float32 runs on the CUDA cores; its fraction is of that same peak)."""
    import torch

    import exact_attention_34_gb300 as ea

    rows = {}
    for T, d, causal, dt in GRID_ROWS:
        p = W.grid(T, d, causal, dt)
        g = torch.Generator(device=dev).manual_seed(0)
        q, k, v, do = (torch.randn(p.B, T, p.Hq, d, device=dev, generator=g).to(W.DTYPES[dt]) for _ in range(4))
        F = 3.5 * W.fwd_flops(p)

        def call():
            o2, lse2 = ea.forward(q, k, v, causal=causal)
            ea.backward(q, k, v, o2, lse2, do, causal=causal)

        one = _timed_q(call, 1, repeats=1)[1]
        n = max(1, min(100, int(25.0 / max(one, 1e-3))))
        q1, med, q3 = _timed_q(call, n)
        tf = F / med / 1e9
        rows[f"T{T}_d{d}_{'causal' if causal else 'full'}_{dt}"] = {
            "fwd_bwd_ms": round(med, 4), "q1_q3_ms": [round(q1, 4), round(q3, 4)], "tflops": round(tf, 1),
            "frac_bf16_burst": round(tf / peaks["bf16_tflops"], 4), "steps_per_repeat": n}
        del q, k, v, do
        torch.cuda.empty_cache()
    return rows


def decode_row(dev, g, peaks, timed, Lq, causal, Lkv=131072):
    """One split-KV decode row (B8 Hq32 Hkv8 d128 bf16, KV lengths uniform in
    [4096, Lkv]): decode + combine time, and GB/s over the algorithmic bytes
    (K and V of the valid keys, q, o, lse and the fp32 partials written and
    read once)."""
    import torch

    import exact_attention_34_gb300 as ea

    p = W.decode(Lq, causal, Lkv=Lkv)
    q = torch.randn(p.B, p.Lq, p.Hq, p.d, device=dev, generator=g).to(torch.bfloat16)
    k = torch.randn(p.B, p.Lkv, p.Hkv, p.d, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn_like(k)
    kl = torch.tensor(p.kv_lens, dtype=torch.int32, device=dev)
    S = ea.attn_decode_num_splits(p.B, p.Lq, p.Lkv, p.Hq, p.Hkv, p.d)
    ms = timed(lambda: ea.decode(q, k, v, causal=causal, kv_lens=kl, num_splits=S))
    kv_bytes = sum(p.kv_lens) * p.Hkv * p.d * 2 * 2
    part_bytes = 2 * p.B * p.Hq * S * p.Lq * (p.d + 1) * 4
    io_bytes = 2 * p.B * p.Lq * p.Hq * p.d * 2 + p.B * p.Hq * p.Lq * 4
    gbs = (kv_bytes + part_bytes + io_bytes) / (ms * 1e-3) / 1e9
    del q, k, v
    return {"ms": round(ms, 4), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
            "num_splits": S, "bytes": kv_bytes + part_bytes + io_bytes}


def run_decode_suite(args):
    """The split-KV decode rows alone ("Attention performance", section
    "Grouped-query attention and decoding"): Lq = 1 and Lq = 16 with the causal
    offset, B8 Hq32 Hkv8 d128 bf16, cache length --decode-lkv (lengths uniform
    in [4096, that]).  One JSON line per row; a short cache keeps an ncu
    capture to about a GB of device memory."""
    import torch

    from exact_attention_34_gb300 import build as eb

    eb.build()
    dev = torch.device("cuda", 0)
    peaks = measured_peaks()

    def timed(fn, n=max(3, args.steps)):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    for Lq, causal in ((1, False), (16, True)):
        g = torch.Generator(device=dev).manual_seed(0)
        row = decode_row(dev, g, peaks, timed, Lq, causal, Lkv=args.decode_lkv)
        print(json.dumps({"suite": "decode", "Lq": Lq, "causal": causal, "Lkv": args.decode_lkv, **row}), flush=True)


# ----------------------------------------------------------------------------
# the fp64 CPU oracle, timed on a bounded sample
# ----------------------------------------------------------------------------

class OracleSampler:
    """The fp64 oracle's fwd+bwd on a bounded sample of the headline workload:
    query rows (spread evenly over the sequence) of one or more (batch, head)
    slices, FLOPs counted by the pages' rule over the sampled rows' valid keys."""

    def __init__(self):
        import numpy as np

        self.np = np
        p = W.headline()
        self.p = p
        self.q, self.k, self.v, self.do = W.make_inputs(p, seed=0)

    def rows(self, n):
        n = max(1, min(int(n), self.p.Lq))
        return self.np.unique(self.np.linspace(0, self.p.Lq - 1, n).astype(self.np.int64))

    def flops(self, rows):
        # causal: row i sees i + 1 keys; fwd = 4 d per (row, key) pair, fwd+bwd = 3.5x
        return 3.5 * 4.0 * self.p.d * float(self.np.sum(rows + 1))

    def run(self, sample):
        """sample = (n_heads, rows): the same rows of the first n_heads (batch, head) slices."""
        import oracle

        n_heads, rows = sample
        fl = 0.0
        for i in range(n_heads):
            b, h = i % self.p.B, (i // self.p.B) % self.p.Hq
            sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
            oracle.forward(self.q[sl], self.k[sl], self.v[sl], causal=True, rows=rows)
            oracle.backward(self.q[sl], self.k[sl], self.v[sl], self.do[sl], causal=True, rows=rows)
            fl += self.flops(rows)
        return fl

    def calibrate(self, budget_s):
        """A sample taking about budget_s seconds: as many rows of one slice as fit, then whole slices."""
        probe = (1, self.rows(512))
        t0 = time.perf_counter()
        self.run(probe)
        per_row = (time.perf_counter() - t0) / len(probe[1])
        n_rows = budget_s / max(per_row, 1e-9)
        if n_rows <= self.p.Lq:
            return (1, self.rows(n_rows))
        return (int(min(self.p.B * self.p.Hq, max(1, round(n_rows / self.p.Lq)))), self.rows(self.p.Lq))

    @staticmethod
    def describe(sample):
        n_heads, rows = sample
        return f"{len(rows)} of 8192 query rows (evenly spaced) of {n_heads} of 32 (batch, head) slices"


def blas_threads():
    """Threads the oracle's BLAS uses: threadpoolctl's answer where it is
    installed, else the thread count set for it before numpy was loaded."""
    try:
        from threadpoolctl import threadpool_info

        n = [int(i["num_threads"]) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:  # noqa: BLE001 - optional module; fall back to the environment
        pass
    return int(os.environ.get("OPENBLAS_NUM_THREADS", host_cores()))


def cpu_baseline_sample(budget_s: float = 15.0):
    """Oracle timed on the host cores on a ~budget_s sample (GPU arm, rank 0)."""
    smp = OracleSampler()
    sample = smp.calibrate(budget_s)
    t0 = time.perf_counter()
    fl = smp.run(sample)
    dt = time.perf_counter() - t0
    return {"value": round(fl / dt / 1e12, 6), "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "host_cores": host_cores(),
            "sample": f"{smp.describe(sample)}, B4 H8 T8192 d128 causal, fwd+bwd in fp64 numpy "
                      f"({blas_threads()} BLAS threads) in {dt:.1f} s"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return None
    smp = OracleSampler()
    budget = max(0.05, args.reference_budget_s / (args.steps + args.warmup))
    smp_rows = smp.calibrate(budget)
    for _ in range(args.warmup):
        smp.run(smp_rows)
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += smp.run(smp_rows)
    dt = time.perf_counter() - t0
    value = fl / dt / 1e12
    sample = f"{smp.describe(smp_rows)} per step, fwd+bwd in fp64 numpy ({blas_threads()} BLAS threads)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "bf16 causal attention fwd+bwd, B4 H8 T8192 d128 (inputs bf16, oracle in fp64)",
                   "global_batch": 4, "seq_len": 8192, "sample_per_step": sample},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                         "host_cores": host_cores(), "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def sweep_key(T, d, causal, dtype):
    """Identity of one case of the attention grid."""
    return (int(T), int(d), bool(causal), str(dtype))


def sweep_done_keys(path):
    """Keys of the cases already recorded in an --append file: one JSON object
    per line; a line cut short by a killed run (not valid JSON) is ignored, so
    that case runs again."""
    done = set()
    if not path or not os.path.exists(path):
        return done
    with open(path) as f:
        for line in f:
            try:
                r = json.loads(line)
                done.add(sweep_key(r["T"], r["d"], r["causal"], r["dtype"]))
            except (ValueError, KeyError, TypeError):
                continue
    return done


def sweep_end_partial_line(path):
    """Terminate a last line cut short by a killed run, so the next appended
    line starts on a line of its own."""
    if not path or not os.path.exists(path) or os.path.getsize(path) == 0:
        return
    with open(path, "rb") as f:
        f.seek(-1, os.SEEK_END)
        last = f.read(1)
    if last != b"\n":
        with open(path, "a") as f:
            f.write("\n")


def run_sweep(args):
    """The pages' attention grid ("Attention performance", section "Time"): B4 H8,
    d in {64, 128}, T in {128 ... 8192} plus the ragged 600 / 1500 / 3000, causal
    and not, bf16; fwd and fwd+bwd TFLOP/s (deterministic backward).  One JSON
    line per case, median of 5 repeats with the quartiles.  Also head_dim 32
    (bf16) and fp32 at d=128 for T <= 2048.  Each case is timed twice: as eager
    calls (host work of every call included: the Python binding, tensor
    allocation, tensor-map encoding and launches), fwd+bwd also as eager calls
    of the C-name entry points into buffers allocated once
    (`prealloc_fwd_bwd_ms`), and as replays of a CUDA graph that captured the
    same calls (device time; what a compiled training step sees).  With
    --append FILE each finished case is also appended to FILE, and cases
    already there are skipped, so a killed sweep resumes where it stopped."""
    import torch

    import exact_attention_34_gb300 as ea
    from exact_attention_34_gb300 import build as eb

    eb.build()
    dev = torch.device("cuda", 0)

    def timed(fn, n, repeats=5):
        """(q1, median, q3) in ms of `repeats` runs of n back-to-back calls each."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        runs = []
        for _ in range(repeats):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(n):
                fn()
            b.record()
            torch.cuda.synchronize()
            runs.append(a.elapsed_time(b) / n)
        runs.sort()
        return runs[len(runs) // 4], runs[len(runs) // 2], runs[(3 * len(runs)) // 4]

    def graph_timed(fn, n):
        """timed() of replays of a CUDA graph holding one fn() call."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        return timed(graph.replay, n)

    cases = [(T, d, c, "bf16") for d in (64, 128) for T in W.GRID_T + W.RAGGED_T for c in (False, True)]
    cases += [(T, 32, c, "bf16") for T in W.GRID_T for c in (False, True)]  # head_dim 32 (runs as 64)
    cases += [(T, 128, c, "fp32") for T in (128, 512, 1024, 2048) for c in (False, True)]
    done = sweep_done_keys(args.append)
    sweep_end_partial_line(args.append)
    cases = [cs for cs in cases if sweep_key(*cs) not in done]
    for T, d, c, dt in cases:
        p = W.grid(T, d, c, dt)
        g = torch.Generator(device=dev).manual_seed(0)
        q, k, v, do = (torch.randn(p.B, T, p.Hq, d, device=dev, generator=g).to(W.DTYPES[dt]) for _ in range(4))
        n = max(3, min(200, int(2e12 / max(W.fwd_flops(p), 1.0))))
        def fwd_call():
            return ea.forward(q, k, v, causal=c)

        def fwd_bwd_call():
            o2, lse2 = ea.forward(q, k, v, causal=c)
            return ea.backward(q, k, v, o2, lse2, do, causal=c)

        # the same step through the C-name calls into buffers allocated once:
        # no tensor allocation per call
        o3, lse3 = ea.forward(q, k, v, causal=c)
        ws3 = torch.empty(ea.attn_bwd_workspace_size(p.B, T, p.Hq, d, True, q.dtype), dtype=torch.uint8, device=dev)
        g3 = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))

        def fwd_bwd_prealloc():
            ea.attn_fwd(q, k, v, o3, lse3, causal=c)
            ea.attn_bwd(q, k, v, o3, lse3, do, *g3, ws3, causal=c)

        qf = timed(fwd_call, n)
        qb = timed(fwd_bwd_call, n)
        qp = timed(fwd_bwd_prealloc, n)
        gf = graph_timed(fwd_call, n)
        gb = graph_timed(fwd_bwd_call, n)
        F = W.fwd_flops(p)
        line = json.dumps({"T": T, "d": d, "causal": c, "dtype": dt, "fwd_ms": round(qf[1], 4),
                          "fwd_ms_q1_q3": [round(qf[0], 4), round(qf[2], 4)],
                          "fwd_tflops": round(F / qf[1] / 1e9, 1), "fwd_bwd_ms": round(qb[1], 4),
                          "fwd_bwd_ms_q1_q3": [round(qb[0], 4), round(qb[2], 4)],
                          "fwd_bwd_tflops": round(3.5 * F / qb[1] / 1e9, 1),
                          "prealloc_fwd_bwd_ms": round(qp[1], 4),
                          "graph_fwd_ms": round(gf[1], 4), "graph_fwd_tflops": round(F / gf[1] / 1e9, 1),
                          "graph_fwd_bwd_ms": round(gb[1], 4),
                          "graph_fwd_bwd_tflops": round(3.5 * F / gb[1] / 1e9, 1)})
        print(line, flush=True)
        if args.append:  # one line per finished case: a killed sweep resumes after it
            with open(args.append, "a") as f:
                f.write(line + "\n")


def _timed_q(fn, n, repeats=5):
    """(q1, median, q3) ms of `repeats` runs of n back-to-back calls (after 3 warm-up calls)."""
    import torch

    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    runs = []
    for _ in range(repeats):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(n):
            fn()
        b.record()
        torch.cuda.synchronize()
        runs.append(a.elapsed_time(b) / n)
    runs.sort()
    return runs[len(runs) // 4], runs[len(runs) // 2], runs[(3 * len(runs)) // 4]


def _call_peak_bytes(fn):
    """Device bytes one call allocates at its peak beyond what was live before it."""
    import torch

    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    out = fn()
    torch.cuda.synchronize()
    peak = torch.cuda.max_memory_allocated() - base
    del out
    torch.cuda.empty_cache()
    return peak


def run_gqa_suite(args):
    """The pages' GQA workload ("Attention performance", section "Grouped-query
    attention and decoding"): 32 query heads, head_dim 128, batch 1,
    Lq = Lkv = T, bf16, non-causal; 8 KV heads (native GQA: the kernels read KV
    head h // G) against 32 (plain multi-head).  Per case: fwd and fwd+bwd
    TFLOP/s (median of five repeats) and the device peak of one fwd+bwd call
    beyond its inputs; for GQA also the same call on K/V repeated to 32 heads
    (the repeat, the 32-head gradients and their sum over the group)."""
    import torch

    import exact_attention_34_gb300 as ea
    from exact_attention_34_gb300 import build as eb

    eb.build()
    dev = torch.device("cuda", 0)
    Hq, d = 32, 128
    for T in (1024, 2048, 4096, 8192, 16384):
        for Hkv in (8, 32):
            g = torch.Generator(device=dev).manual_seed(0)
            q = torch.randn(1, T, Hq, d, device=dev, generator=g).to(torch.bfloat16)
            k = torch.randn(1, T, Hkv, d, device=dev, generator=g).to(torch.bfloat16)
            v = torch.randn_like(k)
            do = torch.randn_like(q)
            o, lse = ea.forward(q, k, v)
            F = 4.0 * Hq * T * T * d
            n = max(3, min(100, int(5e11 / F)))
            qf = _timed_q(lambda: ea.forward(q, k, v), n)
            qb = _timed_q(lambda: (ea.forward(q, k, v), ea.backward(q, k, v, o, lse, do)), n)

            def native():
                o2, l2 = ea.forward(q, k, v)
                return ea.backward(q, k, v, o2, l2, do)

            line = {"suite": "gqa", "T": T, "Hq": Hq, "Hkv": Hkv, "d": d, "B": 1, "causal": False, "dtype": "bf16",
                    "fwd_ms": round(qf[1], 4), "fwd_tflops": round(F / qf[1] / 1e9, 1),
                    "fwd_bwd_ms": round(qb[1], 4), "fwd_bwd_ms_q1_q3": [round(qb[0], 4), round(qb[2], 4)],
                    "fwd_bwd_tflops": round(3.5 * F / qb[1] / 1e9, 1),
                    "peak_mb_fwd_bwd": round(_call_peak_bytes(native) / 2**20, 1)}
            if Hkv < Hq:
                G = Hq // Hkv

                def repeated():
                    kr, vr = k.repeat_interleave(G, dim=2), v.repeat_interleave(G, dim=2)
                    o2, l2 = ea.forward(q, kr, vr)
                    dq, dkr, dvr = ea.backward(q, kr, vr, o2, l2, do)
                    return dq, dkr.view(1, T, Hkv, G, d).sum(3), dvr.view(1, T, Hkv, G, d).sum(3)

                line["peak_mb_fwd_bwd_repeated_kv"] = round(_call_peak_bytes(repeated) / 2**20, 1)
            print(json.dumps(line), flush=True)
            del q, k, v, do, o, lse
            torch.cuda.empty_cache()


def run_memory_suite(args):
    """The pages' memory measurements ("Attention performance", section
    "Memory"): bf16, head_dim 64, 8 heads, non-causal.  (1) The device peak of
    one fwd+bwd call beyond its inputs at batch 4 for T = 1024 ... 65536 (the
    pages' search stops at 65,536; every T up to there runs).  (2) The bytes
    kept for the backward at batch 2: the output and the log-sum-exp (no T x T
    buffer), as allocated by the forward."""
    import torch

    import exact_attention_34_gb300 as ea
    from exact_attention_34_gb300 import build as eb

    eb.build()
    dev = torch.device("cuda", 0)
    H, d = 8, 64
    for T in (1024, 2048, 4096, 8192, 16384, 32768, 65536):
        g = torch.Generator(device=dev).manual_seed(0)
        q, k, v, do = (torch.randn(4, T, H, d, device=dev, generator=g).to(torch.bfloat16) for _ in range(4))

        def call():
            o, lse = ea.forward(q, k, v)
            return ea.backward(q, k, v, o, lse, do)

        peak = _call_peak_bytes(call)
        inputs = 4 * q.numel() * q.element_size()
        q2 = q[:2].contiguous()
        k2, v2 = k[:2].contiguous(), v[:2].contiguous()
        res = _call_peak_bytes(lambda: ea.forward(q2, k2, v2))
        print(json.dumps({"suite": "memory", "T": T, "H": H, "d": d, "dtype": "bf16", "causal": False,
                          "peak_mb_fwd_bwd_B4": round(peak / 2**20, 2), "inputs_mb_B4": round(inputs / 2**20, 2),
                          "residual_mb_B2": round(res / 2**20, 2),
                          "ran": True}), flush=True)
        del q, k, v, do, q2, k2, v2
        torch.cuda.empty_cache()


PROFILE_CASES = {
    # name: (workload, dtype, backward variant)
    "headline": ("B4 H8 T8192 d128 causal", "bf16", True),
    "single_pass": ("B4 H8 T8192 d128 causal", "bf16", False),
    "ordered": ("B4 H8 T8192 d128 causal", "bf16", 2),
    "fp32": ("B4 H8 T2048 d128", "fp32", True),
    "d64": ("B4 H8 T8192 d64 causal", "bf16", True),
}


def run_profile_suite(args):
    """A fixed number of fwd+bwd steps of one case, for profilers: no timing,
    no other rows.  `--case` picks the workload and backward variant (see
    PROFILE_CASES); each step is one forward and one backward call."""
    import torch

    import exact_attention_34_gb300 as ea
    from exact_attention_34_gb300 import build as eb

    eb.build()
    dev = torch.device("cuda", 0)
    _, dt, det = PROFILE_CASES[args.case]
    p = W.grid(2048, 128, False, "fp32") if dt == "fp32" else W.grid(8192, 64, True) if args.case == "d64" else \
        W.headline()
    g = torch.Generator(device=dev).manual_seed(0)
    q, k, v, do = (torch.randn(p.B, p.Lq, p.Hq, p.d, device=dev, generator=g).to(W.DTYPES[dt]) for _ in range(4))
    for _ in range(args.iters):
        o, lse = ea.forward(q, k, v, causal=p.causal)
        ea.backward(q, k, v, o, lse, do, causal=p.causal, deterministic=det)
    torch.cuda.synchronize()
    st, code, site = ea.attn_device_status()
    print(json.dumps({"suite": "profile", "case": args.case, "iters": args.iters, "device_status": code}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--kernel-steps", type=int, default=20, help="steps of the per-kernel timing pass")
    ap.add_argument("--cpu-budget-s", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--reference-budget-s", type=float, default=120.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the other rows (KVLen+GQA, decode)")
    ap.add_argument("--sweep", action="store_true", help="print the attention grid (one JSON line per case) and exit")
    ap.add_argument("--append", default=None,
                    help="with --sweep: also append each case's line to this file and skip cases already in it")
    ap.add_argument("--suite", choices=("gqa", "memory", "decode", "profile"),
                    help="print the GQA, the memory or the decode suite and exit; `profile` runs --iters steps of "
                         "--case for a profiler")
    ap.add_argument("--case", choices=tuple(PROFILE_CASES), default="headline", help="with --suite profile")
    ap.add_argument("--iters", type=int, default=3, help="with --suite profile: fwd+bwd steps to run")
    ap.add_argument("--decode-lkv", type=int, default=131072, help="cache length of --suite decode")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.sweep:
        run_sweep(args)
        return
    if args.suite:
        {"gqa": run_gqa_suite, "memory": run_memory_suite, "decode": run_decode_suite,
         "profile": run_profile_suite}[args.suite](args)
        return
    rank, _, world = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    res = run_reference(args) if args.impl == "reference" else run_gpu(args)
    if res is not None and rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
