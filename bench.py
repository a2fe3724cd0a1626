"""Benchmark of one sequence-parallel attention step on a GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload c5] [--impl ours|reference]
  python bench.py --sweep          # standalone exchange permute sweep, 1 MB .. 4 GB

A step is one pass of the whole path over one batch of synthetic input:
pad + mask -> tile -> send_recv_heads -> attention -> gather_heads ->
gather_output (cropped to the caller's length), all in the library's CUDA
kernels through the C ABI.  Inputs are resident in HBM when the timed region
starts (``value``); ``e2e`` repeats the measurement with pinned host inputs,
host->device copies of Q/K/V and the device->host copy of the output inside
the timed region.

Metric: masked-attention TFLOP/s per SP step (dense FLOPs 4*B*H*Tq*Tk*D on the
unpadded sequence, pad rows and columns not credited) with the head-exchange
GB/s (bytes read + written by send_recv_heads and gather_heads over their
kernel time) alongside.

Under torchrun (N > 1) every rank runs the same workload on its own GPU with
no collective on the data path (independent problems, weak scaling); the
barrier and the max-over-ranks timing reduction are the only collectives.
"""
from __future__ import annotations

import argparse
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

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "masked-attn TFLOP/s + head-exchange GB/s per SP step, 1 GB300"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "c5"
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)
        return False

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Max of a per-rank scalar (timing only; no data-path collective)."""
    if world <= 1:
        return x
    import torch.distributed as dist

    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(flops_per_rank: float, world: int, seconds_max: float) -> float:
    """Whole-job TFLOP/s: the units all ranks processed over the slowest rank's time."""
    return flops_per_rank * world / seconds_max / 1e12


def attention_traffic_bytes(name: str):
    """DRAM bytes (read + write) per attention launch from the committed ncu
    summary (profiles/attention_dram.md), or None when it has no row."""
    import re

    path = os.path.join(ROOT, "profiles", "attention_dram.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            m = re.match(r"\|\s*(c\d)\s*\|\s*([0-9.]+)\s*\|\s*([0-9.]+)\s*\|", line)
            if m and m.group(1) == name:
                return int(round((float(m.group(2)) + float(m.group(3))) * 1e6))
    return None


def workload_config(wl, world: int, big_inputs: bool) -> dict:
    return {
        "workload": f"{wl.name}: W={wl.W} virtual ranks, B={wl.B}, "
                    + (f"Tq={wl.Tq}, Tk={wl.T}" if wl.cross else f"T={wl.T}")
                    + f", H={wl.H}, D={wl.D}, {wl.dtype}, {wl.mask} mask",
        "W": wl.W, "B": wl.B, "T": wl.T, "Tq": wl.q_len, "H": wl.H, "D": wl.D,
        "parallelism": f"sp{wl.W} virtual ranks on 1 GPU" + (f", x{world} independent replicas" if world > 1 else ""),
        "l2": "inputs larger than L2" if big_inputs else f"L2 flushed between steps ({L2_FLUSH_BYTES >> 20} MB write)",
    }


def inputs_exceed_l2(wl) -> bool:
    in_bytes = (wl.q_len + 2 * wl.T) * wl.B * wl.H * wl.D * wl.elt
    return in_bytes > 2 * L2_FLUSH_BYTES


# ---------------------------------------------------------------- CPU oracle
def oracle_sample_tflops(wl, budget_s: float, threads: int, seed: int = 0):
    """Oracle attention on a bounded random sample of output rows of the
    workload (each row over the full key sequence); returns (TFLOP/s, rows, s)."""
    import numpy as np

    import oracle

    inp = workloads.make_inputs(wl)
    q, k, v = (inp[n].float().numpy() for n in ("q", "k", "v"))
    rng = np.random.default_rng(seed)
    um = inp["user_mask"]
    kind, mask = (oracle.MASK_FULL, um.numpy()) if um is not None else (oracle.MASK_NONE, None)

    def rows(n):
        return np.stack([rng.integers(0, wl.B, n), rng.integers(0, wl.q_len, n), rng.integers(0, wl.H, n)], 1)

    n = max(threads, 8)
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, rows(n), kind, mask, threads=threads)
    dt = time.perf_counter() - t0
    n2 = max(n, int(n * budget_s / max(dt, 1e-6)))
    t0 = time.perf_counter()
    oracle.attention_rows(q, k, v, rows(n2), kind, mask, threads=threads)
    dt2 = time.perf_counter() - t0
    flops = 4.0 * wl.T * wl.D * n2
    return flops / dt2 / 1e12, n2, dt2


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import sequence_video_dit_gb300 as sp
    from sequence_video_dit_gb300.step import StageTimer

    wl = workloads.get(args.workload)
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = workloads.make_inputs(wl)
    host = {n: inp[n].pin_memory() for n in ("q", "k", "v")}
    um_host = inp["user_mask"].pin_memory() if inp["user_mask"] is not None else None
    d_in = {n: host[n].to(dev) for n in host}
    d_um = um_host.to(dev) if um_host is not None else None
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq, device=dev)
    out_host = torch.empty(step.out.shape, dtype=step.out.dtype).pin_memory()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    in_bytes = sum(t.numel() * t.element_size() for t in d_in.values())
    big_inputs = inputs_exceed_l2(wl)
    flops = wl.flops()

    def one(timer=None):
        step(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um, timer=timer)

    for _ in range(args.warmup):
        one()
    torch.cuda.synchronize()
    st = sp.sp_workspace_status(step.ws_exchange)[0] | sp.sp_workspace_status(step.ws_attn)[0]
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")

    # ---- device-resident timed region: K steps, per-stage events
    timer = StageTimer()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    n0 = sp.lib().sp_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            if not big_inputs:
                flush.zero_()  # L2 flush between steps, outside the step's events
            starts[i].record()
            one(timer)
            ends[i].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)
    launches = int(sp.lib().sp_launch_count() - n0)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    ms_max = max_over_ranks(ms, world)
    stage_ms = timer.totals_ms()
    stage_n = timer.counts()
    attn_ms = stage_ms["attention"] / stage_n["attention"]
    x_ms = stage_ms.get("send_recv_heads", 0.0) + stage_ms.get("gather_heads", 0.0)
    x_bytes = step.exchange_bytes_per_launch() * step.n_exchange_launches() * args.steps
    exch_gbs = x_bytes / (x_ms / 1e3) / 1e9 if x_ms > 0 else None

    # ---- the same step through the fused exchange entry points (pad + tile +
    # exchange in one pass per tensor; inverse exchange + gather + unpad in one)
    fused = time_fused_step(wl, d_in, d_um, dev, args, world, flops, big_inputs, flush)
    direct = time_fused_step(wl, d_in, d_um, dev, args, world, flops, big_inputs, flush, direct=True) \
        if direct_eligible(wl, world) else None
    graphed = time_graph_step(step, d_in, d_um, args, world, flops, big_inputs, flush)
    # ---- end to end: pinned host inputs copied in and the output copied out
    # every step, inside the timed region.  Copies run on their own stream so
    # step i+1's uploads and step i's download overlap step i's compute (two
    # input and two output buffers, ordered by events), as a streaming user
    # of the library would run it.
    h2d = in_bytes + (um_host.numel() if um_host is not None else 0)
    d2h = out_host.numel() * out_host.element_size()
    e2e_ms = run_e2e_pipelined(step, host, um_host, out_host, args.steps, world, dev)
    peaks = load_peaks()
    achieved = flops / (attn_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops_sustained"]
    traffic = attention_traffic_bytes(wl.name)
    result = {
        "metric": METRIC,
        "value": round(weak_scaling_value(flops, world, ms_max / 1e3), 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) inputs shaped like the workload; no weights involved)",
        "config": workload_config(wl, world, big_inputs),
        "head_exchange": {"value": round(exch_gbs, 1) if exch_gbs else None, "unit": "GB/s",
                          "launches_per_step": step.n_exchange_launches(),
                          "bytes_per_launch": step.exchange_bytes_per_launch()},
        "stage_ms": {k: round(v / stage_n[k], 4) for k, v in stage_ms.items()},
        "fused_step": fused,
        "direct_step": direct,
        "graph_step": graphed,
        "e2e": {"value": round(weak_scaling_value(flops, world, e2e_ms / 1e3), 3), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "copies": "pinned host buffers; H2D of step i+1 and D2H of step i overlap step i's compute"},
        "gpu_launches": launches,
        "roofline": {"bound": "tensor", "kernel": "attn_tc_kernel", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_kind": f"bf16 sustained, {peaks['source']}",
                     "algorithmic_flops_per_launch": flops},
        "clocks": clk.summary(),
        "wall_s_timed": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        tf, nrows, secs = oracle_sample_tflops(wl, args.cpu_budget, threads)
        result["cpu_baseline"] = {"value": round(tf, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                                  "sample": f"{nrows} random output rows of {wl.name}, each over all {wl.T} keys "
                                            f"(fp64 C oracle, {secs:.1f} s)"}
    return result


def direct_eligible(wl, world=1) -> bool:
    """The exchange-free step (attention reading the callers' tensors as token
    shards) applies when the shards are whole 128-row tiles and need no pad."""
    return (wl.dtype == "bf16" and wl.D in (64, 128) and wl.T % wl.W == 0 and (wl.T // wl.W) % 128 == 0
            and wl.mask == "key")


def time_fused_step(wl, d_in, d_um, dev, args, world, flops, big_inputs, flush, direct=False) -> dict:
    """Device-resident timing of the step built with ``fused=True`` (and with
    ``direct=True``: the exchange fused into the attention, in place), same
    inputs and the same output bits, reported beside the staged step."""
    import sequence_video_dit_gb300 as sp
    from sequence_video_dit_gb300.step import StageTimer

    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq, device=dev,
                     fused=True, direct=direct)
    for _ in range(args.warmup):
        step(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um)
    timer = StageTimer()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    n0 = sp.lib().sp_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        if not big_inputs:
            flush.zero_()
        starts[i].record()
        step(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um, timer=timer)
        ends[i].record()
    torch.cuda.synchronize()
    barrier(world)
    launches = int(sp.lib().sp_launch_count() - n0)
    st = sp.sp_workspace_status(step.ws_exchange)[0] | sp.sp_workspace_status(step.ws_attn)[0]
    if st != 0:
        raise RuntimeError(f"device status {st} after the fused step")
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps, world)
    tot, cnt = timer.totals_ms(), timer.counts()
    out = {"value": round(weak_scaling_value(flops, world, ms / 1e3), 3), "unit": UNIT, "ms_per_step": round(ms, 4),
           "stage_ms": {k: round(v / cnt[k], 4) for k, v in tot.items()}, "gpu_launches": launches}
    del step
    torch.cuda.empty_cache()
    return out


def time_graph_step(step, d_in, d_um, args, world, flops, big_inputs, flush) -> dict:
    """The staged step captured once as a CUDA graph and replayed: the same
    kernels with one host launch per step (what latency-bound shapes gain)."""
    import sequence_video_dit_gb300 as sp

    n0 = sp.lib().sp_launch_count()
    step(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um)
    per_step = int(sp.lib().sp_launch_count() - n0)
    g = step.capture(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um)
    for _ in range(args.warmup):
        g.replay()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        if not big_inputs:
            flush.zero_()
        starts[i].record()
        g.replay()
        ends[i].record()
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / args.steps, world)
    del g
    return {"value": round(weak_scaling_value(flops, world, ms / 1e3), 3), "unit": UNIT, "ms_per_step": round(ms, 4),
            "kernels_per_replay": per_step}


def run_e2e_pipelined(step, host, um_host, out_host, steps: int, world: int, dev) -> float:
    """Mean ms per step of `steps` end-to-end steps (H2D of every step's inputs,
    the step, D2H of its output), copies overlapped with compute."""
    main = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(device=dev)
    d_in = [{n: torch.empty_like(host[n], device=dev) for n in host} for _ in range(2)]
    d_um = [um_host.to(dev) if um_host is not None else None for _ in range(2)]
    d_out = [torch.empty_like(step.out) for _ in range(2)]
    out_pin = [out_host, torch.empty_like(out_host).pin_memory()]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def upload(slot):
        for n in host:
            d_in[slot][n].copy_(host[n], non_blocking=True)
        if um_host is not None:
            d_um[slot].copy_(um_host, non_blocking=True)
        ev_in[slot].record(copy)

    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(main)
    copy.wait_event(t0)
    with torch.cuda.stream(copy):
        upload(0)
    for i in range(steps):
        b = i % 2
        main.wait_event(ev_in[b])
        if i >= 2:
            main.wait_event(ev_d2h[b])  # d_out[b] is free again
        step(d_in[b]["q"], d_in[b]["k"], d_in[b]["v"], user_mask=d_um[b], out=d_out[b])
        ev_done[b].record(main)
        with torch.cuda.stream(copy):
            if i + 1 < steps:
                if i >= 1:
                    copy.wait_event(ev_done[1 - b])  # step i-1 is done with d_in[1-b]
                upload(1 - b)
            copy.wait_event(ev_done[b])
            out_pin[b].copy_(d_out[b], non_blocking=True)
            ev_d2h[b].record(copy)
    main.wait_stream(copy)
    t1.record(main)
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(t0.elapsed_time(t1) / steps, world)


# ---------------------------------------------------------------- reference arm (the oracle)
def run_reference(args, world, rank):
    wl = workloads.get(args.workload)
    if rank != 0:
        return None
    threads = os.cpu_count() or 1
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample_tflops(wl, per_step / 4, threads, seed=1)
    vals, secs, rows = [], 0.0, 0
    for i in range(args.steps):
        tf, n, s = oracle_sample_tflops(wl, per_step, threads, seed=100 + i)
        vals.append(tf)
        secs += s
        rows += n
    v = statistics.mean(vals)
    sample = f"{rows} random output rows of {wl.name} over {args.steps} steps, each row over all {wl.T} keys"
    return {
        "metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
        "data": "synthetic (seeded N(0,1) inputs shaped like the workload)",
        "config": workload_config(wl, world, inputs_exceed_l2(wl)),
        "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------- exchange sweep
def run_sweep(args):
    import sequence_video_dit_gb300 as sp

    dev = torch.device("cuda", torch.cuda.current_device())
    W, H, D = 8, 32, 128
    ws = sp.new_workspace(device=dev)
    peaks = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    for mb in [1, 4, 16, 64, 256, 1024, 4096]:
        tokens = mb * (1 << 20) // (H * D * 2)
        Tl = tokens // W
        shards = [torch.randn(1, Tl, H, D, device=dev).bfloat16() for _ in range(W)]
        heads = [torch.empty(1, W * Tl, H // W, D, dtype=torch.bfloat16, device=dev) for _ in range(W)]
        for _ in range(3):
            sp.sp_send_recv_heads(shards, heads, ws)
        reps = max(3, min(50, int(2e9 // (mb << 20))))
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * reps)]
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        for i in range(reps):
            flush.zero_()
            ev[2 * i][0].record()
            sp.sp_send_recv_heads(shards, heads, ws)
            ev[2 * i][1].record()
            flush.zero_()
            ev[2 * i + 1][0].record()
            sp.sp_gather_heads(heads, shards, ws)
            ev[2 * i + 1][1].record()
        torch.cuda.synchronize()
        t_send = statistics.median(s.elapsed_time(e) for s, e in ev[0::2])
        t_gath = statistics.median(s.elapsed_time(e) for s, e in ev[1::2])
        nbytes = 2 * Tl * W * H * D * 2
        line = {"sweep": "exchange", "mbytes": mb, "tokens": Tl * W,
                "send_gbs": round(nbytes / t_send / 1e6, 1), "gather_gbs": round(nbytes / t_gath / 1e6, 1),
                "send_ms": round(t_send, 4), "gather_ms": round(t_gath, 4),
                "hbm_frac_send": round(nbytes / t_send / 1e6 / peaks["hbm_gbs"], 3),
                "l2_resident": (mb << 20) < 4 * l2}
        print(json.dumps(line), flush=True)
        del shards, heads
        torch.cuda.empty_cache()
    st = sp.sp_workspace_status(ws)[0]
    if st:
        raise RuntimeError(f"exchange status {st}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours" and not args.sweep:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    world, rank, local = dist_setup(args.gpus)
    if args.sweep:
        if rank == 0:
            run_sweep(args)
        return
    res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
