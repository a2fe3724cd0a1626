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

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "masked-attn TFLOP/s + head-exchange GB/s per SP step, 1 GB300"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "c5"
L2_FLUSH_BYTES = 512 << 20
E2E_REPEATS = 3  # timed runs of the end-to-end loop; the line reports their median


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


# DRAM traffic of the attention kernel comes from one ncu capture, recorded
# as JSON beside the profiles together with a digest of the kernel's source;
# a record taken on other source is stale and gives no traffic figure.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "attention_dram.json")
ATTN_SOURCES = ("sequence_video_dit_gb300/csrc/sp_attn_tc.cu", "sequence_video_dit_gb300/csrc/sp_attn.cuh",
                "sequence_video_dit_gb300/csrc/sp_internal.cuh")


def attention_source_digest() -> str:
    h = hashlib.sha256()
    for rel in ATTN_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def attention_traffic(name: str):
    """(DRAM bytes read + written per attention launch, provenance) for
    workload `name`, or (None, why not)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no ncu record"
    with open(TRAFFIC_FILE) as f:
        rec = json.load(f).get(name)
    if not rec:
        return None, f"no ncu record for {name}"
    if rec.get("source_digest") != attention_source_digest():
        return None, "ncu record taken on other attention source (stale)"
    return int(rec["dram_bytes_per_launch"]), f"ncu, attention source {rec['source_digest']}"


_UNIT_SCALE = {"byte": 1, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12}


def record_traffic(csv_path: str, name: str, command: str) -> dict:
    """Reads an ncu --csv metrics log (dram__bytes_read.sum and
    dram__bytes_write.sum of attn_tc_kernel launches) and stores the mean
    per-launch traffic for workload `name` in the JSON record."""
    import csv

    per_launch = {}
    with open(csv_path, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    head = next(i for i, r in enumerate(rows) if "Metric Name" in r)
    cols = rows[head]
    c_id, c_k, c_m, c_u, c_v = (cols.index(n) for n in ("ID", "Kernel Name", "Metric Name", "Metric Unit",
                                                         "Metric Value"))
    for r in rows[head + 1:]:
        if len(r) <= c_v or "attn_tc_kernel" not in r[c_k]:
            continue
        if r[c_m] not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        val = float(r[c_v].replace(",", "")) * _UNIT_SCALE.get(r[c_u].strip().lower(), 1)
        per_launch.setdefault(r[c_id], {})[r[c_m]] = val
    full = [d for d in per_launch.values() if len(d) == 2]
    if not full:
        raise SystemExit(f"no attn_tc_kernel DRAM counters in {csv_path}")
    rd = statistics.mean(d["dram__bytes_read.sum"] for d in full)
    wr = statistics.mean(d["dram__bytes_write.sum"] for d in full)
    data = {}
    if os.path.exists(TRAFFIC_FILE):
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
    data[name] = {"kernel": "attn_tc_kernel", "launches": len(full), "dram_read_bytes": int(rd),
                  "dram_write_bytes": int(wr), "dram_bytes_per_launch": int(rd + wr),
                  "source_digest": attention_source_digest(), "command": command}
    with open(TRAFFIC_FILE, "w") as f:
        json.dump(data, f, indent=1, sort_keys=True)
        f.write("\n")
    return data[name]


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

    # ---- end to end, right after the device-resident steps (same state of the
    # GPU): pinned host inputs copied in and the output copied out every step,
    # inside the timed region.  Uploads and downloads run on two copy streams,
    # so step i+1's uploads and step i-1's download overlap step i's compute
    # (two input and two output buffers, ordered by events), as a streaming
    # user of the library would run it.
    h2d = in_bytes + (um_host.numel() if um_host is not None else 0)
    d2h = out_host.numel() * out_host.element_size()
    with ClockSampler(dev.index) as clk_e2e:
        e2e_runs = run_e2e_pipelined(step, host, um_host, out_host, args.steps, world, dev, warmup=args.warmup,
                                     repeats=E2E_REPEATS)
    e2e_ms = statistics.median(e2e_runs)
    link = measure_link(host, out_host, dev)
    # ---- the same step through the fused exchange entry points (pad + tile +
    # exchange in one pass per tensor; inverse exchange + gather + unpad in one)
    fused, direct = time_variants(wl, d_in, d_um, dev, args, world, flops, big_inputs, flush,
                                  with_direct=direct_eligible(wl, world))
    graphed = time_graph_step(step, d_in, d_um, args, world, flops, big_inputs, flush)
    # lower bound of the pipelined end-to-end step: the slower of the device
    # step (eager or graph-replayed, whichever is faster: the end-to-end loop
    # replays graphs) and the step's copies over the link (both directions at once)
    e2e_bound_ms = max(min(ms, graphed["ms_per_step"]), link["both_directions_ms"])
    peaks = load_peaks()
    achieved = flops / (attn_ms / 1e3) / 1e12
    peak = peaks["bf16_tflops_sustained"]
    traffic, traffic_src = attention_traffic(wl.name)
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
                "copies": "pinned host buffers on two copy streams; H2D of step i+1 and D2H of step i-1 overlap "
                          "step i's compute (the step replayed from a CUDA graph per buffer set)",
                "runs_ms_per_step": [round(x, 4) for x in e2e_runs],
                "timing": f"median of {E2E_REPEATS} timed runs of {args.steps} steps each, after "
                          f"{args.warmup} warm-up steps of the same pipeline",
                "link": link, "bound_ms_per_step": round(e2e_bound_ms, 4),
                "frac_of_bound": round(e2e_bound_ms / e2e_ms, 4), "clocks": clk_e2e.summary()},
        "gpu_launches": launches,
        "roofline": {"bound": "tensor", "kernel": "attn_tc_kernel", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                     "traffic_source": traffic_src, "peak_kind": f"bf16 sustained, {peaks['source']}",
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
    """The exchange-free step (attention reading the callers' tensors in place
    as token shards) needs the tensor-core kernel: bf16, D = 64 or 128."""
    return wl.dtype == "bf16" and wl.D in (64, 128)


def time_variants(wl, d_in, d_um, dev, args, world, flops, big_inputs, flush, with_direct=True):
    """Device-resident timing of the step built with ``fused=True`` and of the
    one with ``direct=True, fused=True`` (the exchange inside the attention, in
    place), on the same inputs.  Their steps alternate inside one timed loop,
    so a slow drift of the clocks over the run affects both alike."""
    import sequence_video_dit_gb300 as sp
    from sequence_video_dit_gb300.step import StageTimer

    steps = {"fused": sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq,
                                device=dev, fused=True)}
    if with_direct:
        steps["direct"] = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq,
                                    device=dev, fused=True, direct=True)
    for _ in range(args.warmup):
        for st in steps.values():
            st(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um)
    timers = {n: StageTimer() for n in steps}
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)] for n in steps}
    launches = {n: 0 for n in steps}
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        for n, st in steps.items():
            if not big_inputs:
                flush.zero_()
            n0 = sp.lib().sp_launch_count()
            ev[n][i][0].record()
            st(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um, timer=timers[n])
            ev[n][i][1].record()
            launches[n] += int(sp.lib().sp_launch_count() - n0)
    torch.cuda.synchronize()
    barrier(world)
    out = {}
    for n, st in steps.items():
        code = sp.sp_workspace_status(st.ws_exchange)[0] | sp.sp_workspace_status(st.ws_attn)[0]
        if code != 0:
            raise RuntimeError(f"device status {code} after the {n} step")
        ms = max_over_ranks(sum(a.elapsed_time(z) for a, z in ev[n]) / args.steps, world)
        tot, cnt = timers[n].totals_ms(), timers[n].counts()
        out[n] = {"value": round(weak_scaling_value(flops, world, ms / 1e3), 3), "unit": UNIT,
                  "ms_per_step": round(ms, 4), "stage_ms": {k: round(v / cnt[k], 4) for k, v in tot.items()},
                  "gpu_launches": launches[n]}
    del steps
    torch.cuda.empty_cache()
    return out["fused"], out.get("direct")


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


def run_e2e_pipelined(step, host, um_host, out_host, steps: int, world: int, dev, warmup: int = 3,
                      repeats: int = 1) -> list:
    """Mean ms per step of `steps` end-to-end steps (H2D of every step's inputs,
    the step, D2H of its output), after `warmup` untimed runs of the same
    pipeline; `repeats` timed runs of `steps` steps each, one figure per run.  Two input and two output buffer sets, each with the step
    captured once as a CUDA graph (SPStep.capture), so the host issues one
    replay per step.  Uploads and downloads run on two copy streams of their
    own: step i+1's uploads, step i's compute and step i-1's download can all
    be in flight at once (ordered by events)."""
    main = torch.cuda.current_stream(dev)
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    d_in = [{n: torch.empty_like(host[n], device=dev) for n in host} for _ in range(2)]
    d_um = [um_host.to(dev) if um_host is not None else None for _ in range(2)]
    d_out = [torch.empty_like(step.out) for _ in range(2)]
    out_pin = [out_host, torch.empty_like(out_host).pin_memory()]
    for b in range(2):
        for n in host:
            d_in[b][n].copy_(host[n])
    graphs = [step.capture(d_in[b]["q"], d_in[b]["k"], d_in[b]["v"], user_mask=d_um[b], out=d_out[b])
              for b in range(2)]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def upload(slot):
        with torch.cuda.stream(up):
            for n in host:
                d_in[slot][n].copy_(host[n], non_blocking=True)
            if um_host is not None:
                d_um[slot].copy_(um_host, non_blocking=True)
            ev_in[slot].record(up)

    def pipeline(n, t0, t1):
        t0.record(main)
        up.wait_event(t0)
        down.wait_event(t0)
        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                if i >= 1:
                    up.wait_event(ev_done[1 - b])  # step i-1 is done with d_in[1-b]
                upload(1 - b)
            main.wait_event(ev_in[b])
            if i >= 2:
                main.wait_event(ev_d2h[b])  # step i-2's output has left d_out[b]
            graphs[b].replay()
            ev_done[b].record(main)
            down.wait_event(ev_done[b])
            with torch.cuda.stream(down):
                out_pin[b].copy_(d_out[b], non_blocking=True)
                ev_d2h[b].record(down)
        main.wait_stream(up)
        main.wait_stream(down)
        t1.record(main)

    torch.cuda.synchronize()
    if warmup > 0:
        pipeline(warmup, torch.cuda.Event(), torch.cuda.Event())
    runs = []
    for _ in range(repeats):
        barrier(world)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        pipeline(steps, t0, t1)
        torch.cuda.synchronize()
        barrier(world)
        runs.append(max_over_ranks(t0.elapsed_time(t1) / steps, world))
    del graphs
    return runs


def measure_link(host, out_host, dev, reps: int = 3) -> dict:
    """Host link bandwidth for this step's copies, measured with plain pinned
    copies of the same tensors: uploads alone, the download alone, and both
    directions at once on two streams (best of `reps`, CUDA events)."""
    d_in = {n: torch.empty_like(host[n], device=dev) for n in host}
    d_out = torch.empty(out_host.shape, dtype=out_host.dtype, device=dev)
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host.numel() * out_host.element_size()

    def timed(do_up, do_down):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            main = torch.cuda.current_stream(dev)
            a.record(main)
            up.wait_event(a)
            down.wait_event(a)
            if do_up:
                with torch.cuda.stream(up):
                    for n in host:
                        d_in[n].copy_(host[n], non_blocking=True)
            if do_down:
                with torch.cuda.stream(down):
                    out_host.copy_(d_out, non_blocking=True)
            main.wait_stream(up)
            main.wait_stream(down)
            z.record(main)
            torch.cuda.synchronize()
            best = min(best, a.elapsed_time(z))
        return best

    t_up, t_down, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_gbs": round(h2d / t_up / 1e6, 1), "d2h_gbs": round(d2h / t_down / 1e6, 1),
            "h2d_ms": round(t_up, 3), "d2h_ms": round(t_down, 3), "both_directions_ms": round(t_both, 3)}


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


def run_profile(args):
    """`--steps` steps of one variant of the step (staged, fused or direct)
    on the workload's inputs, with no timing and no output: a short program
    for ncu captures of single kernels."""
    import sequence_video_dit_gb300 as sp

    wl = workloads.get(args.workload)
    if args.tokens:  # the workload's shape with a shorter sequence (a small case for long captures)
        wl = workloads.make_custom(f"{wl.name}-T{args.tokens}", W=wl.W, B=wl.B, T=args.tokens, H=wl.H, D=wl.D,
                                   dtype=wl.dtype, mask=wl.mask, Tq=wl.Tq, input_scale=wl.input_scale,
                                   index=wl.index)
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = workloads.make_inputs(wl)
    d_in = {n: inp[n].to(dev) for n in ("q", "k", "v")}
    d_um = inp["user_mask"].to(dev) if inp["user_mask"] is not None else None
    step = sp.SPStep(wl.W, wl.B, wl.T, wl.H, wl.D, dtype=wl.torch_dtype, mask=wl.mask, Tq=wl.Tq, device=dev,
                     fused=args.profile in ("fused", "direct"), direct=args.profile == "direct")
    for _ in range(args.steps):
        step(d_in["q"], d_in["k"], d_in["v"], user_mask=d_um)
    torch.cuda.synchronize()
    st = sp.sp_workspace_status(step.ws_exchange)[0] | sp.sp_workspace_status(step.ws_attn)[0]
    if st != 0:
        raise RuntimeError(f"device status {st}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--profile", choices=["staged", "fused", "direct"],
                    help="run --steps steps of this step variant untimed (a target for ncu) and exit")
    ap.add_argument("--tokens", type=int, default=0,
                    help="with --profile: the workload's shape with this sequence length instead")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="store the attention kernel's DRAM bytes per launch from an ncu --csv metrics log "
                         "(taken on --workload) and exit")
    ap.add_argument("--traffic-command", default="", help="the ncu command that wrote NCU_CSV (stored with it)")
    args = ap.parse_args()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, args.workload, args.traffic_command)))
        return
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
    if args.profile:
        run_profile(args)
        return
    res = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
