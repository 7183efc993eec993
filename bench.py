"""Throughput bench for the exact attention forward on GB300.

One step = one attention forward (QK^T, online softmax, PV, epilogue: the
whole path) over one batch of seeded synthetic inputs already resident in
device memory.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference]

Metric: TFLOP/s with FLOP = 4*B*H*N^2*d (halved with the causal mask).
``--impl reference`` times the float64 CPU oracle on the host cores on a
bounded sample of the same workload (the only other place this file runs the
oracle besides the ``cpu_baseline`` leg).
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
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attention_attn_fwd_05_gb300.inputs import WORKLOADS, make_workload_inputs  # noqa: E402

DEFAULT_WORKLOAD = "bf16_B1_H32_N16384_d128_causal"
METRIC = "attention fwd TFLOP/s (4*B*H*N^2*d, causal halved) and % of GB300 bf16 peak"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_BF16_DENSE_TFLOPS = 2250.0  # GB300 tensor cores, dense bf16, nominal
KERNEL_SRC = {"bf16": "attention_attn_fwd_05_gb300/csrc/attn_fwd_tc.cu",
              "f32": "attention_attn_fwd_05_gb300/csrc/attn_fwd_f32.cu"}
KERNEL_NAME = {"bf16": "attn_fwd_bf16_tc_kernel", "f32": "attn_fwd_f32_kernel"}


# ----------------------------------------------------------------- helpers ---

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, device=None):
    """Element-wise maximum of `values` over all ranks of the initialised
    process group (the slowest rank's time is the job's time); the values
    themselves with one rank."""
    t = torch.tensor([float(x) for x in values], dtype=torch.float64)
    import torch.distributed as tdist
    if tdist.is_available() and tdist.is_initialized() and tdist.get_world_size() > 1:
        if device is not None:
            t = t.to(device)
        tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Throughput of the whole job: every rank processes `units_per_rank`
    (weak scaling) and the job takes the slowest rank's `seconds`."""
    return units_per_rank * world / seconds


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_hash(dtype: str) -> str:
    with open(os.path.join(ROOT, KERNEL_SRC[dtype]), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_value(dtype: str, workload: str, key: str, kernel: str = None):
    """A figure (``key: value`` line) from the committed ncu summary for this
    kernel (by default the dtype's main kernel) and workload, or None when
    there is none or the kernel source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", f"{kernel or KERNEL_NAME[dtype]}_{workload}.md")
    if not os.path.exists(p):
        return None
    text = open(p).read()
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    t = re.search(key + r":\s*([0-9.eE+]+)", text)
    if not h or not t or h.group(1) != kernel_hash(dtype):
        return None
    return float(t.group(1))


def profiled_traffic(dtype: str, workload: str, kernel: str = None):
    """DRAM bytes per launch (read + write) from the committed ncu summary."""
    return profiled_value(dtype, workload, "traffic_bytes_per_launch", kernel)


class ClockSampler:
    """nvidia-smi samples (every 10 ms) of SM clock, power and throttle reasons
    around a region.  ``mark_start``/``mark_end`` bracket the timed region on
    the host clock, so the summary can say how many samples fell inside it."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 10

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"attn_clocks_{os.getpid()}.csv")
        self.t_start = self.t_end = None

    def __enter__(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.PERIOD_MS)],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    @staticmethod
    def _epoch(stamp: str):
        """nvidia-smi timestamp ('YYYY/MM/DD HH:MM:SS.mmm', local time) -> epoch s."""
        import datetime
        try:
            return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((self._epoch(parts[0]), float(parts[2]), float(parts[3]),
                             float(parts[4]), parts[6:10]))
            except ValueError:
                continue
        os.remove(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        max_mhz = max(r[2] for r in rows)
        inside = []
        if self.t_start is not None and self.t_end is not None:
            inside = [r for r in rows if r[0] is not None and self.t_start <= r[0] <= self.t_end]
        loaded = [r for r in rows if r[3] > 200.0]
        # Clocks reported: the samples inside the timed region, else those
        # under load, else all.
        use = inside or loaded or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in (inside or loaded or rows) for i, v in enumerate(r[4])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max_mhz,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "samples_in_timed_region": len(inside),
                "timed_region_s": (self.t_end - self.t_start)
                if self.t_start is not None and self.t_end is not None else None,
                "period_ms": self.PERIOD_MS,
                "basis": "timed region" if inside else ("under load" if loaded else "all")}


# ------------------------------------------------------------- CPU oracle ---

def sample_rows(w, n_rows: int, seed: int = 0):
    """A deterministic spread of (bh, row) pairs covering every position range."""
    rng = np.random.default_rng(seed)
    BH = w.B * w.H
    bh = rng.integers(0, BH, size=n_rows)
    rows = np.linspace(0, w.N - 1, n_rows).round().astype(np.int64)
    return bh.astype(np.int64), rows


def sample_flops(w, rows) -> float:
    visible = (rows + 1) if w.causal else np.full(rows.shape, w.N)
    return float(4.0 * w.d * visible.sum())


def time_oracle(w, q, k, v, budget_s: float):
    """Time the oracle, as it stands, on a row sample sized to ~budget_s seconds."""
    import oracle
    cores = oracle.max_threads()
    n_cal = 8 * cores
    bh, rows = sample_rows(w, n_cal, seed=1)
    oracle.attn_fwd_rows(q, k, v, w.scale, w.causal, bh[:cores], rows[:cores])  # warm threads
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q, k, v, w.scale, w.causal, bh, rows)
    t_cal = time.perf_counter() - t0
    n = int(min(w.B * w.H * w.N, max(cores, n_cal * budget_s / max(t_cal, 1e-6))))
    bh, rows = sample_rows(w, n, seed=2)
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(q, k, v, w.scale, w.causal, bh, rows)
    dt = time.perf_counter() - t0
    return sample_flops(w, rows) / dt / 1e12, cores, n, dt


# ------------------------------------------------------------------ arms ---

def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    q, k, v = make_workload_inputs(w)
    # About a minute of oracle work for short runs (2 s per step at most), and
    # 0.5 s per step for long ones, so a 200-step run ends in about two minutes.
    per_step = min(2.0, max(0.5, 60.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(w, q, k, v, min(per_step, 2.0))
    vals, samples = [], []
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tf, cores, n, dt = time_oracle(w, q, k, v, per_step)
        vals.append(tf)
        samples.append((n, dt))
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall * 1e3 / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{samples[-1][0]} query rows of {w.name} spread over all "
                                   f"positions, {samples[-1][1]:.1f} s per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    io = w.io_bytes
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "dtype": w.dtype, "inputs": w.dist, "seed": w.seed,
            "global_batch": w.B, "seq_len": w.N, "parallelism": "replicas (weak)",
            "l2": ("inputs+outputs %.0f MB > %d MB L2, no flush" % (io / 1e6, L2_BYTES >> 20))
            if io > 2 * L2_BYTES else "L2 flushed (256 MB write) before each timed step"}


def kernels_per_call(w, sms: int) -> list:
    """Kernels one attn_fwd call launches.  bf16: the main kernel for whole
    waves of 256-row items, and the split-CTA kernel when some items go to
    split CTAs (all items of a grid filling at most half the SMs; without the
    causal mask, also a last wave filling at most half of them).  fp32: one
    kernel."""
    if w.dtype != "bf16":
        return [KERNEL_NAME["f32"]]
    n_items = w.B * w.H * ((w.N + 255) // 256)
    if 2 * n_items <= sms:
        n_split = n_items
    elif not w.causal and 0 < n_items % sms and 2 * (n_items % sms) <= sms:
        n_split = n_items % sms
    else:
        n_split = 0
    names = [KERNEL_NAME["bf16"]] if n_items - n_split > 0 else []
    return names + (["attn_fwd_bf16_tc_split_kernel"] if n_split > 0 else [])


def launches_per_call(w, sms: int) -> int:
    return len(kernels_per_call(w, sms))


EAGER_MAX_SCORE_BYTES = 64 << 30  # S alone; S and P together at most 128 GiB


def eager_context(w, qd, kd, vd, our_ms: float, our_extra: int, dev, reps: int = 5):
    """The pages' own baseline re-run on this GPU, as context only: PyTorch
    eager fp32 softmax(scale * Q K^T) V with S and P materialised (inputs
    upcast to fp32, no TF32), timed with CUDA events, and the device memory it
    takes beyond its inputs.  Not part of `value` and never a fallback."""
    scores = w.B * w.H * w.N * w.N * 4
    if scores > EAGER_MAX_SCORE_BYTES:
        return {"skipped": f"S and P would need {2 * scores / 2**30:.1f} GiB"}
    q32, k32, v32 = (t.float() for t in (qd, kd, vd))
    mask = torch.ones(w.N, w.N, dtype=torch.bool, device=dev).triu_(1) if w.causal else None

    def run():
        s_ = torch.matmul(q32, k32.transpose(-1, -2)) * w.scale
        if mask is not None:
            s_ = s_.masked_fill(mask, float("-inf"))
        return torch.matmul(torch.softmax(s_, dim=-1), v32)

    tf32 = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        run()
        torch.cuda.synchronize(dev)
        base = torch.cuda.memory_allocated(dev)
        torch.cuda.reset_peak_memory_stats(dev)
        out = run()
        torch.cuda.synchronize(dev)
        peak = torch.cuda.max_memory_allocated(dev) - base
        del out
        times = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = tf32
    eager_ms = statistics.median(times)
    ours_bytes = w.B * w.H * w.N * (w.d * (2 if w.dtype == "bf16" else 4) + 4) + our_extra
    return {"kind": "context: PyTorch eager fp32 on this GPU (the pages' baseline)",
            "ms": eager_ms, "speedup_of_ours": eager_ms / our_ms,
            "eager_peak_bytes_beyond_inputs": peak,
            "ours_bytes_beyond_inputs": ours_bytes,
            "memory_reduction": 1.0 - ours_bytes / peak if peak > 0 else None}


def run_ours(args, w):
    from attention_attn_fwd_05_gb300 import attn_fwd, attn_fwd_host, device_status
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    q, k, v = make_workload_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    od = torch.empty_like(qd)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = w.io_bytes <= 2 * L2_BYTES
    scratch = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev) if flush \
        else None

    def step():
        attn_fwd(qd, kd, vd, w.scale, w.causal, out=od, lse=lse, stream=stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    if device_status(device=dev) != 0:
        raise RuntimeError("device status reports a timeout during warm-up")
    # Device memory the call itself takes (driver view, so any allocation inside
    # the library would show), beside what materialising the scores would take.
    free0 = torch.cuda.mem_get_info(dev)[0]
    step()
    torch.cuda.synchronize(dev)
    extra = max(0, free0 - torch.cuda.mem_get_info(dev)[0])
    scores = w.B * w.H * w.N * w.N * 4
    memory = {"extra_device_bytes_per_call": extra, "io_bytes": w.io_bytes,
              "scores_fp32_bytes": scores,
              "eager_peak_bytes": w.io_bytes + 2 * scores,
              "reduction_vs_eager": 1.0 - (w.io_bytes + extra) / (w.io_bytes + 2 * scores),
              "eager_model": "inputs, outputs, S and P materialised in fp32"}

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        clk.mark_start()
        t_begin.record(stream)
        for i in range(args.steps):
            if flush:
                scratch.fill_(float(i))
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
    if world > 1:
        torch.distributed.barrier()
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    region_ms = t_begin.elapsed_time(t_end)
    step_ms = sum(kernel_ms) / len(kernel_ms) if flush else region_ms / args.steps
    if device_status(device=dev) != 0:
        raise RuntimeError("device status reports a timeout during the timed region")

    # End to end through the public host-memory call: H2D of Q, K, V from pinned
    # memory, the kernel, D2H of O and LSE, every step.
    # Two steps in flight: step i runs on stream i % 2 with its own workspace
    # and host outputs, and its result is waited for before step i + 2 reuses
    # them, so step i + 1's copy in overlaps step i's forward and copy out.
    # Every step still copies its inputs in and its result out.
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    e2e_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    e2e_bufs = [{}, {}]
    for i in range(4):
        attn_fwd_host(qh, kh, vh, w.scale, w.causal, device=dev, stream=e2e_streams[i % 2],
                      buffers=e2e_bufs[i % 2])
    # Three rounds of e2e_steps steps each; the median round is reported, so a
    # single host-side stall (another tenant, a page fault) in a window of a
    # few tens of milliseconds does not stand for the whole run.
    e2e_steps = max(4, min(args.steps, 10))
    rounds = []
    for _ in range(3):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            if i >= 2:
                e2e_streams[i % 2].synchronize()  # step i - 2's result is on the host
            attn_fwd_host(qh, kh, vh, w.scale, w.causal, device=dev, stream=e2e_streams[i % 2],
                          buffers=e2e_bufs[i % 2], wait=False)
        for st_ in e2e_streams:
            st_.synchronize()
        rounds.append((time.perf_counter() - t0) / e2e_steps)
    e2e_s = statistics.median(rounds)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = od.numel() * od.element_size() + lse.numel() * 4

    step_ms, e2e_ms = max_over_ranks([step_ms, e2e_s * 1e3], device=dev)
    if rank != 0:
        return
    tflops = whole_job_rate(w.flops, world, step_ms * 1e-3) / 1e12
    e2e_tflops = whole_job_rate(w.flops, world, e2e_ms * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    sustained = region_ms > 1000.0
    if w.dtype == "bf16":
        peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        kernel_tflops = w.flops / (statistics.mean(kernel_ms) * 1e-3) / 1e12
        kernels = kernels_per_call(w, torch.cuda.get_device_properties(dev).multi_processor_count)
        # The traffic and tensor-pipe figures are those of the first (dominant)
        # kernel's committed capture.
        traffic = profiled_traffic("bf16", w.name, kernels[0])
        roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak,
                    "unit": "TFLOP/s", "frac": kernel_tflops / peak, "traffic": traffic,
                    "kernel": " + ".join(kernels),
                    "peak_source": f"{peak_src} {'sustained' if sustained else 'burst'} "
                                   "bf16 dense (MEASURED_PEAKS.json)",
                    "algorithmic_flops_per_launch": w.flops,
                    # The tensor pipe's own nominal dense rate (2.25 PFLOP/s bf16)
                    # and the ncu tensor-pipe activity of the committed capture.
                    "frac_of_nominal_dense": kernel_tflops / NOMINAL_BF16_DENSE_TFLOPS,
                    "ncu_tensor_pipe_active_pct": profiled_value(
                        "bf16", w.name, "tensor_pipe_active_pct", kernels[0])}
    else:
        kernel_tflops = w.flops / (statistics.mean(kernel_ms) * 1e-3) / 1e12
        # fp32 FMA pipe: 152 SMs x 128 lanes x 2 FLOP x max SM clock.
        alu_peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        roofline = {"bound": "alu", "achieved": kernel_tflops, "peak": alu_peak,
                    "unit": "TFLOP/s", "frac": kernel_tflops / alu_peak,
                    "traffic": profiled_traffic("f32", w.name), "kernel": KERNEL_NAME["f32"],
                    "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock",
                    "algorithmic_flops_per_launch": w.flops}
    roofline["algorithmic_bytes_per_launch"] = w.io_bytes
    roofline["hbm_gbs_algorithmic"] = w.io_bytes / (statistics.mean(kernel_ms) * 1e-3) / 1e9

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        tf, cores, n, dt = time_oracle(w, q, k, v, args.cpu_budget)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} query rows of {w.name} spread over all positions "
                         f"(row_flops = 4*d*visible keys), {dt:.1f} s"}

    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic", "config": config_of(w),
        "pct_of_bf16_peak": 100.0 * tflops / world / roofline["peak"]
        if w.dtype == "bf16" else None,
        "pct_of_nominal_bf16_dense": 100.0 * tflops / world / NOMINAL_BF16_DENSE_TFLOPS
        if w.dtype == "bf16" else None,
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": e2e_tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "rounds_ms_per_step": [r * 1e3 for r in rounds],
                "pipeline": "attn_fwd_host, two steps in flight on two streams; median of "
                            "3 rounds of %d steps" % e2e_steps},
        "gpu_launches": args.steps * launches_per_call(
            w, torch.cuda.get_device_properties(dev).multi_processor_count),
        "clocks": clk.summary(),
        "memory": memory,
        "gpu": torch.cuda.get_device_name(dev),
    }
    if args.context_eager:
        line["context_eager"] = eager_context(w, qd, kd, vd, step_ms, extra, dev)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_memop(args):
    """Bench one of the HBM-bound kernels: GB/s against the measured copy bandwidth."""
    from attention_attn_fwd_05_gb300 import add_rmsnorm, device_status, row_softmax
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    t = torch.float32 if args.dtype == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(7)
    rows, width = args.rows, args.width
    x = torch.randn(rows, width, generator=g).to(t).to(dev)
    if args.op == "row_softmax":
        if t != torch.float32:
            raise SystemExit("row_softmax is fp32")
        y = torch.empty_like(x)
        lse = None

        def step():
            row_softmax(x, out=y)
        nbytes = 2 * x.numel() * 4  # read x once, write y once
        # Aligned rows up to 12288 floats take the streamed kernel.
        kname = "row_softmax_stream_kernel" if width % 4 == 0 and width <= 12288 \
            else "row_softmax_kernel"
    else:
        r = torch.randn(rows, width, generator=g).to(t).to(dev)
        w = torch.randn(width, generator=g).to(t).to(dev)
        out, ho = torch.empty_like(x), torch.empty_like(x)

        def step():
            add_rmsnorm(x, w, r, 1e-6, out=out, res_out=ho)
        nbytes = 4 * x.numel() * x.element_size() + w.numel() * w.element_size()
        # bf16 rows of up to 8192 elements (a multiple of 8) take the streamed kernel.
        kname = "add_rmsnorm_stream_kernel" if (t == torch.bfloat16 and width % 8 == 0
                                                and width <= 8192) else "add_rmsnorm_kernel"
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index or 0) as clk:
        clk.mark_start()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        clk.mark_end()
    if device_status(device=dev) != 0:
        raise RuntimeError("device status reports a timeout")
    ms = e0.elapsed_time(e1) / args.steps
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, src = load_peaks()
    line = {"metric": f"{args.op} GB/s (algorithmic bytes)", "value": gbs, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.dtype,
            "data": "synthetic",
            "config": {"workload": f"{args.op}_{args.dtype}_rows{rows}_width{width}",
                       "rows": rows, "width": width,
                       "l2": "inputs and outputs larger than L2, no flush"
                       if nbytes > 2 * L2_BYTES else "smaller than L2: L2-resident"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": None, "kernel": kname,
                         "peak_source": f"{src} copy bandwidth (MEASURED_PEAKS.json)",
                         "algorithmic_bytes_per_launch": nbytes},
            "gpu_launches": args.steps, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_bwd(args, w):
    """Bench the backward: TFLOP/s with FLOP = 10*B*H*N^2*d (the five N x N x d
    products of the backward; halved with the causal mask).  bf16 runs on the
    tensor-core kernels (which recompute S and dP for dQ: 14*B*H*N^2*d of MMA
    work) and is reported against the bf16 peak; fp32 runs on CUDA cores and
    is reported against the fp32 FMA-pipe peak."""
    from attention_attn_fwd_05_gb300 import attn_bwd, attn_fwd, device_status
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in make_workload_inputs(w))
    o, lse = attn_fwd(q, k, v, w.scale, w.causal)
    g = torch.randn(q.shape, generator=torch.Generator().manual_seed(9)).to(q.dtype).to(dev)

    def step():
        attn_bwd(q, k, v, o, lse, g, w.scale, w.causal)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        clk.mark_start()
        e0.record()
        for _ in range(args.steps):
            step()
        e1.record()
        torch.cuda.synchronize(dev)
        clk.mark_end()
    if device_status(device=dev) != 0:
        raise RuntimeError("device status reports a timeout")
    ms = e0.elapsed_time(e1) / args.steps
    flops = 10.0 * w.B * w.H * w.N * w.N * w.d / (2 if w.causal else 1)
    tf = flops / (ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    if w.dtype == "bf16":
        peak = peaks["bf16_tflops_sustained" if ms * args.steps > 1000.0 else "bf16_tflops"]
        roofline = {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                    "frac": tf / peak, "traffic": None,
                    "kernel": "bwd_dkdv_tc_kernel + bwd_dq_tc_kernel",
                    "mma_flops_per_launch": flops * 1.4,
                    "peak_source": f"{peak_src} bf16 dense (MEASURED_PEAKS.json)"}
    else:
        alu_peak = 152 * 128 * 2 * peaks.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        roofline = {"bound": "alu", "achieved": tf, "peak": alu_peak, "unit": "TFLOP/s",
                    "frac": tf / alu_peak, "traffic": None,
                    "kernel": "bwd_dkdv_kernel + bwd_dq_kernel",
                    "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock"}
    print(json.dumps({
        "metric": "attention backward TFLOP/s (10*B*H*N^2*d, causal halved)", "value": tf,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic", "config": config_of(w), "roofline": roofline,
        "gpu_launches": 3 * args.steps, "clocks": clk.summary()}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline leg")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--context-eager", action="store_true",
                    help="also time PyTorch eager fp32 attention on the GPU (context only)")
    ap.add_argument("--op", default="attn",
                    choices=["attn", "attn_bwd", "row_softmax", "add_rmsnorm"],
                    help="attn (the hot path, default) or one of the HBM-bound kernels")
    ap.add_argument("--rows", type=int, default=16384)
    ap.add_argument("--width", type=int, default=8192)
    ap.add_argument("--dtype", default="bf16", choices=["f32", "bf16"])
    args = ap.parse_args(argv)
    if args.op == "attn_bwd":
        run_bwd(args, WORKLOADS[args.workload])
        return
    if args.op != "attn":
        run_memop(args)
        return
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
