"""Benchmark: fused softmax cross-entropy forward+backward (gradient written
over the logits) on one GB300, through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workload NAME]

One step is one pass of the whole hot path over one batch: the online
max/log-sum-exp forward, the target gather, the deterministic mean and the
in-place gradient, i.e. one ce_fwd_bwd_inplace call on a fresh synthetic
[M, V] logits matrix already resident in HBM.  Every timed step works on its
own copy of the input (each larger than the 129 MB L2), so no step starts
with a warm L2.  Prints ONE JSON line (rank 0).

--impl reference times the float64 CPU oracle on the host cores on a bounded
sample of the same workload (the slow, obviously correct baseline).
Under torchrun (N > 1) each rank runs its own replica of the workload on its
own GPU (weak scaling); the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from softmax_cross_entropy_online_gb300 import synthetic  # noqa: E402

METRIC = "CE fwd+bwd GB/s and % of GB300 HBM roofline (ms per call) at 1 GPU"
FALLBACK_HBM_GBS = 6800.0

# DRAM traffic per launch of each workload's default kernel, from one
# `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum` capture (a reduced
# row count, scaled to the full launch by the rows processed), keyed by the
# digest of the row-kernel sources the counters were taken on: any change to
# those sources nulls every record until it is captured again.
NCU_TRAFFIC: dict[str, dict[str, int]] = {
    # full-size captures, one launch each (dram__bytes_read.sum + dram__bytes_write.sum)
    "d87fca6c7ad3c81b4d3691c53b03664c8905388105be045da367c706607f86ef": {
        "f32_32768x4096": 537223168 + 475344640,
        "f16_8192x131072_spiked": 2170441728 + 2066544640,
        "bf16_16384x50257": 1647281152 + 1585064704,
    },
}


def algorithmic_bytes(M: int, V: int, es: int, bwd: bool) -> int:
    """Bytes the method must move: one read of the logits (+ one write of the
    gradient), the int64 targets, and the fp32 row_loss and lse outputs."""
    x = M * V * es
    return x * (2 if bwd else 1) + M * 8 + M * 4 * 2 + 4


# The sources that decide which row kernel runs and what it does; the
# tensor-core entry points (ce_api_tc.cu) and kernels do not enter the record.
ROW_KERNEL_SOURCES = ("ce_rows.cuh", "ce_stream.cuh", "ce_launch.cuh", "ce_rows_f32.cu",
                      "ce_rows_f16.cu", "ce_rows_bf16.cu", "ce_api.cu", "ce_host.cuh")


def csrc_digest() -> str:
    d = os.path.join(ROOT, "softmax_cross_entropy_online_gb300", "csrc")
    h = hashlib.sha256()
    for f in ROW_KERNEL_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        if d.get("hbm_gbs"):
            return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def mark(self) -> int:
        """Index of the next sample (to delimit a window of samples)."""
        return len(self.lines)

    @staticmethod
    def summarize(lines) -> dict:
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_median": statistics.median(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}

    def window(self, i0: int, i1: int) -> dict:
        """Summary of the samples taken between two marks."""
        return self.summarize(list(self.lines[i0:i1]))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        return self.summarize(self.lines)


def max_over_ranks(x: float, device) -> float:
    """The slowest rank's value of x (the step time of a replica run): an
    all-reduce of one scalar, on `device` (CUDA under NCCL, CPU under gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world_size: int, bytes_per_step: int, ms_per_step: float) -> float:
    """Whole-job throughput of N replicas: every rank moves bytes_per_step per
    step and the step takes the slowest rank's ms_per_step."""
    return world_size * bytes_per_step / (ms_per_step * 1e-3) / 1e9


def rate_figures(ws: int, M: int, ms_per_step: float, kernel_ms: float, bytes_per_step: int,
                 peak_gbs: float) -> dict:
    """Absolute figures beside the GB/s: microseconds per call, rows per second
    for the whole job, and whether the call is so small that its bytes at the
    peak rate take less than a few microseconds, so launch latency bounds it
    and its roofline fraction says little."""
    return {"us_per_call": kernel_ms * 1e3,
            "rows_per_s": ws * M / (ms_per_step * 1e-3),
            "latency_bound": bytes_per_step / (peak_gbs * 1e9) < 4e-6}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    es = synthetic.ELEM_BYTES[w.dtype]
    sample_rows = max(16, min(w.M, args.ref_rows))
    x = synthetic.make_logits(sample_rows, w.V, w.dtype, w.sigma, w.spike_prob, w.spike_value,
                              w.seed)
    t = synthetic.make_targets(sample_rows, w.V, w.seed)
    x64 = oracle.to_f64(x, w.dtype)
    for _ in range(args.warmup):
        oracle.ce_fwd_bwd(x64[:16], t[:16], "mean")
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.ce_fwd_bwd(oracle.to_f64(x, w.dtype), t, "mean")
        times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    b = algorithmic_bytes(sample_rows, w.V, es, True)
    gbs = b / step_s / 1e9
    sample = f"{sample_rows} of {w.M} rows of {w.name} per step (float64 numpy, 1 thread)"
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(w), "M": w.M, "V": w.V, "sample_rows": sample_rows},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", **host_info(),
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def host_info() -> dict:
    """The host the oracle ran on: its CPU count and model (recorded beside the
    single-thread figure)."""
    model = platform.processor() or platform.machine()
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"host_cpus": os.cpu_count(), "host_cpu": model, "host_arch": platform.machine()}


def workload_desc(w):
    return f"{w.name}: {w.desc}"


def _oracle_rows(job):
    """One host process's share of the all-cores oracle timing: forward and
    backward in float64 over its block of rows."""
    import oracle
    x, t, dtype = job
    oracle.ce_fwd_bwd(oracle.to_f64(x, dtype), t, "mean")
    return len(t)


def oracle_all_cores(x, t, dtype, M: int, V: int, es: int, name: str) -> dict | None:
    """The same sample timed on every host core: the rows split into one
    contiguous block per process (a spawn pool, so it is safe after CUDA has
    started), the timed region including the hand-off of each block."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    rows = len(t)
    if n < 2 or rows < n:
        return None
    blocks = np.array_split(np.arange(rows), n)
    jobs = [(x[b[0]:b[-1] + 1], t[b[0]:b[-1] + 1], dtype) for b in blocks]
    with mp.get_context("spawn").Pool(n) as pool:
        pool.map(_oracle_rows, [(x[:2], t[:2], dtype)] * n, chunksize=1)  # imports done
        t0 = time.perf_counter()
        done = sum(pool.map(_oracle_rows, jobs, chunksize=1))
        dt = time.perf_counter() - t0
    assert done == rows
    return {"value": algorithmic_bytes(rows, V, es, True) / dt / 1e9, "unit": "GB/s",
            "cores": n, "sample": f"the same {rows} of {M} rows of {name} in {n} processes "
                                  f"({dt:.2f} s)"}


def cpu_baseline(w, budget_s: float):
    """Time the oracle (as it stands) on a bounded sample of the workload: on one
    host thread (the reported value), and the same sample on every host core."""
    import oracle
    es = synthetic.ELEM_BYTES[w.dtype]
    probe = max(8, min(w.M, (1 << 22) // w.V))
    x = synthetic.make_logits(probe, w.V, w.dtype, w.sigma, w.spike_prob, w.spike_value, w.seed)
    t = synthetic.make_targets(probe, w.V, w.seed)
    t0 = time.perf_counter()
    oracle.ce_fwd_bwd(oracle.to_f64(x, w.dtype), t, "mean")
    dt = time.perf_counter() - t0
    rows = int(min(w.M, max(probe, probe * budget_s / max(dt, 1e-6))))
    x = synthetic.make_logits(rows, w.V, w.dtype, w.sigma, w.spike_prob, w.spike_value, w.seed)
    t = synthetic.make_targets(rows, w.V, w.seed)
    t0 = time.perf_counter()
    oracle.ce_fwd_bwd(oracle.to_f64(x, w.dtype), t, "mean")
    dt = time.perf_counter() - t0
    gbs = algorithmic_bytes(rows, w.V, es, True) / dt / 1e9
    out = {"value": gbs, "unit": "GB/s", "cores": 1, "kind": "oracle", **host_info(),
           "sample": f"{rows} of {w.M} rows of {w.name}, fwd+bwd in float64 numpy "
                     f"({dt:.1f} s on 1 host thread)"}
    try:
        allc = oracle_all_cores(x, t, w.dtype, w.M, w.V, es, w.name)
    except Exception as e:  # the extra leg never costs the line its one-thread value
        allc = {"error": f"{type(e).__name__}: {e}"[:200]}
    if allc is not None:
        out["all_cores"] = allc
    return out


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------
def flush_l2(scratch) -> None:
    """Write a buffer larger than the L2 (129 MB), so no input starts warm."""
    scratch.fill_(1)


def time_per_call(fn, bufs, pristine, flush, reps: int = 3, warmup: int = 3, refresh=True):
    """Device time of one call (ms): the calls run back to back, one per
    distinct buffer, bracketed by CUDA events on the launch stream; before each
    rep the buffers get fresh inputs and the L2 is flushed (both untimed).
    Returns the median over reps and the per-rep times."""
    import torch
    for i in range(warmup):
        fn(bufs[i % len(bufs)])
    times = []
    for _ in range(reps):
        if refresh:
            for b in bufs:
                b.copy_(pristine)
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for b in bufs:
            fn(b)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / len(bufs))
    return statistics.median(times), times


def traffic_record(workload: str):
    """ncu DRAM bytes per launch of a workload's default kernel, when the row-kernel
    sources are the ones the counters were taken on; else None."""
    rec = NCU_TRAFFIC.get(csrc_digest(), {})
    return rec.get(workload)


def workload_tensors(w, dev):
    import torch
    x_np = synthetic.make_logits(w.M, w.V, w.dtype, w.sigma, w.spike_prob, w.spike_value, w.seed)
    t_np = synthetic.make_targets(w.M, w.V, w.seed)
    if w.dtype == "bf16":
        host = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16)
    else:
        host = torch.from_numpy(x_np)
    return host, torch.from_numpy(t_np)


def sub_record(L, api, w, dev, sh, flush, peak, bwd: bool, n_bufs: int):
    """One more workload timed beside the headline one: ms per call of the
    default kernel (fused fwd+bwd in place, or the forward), GB/s of the
    algorithmic bytes, the roofline fraction, rows/s, and ncu traffic."""
    import torch
    host, t_host = workload_tensors(w, dev)
    pristine = host.to(dev)
    targets = t_host.to(dev)
    del host
    M, V = w.M, w.V
    es = synthetic.ELEM_BYTES[w.dtype]
    code = {"f32": 0, "f16": 1, "bf16": 2}[w.dtype]
    bufs = [pristine.clone() for _ in range(n_bufs)]
    loss = torch.empty((), dtype=torch.float32, device=dev)
    rl = torch.empty(M, dtype=torch.float32, device=dev)
    lse = torch.empty(M, dtype=torch.float32, device=dev)
    entry = L.ce_fwd_bwd_inplace if bwd else L.ce_forward

    def fn(b):
        st = entry(b.data_ptr(), targets.data_ptr(), M, V, code, 0, loss.data_ptr(),
                   rl.data_ptr(), lse.data_ptr(), sh)
        if st != 0:
            raise api.CEError(st, entry.__name__)

    ms, reps = time_per_call(fn, bufs, pristine, flush, refresh=bwd)
    assert api.ce_check_errors() == 0
    nbytes = algorithmic_bytes(M, V, es, bwd)
    graph_us = None
    if nbytes / (peak * 1e9) < 4e-6 and not bwd:
        # launch-bound: Python launches one call every few microseconds, so the
        # device time per call shows only when the same calls replay from a CUDA
        # graph (captured on a side stream after warm-up calls there)
        gs = torch.cuda.Stream(dev)
        gh = gs.cuda_stream

        def gfn(b):
            st = entry(b.data_ptr(), targets.data_ptr(), M, V, code, 0, loss.data_ptr(),
                       rl.data_ptr(), lse.data_ptr(), gh)
            if st != 0:
                raise api.CEError(st, entry.__name__)

        with torch.cuda.stream(gs):
            for b in bufs[:3]:
                gfn(b)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for b in bufs:
                gfn(b)
        gtimes = []
        for _ in range(3):
            flush()
            torch.cuda.synchronize()
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record()
            graph.replay()
            g1.record()
            torch.cuda.synchronize()
            gtimes.append(g0.elapsed_time(g1) / len(bufs) * 1e3)
        graph_us = statistics.median(gtimes)
        assert api.ce_check_errors() == 0
    gbs = nbytes / (ms * 1e-3) / 1e9
    out = {"workload": workload_desc(w), "call": ("ce_fwd_bwd_inplace (mean)" if bwd
                                                  else "ce_forward (mean, row loss, lse)"),
           "M": M, "V": V, "dtype": w.dtype, "ms_per_call": ms, "us_per_call": ms * 1e3,
           "gb_s": gbs, "rows_per_s": M / (ms * 1e-3),
           "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                        "frac": gbs / peak, "bytes_per_launch": nbytes,
                        "traffic": traffic_record(w.name)},
           "latency_bound": nbytes / (peak * 1e9) < 4e-6,
           "graph_us_per_call": graph_us,
           "timing": f"{len(bufs)} distinct buffers back to back, L2 flushed, median of "
                     f"{len(reps)} reps"}
    del bufs, pristine
    torch.cuda.empty_cache()
    return out


def e2e_pipelined(L, api, host, t_host, dbufs, loss, row_loss, lse, M: int, V: int, code: int,
                  stream, steps: int):
    """Milliseconds per step of the end-to-end leg: every step copies its logits
    and targets from pinned host memory, calls ce_fwd_bwd_inplace, and copies the
    gradient and the loss back to pinned host memory.  Pipelined: device buffers
    alternate and the copies run on two copy streams, so one step's input copy
    overlaps the previous step's output copy.  Also returns the same steps run one
    after another on one stream, for reference."""
    import torch
    dev = dbufs[0].device
    sh = stream.cuda_stream
    nb = len(dbufs)
    tgts = [torch.empty_like(t_host, device=dev) for _ in range(nb)]
    # each buffer's own loss, so a later step's call never overwrites a loss whose
    # copy to the host is still queued
    dloss = [torch.empty((), dtype=torch.float32, device=dev) for _ in range(nb)]
    outs = [torch.empty_like(host).pin_memory() for _ in range(nb)]
    losses = [torch.empty((), dtype=torch.float32).pin_memory() for _ in range(nb)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(nb)]
    ev_done = [torch.cuda.Event() for _ in range(nb)]
    ev_free = [torch.cuda.Event() for _ in range(nb)]

    def call(buf, tg, ls):
        st = L.ce_fwd_bwd_inplace(buf.data_ptr(), tg.data_ptr(), M, V, code, 0, ls.data_ptr(),
                                  row_loss.data_ptr(), lse.data_ptr(), sh)
        if st != 0:
            raise api.CEError(st, "ce_fwd_bwd_inplace")

    def run(n):
        for i in range(n):
            b = i % nb
            with torch.cuda.stream(s_in):
                if i >= nb:
                    s_in.wait_event(ev_free[b])  # the buffer's previous gradient is out
                dbufs[b].copy_(host, non_blocking=True)
                tgts[b].copy_(t_host, non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            call(dbufs[b], tgts[b], dloss[b])
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                outs[b].copy_(dbufs[b], non_blocking=True)
                losses[b].copy_(dloss[b], non_blocking=True)
                ev_free[b].record(s_out)

    run(2)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    run(steps)
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize()
    piped = e0.elapsed_time(e1) / steps
    # the same steps one after another on the launch stream
    e0.record(stream)
    for i in range(steps):
        dbufs[0].copy_(host, non_blocking=True)
        tgts[0].copy_(t_host, non_blocking=True)
        call(dbufs[0], tgts[0], dloss[0])
        outs[0].copy_(dbufs[0], non_blocking=True)
        losses[0].copy_(dloss[0], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    return piped, e0.elapsed_time(e1) / steps


# The workloads timed beside the headline one in the default run: (name, fused
# fwd+bwd?, distinct buffers).  The small fp32 case is forward only and bound
# by launch latency; its 300 buffers (> L2) keep every call cold.
SIDE_WORKLOADS = (("small_f32_256x1024", False, 300), ("f16_8192x131072_spiked", True, 6),
                  ("bf16_16384x50257", True, 6))


def run_native(args, w):
    import torch
    import torch.distributed as dist

    from softmax_cross_entropy_online_gb300 import api, build

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    L = api.lib()

    M, V = w.M, w.V
    es = synthetic.ELEM_BYTES[w.dtype]
    code = {"f32": 0, "f16": 1, "bf16": 2}[w.dtype]

    host, t_cpu = workload_tensors(w, dev)
    host = host.pin_memory()
    t_host = t_cpu.pin_memory()
    pristine = host.to(dev)
    targets = t_host.to(dev)
    step_bytes = M * V * es
    n_bufs = args.steps + args.warmup
    if n_bufs * step_bytes > args.max_resident_gb * 1e9:
        n_bufs = max(2, int(args.max_resident_gb * 1e9 // step_bytes))
    bufs = [pristine.clone() for _ in range(n_bufs)]
    loss = torch.empty((), dtype=torch.float32, device=dev)
    row_loss = torch.empty(M, dtype=torch.float32, device=dev)
    lse = torch.empty(M, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    l2_scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def flush():
        flush_l2(l2_scratch)

    def step(buf):
        st = L.ce_fwd_bwd_inplace(buf.data_ptr(), targets.data_ptr(), M, V, code, 0,
                                  loss.data_ptr(), row_loss.data_ptr(), lse.data_ptr(), sh)
        if st != 0:
            raise api.CEError(st, "ce_fwd_bwd_inplace")

    # the clock sampler starts first, so the timed region follows the warm-up and
    # the buffer refresh directly, with no idle gap in which the clocks could drop
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    for i in range(args.warmup):
        step(bufs[(args.steps + i) % n_bufs])
    # refresh every timed buffer with the pristine logits (untimed)
    for b in bufs:
        b.copy_(pristine)
    flush()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()

    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    launches0 = api.ce_launch_count()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    # the K calls back to back between two events on the launch stream (an event
    # between calls would make each call wait for the previous one to drain)
    region0.record(stream)
    for i in range(args.steps):
        step(bufs[i % n_bufs])
    region1.record(stream)
    torch.cuda.synchronize()
    launches = api.ce_launch_count() - launches0
    # a sustained window of the same call over the resident buffers (their contents
    # are by now earlier calls' gradients: the same work per call), long enough for
    # the clock sampler to see it; outside the events that time `value`
    sustained = None
    if rank == 0 and args.sustained_s > 0:
        avg = region0.elapsed_time(region1) / args.steps
        n_sus = max(1, int(args.sustained_s / (avg * 1e-3)))
        mark0 = sampler.mark()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(n_sus):
            step(bufs[i % n_bufs])
        s1.record(stream)
        torch.cuda.synchronize()
        mark1 = sampler.mark()
        sus_ms = s0.elapsed_time(s1) / n_sus
        sustained = {"calls": n_sus, "seconds": s0.elapsed_time(s1) * 1e-3,
                     "ms_per_call": sus_ms,
                     "gb_s": algorithmic_bytes(M, V, es, True) / (sus_ms * 1e-3) / 1e9,
                     "clocks": sampler.window(mark0, mark1)}
    clocks = sampler.stop() if sampler else None
    if clocks is not None and sustained is not None and sustained["clocks"]["samples"]:
        # the clocks under load: the samples of the sustained window, with the
        # whole run's count and reasons beside them
        whole = clocks
        clocks = dict(sustained["clocks"])
        clocks["window"] = "the sustained window of back-to-back calls"
        clocks["samples_whole_run"] = whole["samples"]
        clocks["reasons"] = sorted(set(clocks["reasons"]) | set(whole["reasons"]))
    region_ms = region0.elapsed_time(region1)
    local_kernel_ms = region_ms / args.steps  # this rank's mean time per launch
    region_ms = max_over_ranks(region_ms, dev)
    assert api.ce_check_errors() == 0

    ms_per_step = region_ms / args.steps
    b_step = algorithmic_bytes(M, V, es, True)
    value = aggregate_gbs(ws, b_step, ms_per_step)
    avg_kernel_ms = local_kernel_ms
    peak, peak_kind = measured_peaks()
    achieved = b_step / (avg_kernel_ms * 1e-3) / 1e9
    traffic = traffic_record(w.name)
    if sustained is not None:
        sustained["frac"] = sustained["gb_s"] / peak

    # forward-only pass on the same workload (the first half of the config)
    fwd_ms = sm_ms = probe = None
    if rank == 0:
        nf = min(args.steps, n_bufs)
        fbufs = bufs[:nf]
        fwd_ms, _ = time_per_call(
            lambda b: L.ce_forward(b.data_ptr(), targets.data_ptr(), M, V, code, 0,
                                   loss.data_ptr(), row_loss.data_ptr(), lse.data_ptr(), sh),
            fbufs, pristine, flush, reps=3)
        # the fused softmax (probabilities written over the logits, one read and
        # one write per element) on the same buffers
        sm_ms, _ = time_per_call(
            lambda b: L.ce_softmax_forward(b.data_ptr(), b.data_ptr(), M, V, code, None, sh),
            fbufs, pristine, flush, reps=3)
        assert api.ce_check_errors() == 0
        # stream probes over the same buffers with PyTorch's own kernels (not the
        # library's): an in-place read + write pass (x *= 1) and a read-only pass
        # (the max), the achievable ceilings beside the fused pass
        probe = {}
        for name, fn, nbytes in (("inplace_rw", lambda b: b.mul_(1), 2 * M * V * es),
                                 ("read_only", lambda b: torch.amax(b), M * V * es)):
            pms, _ = time_per_call(fn, fbufs, pristine, flush, reps=3)
            probe[name] = {"ms": pms, "gb_s": nbytes / (pms * 1e-3) / 1e9,
                           "frac": nbytes / (pms * 1e-3) / 1e9 / peak}

    # end to end through the public call: host logits and targets -> device, the
    # call, then the call's outputs -> host: the gradient it wrote over the
    # logits and the loss, every step.  Two device buffers alternate between
    # steps, and the copies run on their own streams, so step i + 1's input copy
    # overlaps step i's output copy (the two directions of the host link run at
    # once, as a training loop prefetching its next batch would).
    e2e_ms, e2e_serial_ms = e2e_pipelined(L, api, host, t_host, bufs[:2], loss, row_loss, lse,
                                          M, V, code, stream, max(3, min(args.steps, 10)))
    e2e_ms = max_over_ranks(e2e_ms, dev)
    e2e_value = aggregate_gbs(ws, b_step, e2e_ms)

    side = None
    if rank == 0 and not args.no_side_workloads and args.rows is None:
        del bufs
        torch.cuda.empty_cache()
        side = {}
        for name, bwd, nb in SIDE_WORKLOADS:
            if name == w.name:
                continue
            side[name] = sub_record(L, api, synthetic.WORKLOADS[name], dev, sh, flush, peak,
                                    bwd, nb)
        if not args.no_linear_side:
            side["linear_ce_8192x4096x128256"] = linear_side_record(L, api, dev, sh, "lean")
            side["linear_ce_8192x4096x128256_fused"] = linear_side_record(L, api, dev, sh,
                                                                          "fused")

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": workload_desc(w), "M": M, "V": V,
                       "call": "ce_fwd_bwd_inplace (mean)",
                       "l2": f"inputs larger than L2: a distinct {step_bytes / 2**20:.0f} MiB "
                             f"logits buffer per step ({n_bufs} resident buffers)",
                       "parallelism": f"replicas x{ws}"},
            "pct_of_hbm_roofline": 100.0 * achieved / peak,
            "ms_per_call": avg_kernel_ms,
            "rates": rate_figures(ws, M, ms_per_step, avg_kernel_ms, b_step, peak),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": traffic,
                         "bytes_per_launch": b_step},
            "forward_only": None if fwd_ms is None else {
                "ms_per_call": fwd_ms,
                "gb_s": algorithmic_bytes(M, V, es, False) / (fwd_ms * 1e-3) / 1e9,
                "frac": algorithmic_bytes(M, V, es, False) / (fwd_ms * 1e-3) / 1e9 / peak},
            "stream_probes": probe,
            "softmax": None if sm_ms is None else {
                "call": "ce_softmax_forward (in place)", "ms_per_call": sm_ms,
                "gb_s": 2 * M * V * es / (sm_ms * 1e-3) / 1e9,
                "frac": 2 * M * V * es / (sm_ms * 1e-3) / 1e9 / peak},
            "e2e": {"value": e2e_value, "unit": "GB/s",
                    "h2d_bytes_per_step": step_bytes + M * 8,
                    "d2h_bytes_per_step": step_bytes + 4,
                    "ms_per_step": e2e_ms,
                    "serial_ms_per_step": e2e_serial_ms,
                    "what": "pinned host logits + targets -> device, ce_fwd_bwd_inplace, "
                            "the gradient (written over the logits) + loss -> pinned host, "
                            "every step; two device buffers in turn, copies on their own "
                            "streams (step i + 1's input copy beside step i's output copy)"},
            "gpu_launches": launches,
            "clocks": clocks,
            "sustained": sustained,
            "side_workloads": side,
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, args.cpu_budget_s)
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# fused linear + cross-entropy (bf16 h [8192, 4096], W [128256, 4096])
# ---------------------------------------------------------------------------
LINEAR_SHAPES = {"linear_ce_8192x4096x128256": (8192, 4096, 128256)}


def measured_tflops(burst: bool = False):
    """bf16 tensor peak: the sustained figure for a kernel timed inside a long
    step, the burst figure for one timed alone."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops" if burst else "bf16_tflops_sustained"
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        if d.get(key):
            return float(d[key]), f"measured ({'burst' if burst else 'sustained'})"
    return (1900.0, "fallback (burst)") if burst else (1700.0, "fallback (sustained)")


def linear_workspace_bytes(L, schedule: str, M: int, H: int, V: int) -> int:
    """The workspace that selects a schedule of linear_ce_fwd_bwd: "lean" (the
    default: no logits stored) or "fused" (fp32 logits chunks, G kept whole)."""
    fn = L.linear_ce_workspace_size if schedule == "lean" else L.linear_ce_workspace_size_fused
    return int(fn(M, H, V))


# the schedules' executed GEMM work per step in units of 2 M V H: the lean one
# computes the logits twice (statistics, then G), the fused one once
LINEAR_GEMMS = {"lean": 4, "fused": 3}


def linear_side_record(L, api, dev, sh, schedule: str, steps: int = 5, warmup: int = 3) -> dict:
    """The fused linear + cross-entropy step on its full workload (bf16 h
    [8192, 4096], W [128256, 4096]) in one schedule, timed beside the headline
    line: ms per step and TFLOP/s of the three GEMMs the loss and its gradients
    need (6 M H V; the lean schedule also recomputes the logits, its executed
    rate is given beside), against the sustained bf16 peak."""
    import torch
    M, H, V = LINEAR_SHAPES["linear_ce_8192x4096x128256"]
    h_np, W_np, t_np = synthetic.make_linear_ce_inputs(M, H, V, seed=0)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    h, W, t = as_bf16(h_np).to(dev), as_bf16(W_np).to(dev), torch.from_numpy(t_np).to(dev)
    del h_np, W_np
    wsb = linear_workspace_bytes(L, schedule, M, H, V)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    dH = torch.empty((M, H), dtype=torch.float32, device=dev)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)

    def step():
        st = L.linear_ce_fwd_bwd(h.data_ptr(), W.data_ptr(), t.data_ptr(), M, H, V,
                                 loss.data_ptr(), dH.data_ptr(), dW.data_ptr(),
                                 work.data_ptr(), wsb, sh)
        if st != 0:
            raise api.CEError(st, "linear_ce_fwd_bwd")

    for _ in range(warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    assert api.ce_check_errors() == 0
    ms = e0.elapsed_time(e1) / steps
    # the clocks under this step's load: about a second of back-to-back steps
    # after the timed ones (untimed), sampled by nvidia-smi, so the record
    # shows whether the tensor-bound step ran at a power-capped clock
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    i0 = sampler.mark()
    for _ in range(max(1, int(1200.0 / ms))):
        step()
    torch.cuda.synchronize()
    i1 = sampler.mark()
    sampler.stop()
    clocks = sampler.window(i0, i1)
    flops = 6.0 * M * V * H
    peak, kind = measured_tflops()
    tf = flops / (ms * 1e-3) / 1e12
    executed = LINEAR_GEMMS[schedule] * 2.0 * M * V * H / (ms * 1e-3) / 1e12
    out = {"workload": f"linear_ce_8192x4096x128256: bf16 h [{M}, {H}] N(0,1), W [{V}, {H}] "
                       "N(0, 0.02^2), int64 targets; loss, dH, dW (fp32)",
           "call": "linear_ce_fwd_bwd", "schedule": schedule,
           "logits_stored": schedule == "fused", "ms_per_step": ms, "tflop_s": tf,
           "executed_tflop_s": executed,
           "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                        "frac": tf / peak, "peak_source": kind,
                        "executed_frac": executed / peak},
           "loss": loss.item(), "steps": steps, "workspace_bytes": wsb,
           "clocks": dict(clocks, window="about 1.2 s of back-to-back steps after the timed ones")}
    del h, W, t, work, dH, dW
    torch.cuda.empty_cache()
    return out


def linear_e2e(L, api, host_in, dev_set, work, wsb: int, M: int, H: int, V: int, steps: int):
    """Milliseconds per step of the linear + CE end-to-end leg: every step copies
    h, W and the targets from pinned host memory, calls linear_ce_fwd_bwd, and
    copies the loss, dH and dW (the call's products) back to pinned host memory.
    Pipelined as a caller streaming batches would run it: two device buffer sets
    alternate, the input copies run on one copy stream and the output copies on
    another, so one step's input copies overlap the previous step's output
    copies.  Also returns the same steps run one after another on one stream."""
    import torch
    h_host, W_host, t_host = host_in
    h0, W0, t0, dH0, dW0, loss0 = dev_set
    dev = h0.device
    sets = [(h0, W0, t0, dH0, dW0, loss0),
            (torch.empty_like(h0), torch.empty_like(W0), torch.empty_like(t0),
             torch.empty_like(dH0), torch.empty_like(dW0), torch.empty_like(loss0))]
    dH_host = torch.empty(dH0.shape, dtype=dH0.dtype).pin_memory()
    dW_host = torch.empty(dW0.shape, dtype=dW0.dtype).pin_memory()
    loss_host = torch.empty((), dtype=torch.float32).pin_memory()
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in sets]
    ev_done = [torch.cuda.Event() for _ in sets]
    ev_free = [torch.cuda.Event() for _ in sets]

    def call(bs, stream):
        h, W, t, dH, dW, loss = bs
        st = L.linear_ce_fwd_bwd(h.data_ptr(), W.data_ptr(), t.data_ptr(), M, H, V,
                                 loss.data_ptr(), dH.data_ptr(), dW.data_ptr(),
                                 work.data_ptr(), wsb, stream.cuda_stream)
        if st != 0:
            raise api.CEError(st, "linear_ce_fwd_bwd")

    def pipelined(n):
        for i in range(n):
            b = i % 2
            h, W, t, dH, dW, loss = sets[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_free[b])  # the set's previous products are out
                h.copy_(h_host, non_blocking=True)
                W.copy_(W_host, non_blocking=True)
                t.copy_(t_host, non_blocking=True)
                ev_in[b].record(s_in)
            comp.wait_event(ev_in[b])
            call(sets[b], comp)
            ev_done[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                loss_host.copy_(loss, non_blocking=True)
                dH_host.copy_(dH, non_blocking=True)
                dW_host.copy_(dW, non_blocking=True)
                ev_free[b].record(s_out)
        comp.wait_stream(s_out)

    def serial(n):
        h, W, t, dH, dW, loss = sets[0]
        for _ in range(n):
            h.copy_(h_host, non_blocking=True)
            W.copy_(W_host, non_blocking=True)
            t.copy_(t_host, non_blocking=True)
            call(sets[0], comp)
            loss_host.copy_(loss, non_blocking=True)
            dH_host.copy_(dH, non_blocking=True)
            dW_host.copy_(dW, non_blocking=True)

    out = []
    for fn in (pipelined, serial):
        fn(1)  # warm: pinned pages, streams
        torch.cuda.synchronize()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(comp)
        fn(steps)
        x1.record(comp)
        torch.cuda.synchronize()
        out.append(x0.elapsed_time(x1) / steps)
    del sets[1]
    return out[0], out[1]


def run_linear(args):
    import torch
    from softmax_cross_entropy_online_gb300 import api, build

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    L = api.lib()
    M, H, V = LINEAR_SHAPES[args.workload]
    if args.rows is not None:
        M = args.rows
    if args.vocab is not None:
        V = args.vocab
    h_np, W_np, t_np = synthetic.make_linear_ce_inputs(M, H, V, seed=0)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    h_host, W_host = as_bf16(h_np).pin_memory(), as_bf16(W_np).pin_memory()
    t_host = torch.from_numpy(t_np).pin_memory()
    h, W, t = h_host.to(dev), W_host.to(dev), t_host.to(dev)
    wsb = linear_workspace_bytes(L, args.schedule, M, H, V)
    work = torch.empty(wsb, dtype=torch.uint8, device=dev)
    loss = torch.empty((), dtype=torch.float32, device=dev)
    dH = torch.empty((M, H), dtype=torch.float32, device=dev)
    dW = torch.empty((V, H), dtype=torch.float32, device=dev)
    sh = torch.cuda.current_stream(dev).cuda_stream

    def step():
        st = L.linear_ce_fwd_bwd(h.data_ptr(), W.data_ptr(), t.data_ptr(), M, H, V,
                                 loss.data_ptr(), dH.data_ptr(), dW.data_ptr(),
                                 work.data_ptr(), wsb, sh)
        if st != 0:
            raise api.CEError(st, "linear_ce_fwd_bwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = api.ce_launch_count()
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    launches = api.ce_launch_count() - n0
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    flops = 6.0 * M * V * H  # the logits, dH and dW GEMMs the step needs
    value = ws * flops / (ms * 1e-3) / 1e12
    executed = ws * LINEAR_GEMMS[args.schedule] * 2.0 * M * V * H / (ms * 1e-3) / 1e12
    assert api.ce_check_errors() == 0
    # the dominant kernel (the logits GEMM of one row chunk), timed live
    mc = min(M, 2048)
    logits = torch.empty((mc, V), dtype=torch.float32, device=dev)
    for _ in range(2):
        L.ce_gemm_bf16_tn(h.data_ptr(), H, W.data_ptr(), H, logits.data_ptr(), V, mc, V, H, 0.0, sh)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(5):
        L.ce_gemm_bf16_tn(h.data_ptr(), H, W.data_ptr(), H, logits.data_ptr(), V, mc, V, H, 0.0, sh)
    g1.record()
    torch.cuda.synchronize()
    gemm_ms = g0.elapsed_time(g1) / 5
    gemm_tf = 2.0 * mc * V * H / (gemm_ms * 1e-3) / 1e12
    peak, peak_kind = measured_tflops()
    del logits
    # end to end: host h, W, targets -> device, the call, loss, dH and dW -> host
    e2e_steps = max(3, min(args.steps, 6))
    e2e_ms, e2e_serial_ms = linear_e2e(L, api, (h_host, W_host, t_host), (h, W, t, dH, dW, loss),
                                       work, wsb, M, H, V, e2e_steps)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    if rank == 0:
        line = {
            "metric": "fused linear+CE fwd+bwd TFLOP/s (6 M V H per step)", "value": value,
            "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{args.workload}: bf16 h [{M}, {H}] N(0,1), W [{V}, {H}] "
                                   "N(0, 0.02^2), int64 targets; loss, dH, dW (fp32)",
                       "M": M, "H": H, "V": V, "workspace_bytes": wsb,
                       "schedule": args.schedule, "logits_stored": args.schedule == "fused"},
            "executed_tflop_s": executed,
            "roofline": {"bound": "tensor", "achieved": gemm_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": gemm_tf / peak, "peak_source": peak_kind,
                         "traffic": None, "kernel": f"logits GEMM [{mc}, {V}, {H}]",
                         "ms_per_launch": gemm_ms},
            "e2e": {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": (M * H + V * H) * 2 + M * 8,
                    "d2h_bytes_per_step": 4 + (M * H + V * H) * 4,
                    "ms_per_step": e2e_ms, "serial_ms_per_step": e2e_serial_ms,
                    "what": "pinned host h, W, targets -> device, linear_ce_fwd_bwd, loss + dH + "
                            "dW -> pinned host, every step; two device buffer sets in turn, "
                            "copies on their own streams"},
            "gpu_launches": launches, "clocks": clocks,
        }
        if ws == 1 and not args.no_cpu_baseline:
            try:
                line["cpu_baseline"] = linear_cpu_baseline(h_np, W_np, t_np, M, H, V,
                                                           args.cpu_budget_s)
            except Exception as e:  # never costs the line its GPU figures
                line["cpu_baseline"] = {"kind": "oracle", "error": f"{type(e).__name__}: {e}"[:200]}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def blas_threads() -> int:
    """Threads numpy's BLAS uses for a matmul (threadpoolctl when present, else
    the host's CPU count, the BLAS default)."""
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads", 0) for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def linear_cpu_baseline(h_bits, W_bits, t, M: int, H: int, V: int, budget_s: float) -> dict:
    """The float64 oracle as it stands (logits = h W^T, the CE pass, dH, dW) on
    a bounded sample of the workload: its first rows of h against the whole W,
    6 V H flops a row as in the full step.  The bf16 decoding is done once,
    outside the timed region."""
    import oracle
    W64 = oracle.to_f64(W_bits, "bf16")
    h64 = oracle.to_f64(h_bits, "bf16")
    t0 = time.perf_counter()
    oracle.linear_ce(h64[:1], W64, t[:1], "mean")
    dt = time.perf_counter() - t0
    rows = int(min(M, max(1, budget_s / max(dt, 1e-6))))
    t0 = time.perf_counter()
    oracle.linear_ce(h64[:rows], W64, t[:rows], "mean")
    dt = time.perf_counter() - t0
    n = blas_threads()
    return {"value": 6.0 * rows * V * H / dt / 1e12, "unit": "TFLOP/s", "cores": n,
            "kind": "oracle", **host_info(),
            "sample": f"{rows} of {M} rows of h against the whole W [{V}, {H}], loss, dH "
                      f"and dW in float64 numpy ({dt:.1f} s, {n} BLAS threads)"}


def run_linear_reference(args):
    """The reference arm of the linear + CE workload: the float64 oracle on the
    host, each step on a bounded sample (the first rows of h against the whole
    W, 6 V H flops a row as in the full step); rank 0 alone."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    M, H, V = LINEAR_SHAPES[args.workload]
    if args.rows is not None:
        M = args.rows
    h_np, W_np, t_np = synthetic.make_linear_ce_inputs(M, H, V, seed=0)
    W64 = oracle.to_f64(W_np, "bf16")
    for _ in range(args.warmup):
        oracle.linear_ce(oracle.to_f64(h_np[:1], "bf16"), W64, t_np[:1], "mean")
    # a one-row probe sizes the steps (timed apart from the warm-up calls, so it
    # exists whatever the warm-up count)
    t0 = time.perf_counter()
    oracle.linear_ce(oracle.to_f64(h_np[:1], "bf16"), W64, t_np[:1], "mean")
    one_row_s = time.perf_counter() - t0
    # rows per step: the steps together take about a minute (at least one row)
    step_budget = max(0.5, 60.0 / max(1, args.steps))
    rows = int(max(1, min(M, args.ref_rows, step_budget / max(one_row_s, 1e-6))))
    h64 = oracle.to_f64(h_np[:rows], "bf16")
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.linear_ce(h64, W64, t_np[:rows], "mean")
        times.append(time.perf_counter() - t0)
    step_s = sum(times) / len(times)
    tf = 6.0 * rows * V * H / step_s / 1e12
    n = blas_threads()
    sample = (f"{rows} of {M} rows of h against the whole W [{V}, {H}] per step, loss, dH "
              f"and dW in float64 numpy ({n} BLAS threads); bf16 decoding outside the steps")
    print(json.dumps({
        "impl": "reference", "metric": "fused linear+CE fwd+bwd TFLOP/s (6 M V H per step)",
        "value": tf, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: bf16 h [{M}, {H}] N(0,1), W [{V}, {H}] "
                               "N(0, 0.02^2), int64 targets; loss, dH, dW",
                   "M": M, "H": H, "V": V, "sample_rows": rows},
        "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": n, "kind": "oracle",
                         **host_info(), "sample": sample},
        "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


# ---------------------------------------------------------------------------
# blockwise attention forward (the flash-attention page's benchmark shape)
# ---------------------------------------------------------------------------
ATTN_SHAPES = {"attn_causal_32x96x512x128": (32, 96, 512, 128, True)}
ATTN_SOURCES = ("ce_attention.cu", "ce_tc.cuh", "ce_rows.cuh")
# DRAM traffic of the attention kernel per launch on the workload above, from
# `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum`, valid only for
# the attention sources it was taken on.
ATTN_NCU_TRAFFIC = {
    # bf16 [32, 96, 512, 128] causal, bf16 output
    "9a59bd1f46a665591a8092ac661dbed087c0e348b35beef0c476b0da869b5981": {
        "workload": "attn_causal_32x96x512x128", "bytes_per_launch": 1208061696 + 383948288},
}


def attention_digest() -> str:
    d = os.path.join(ROOT, "softmax_cross_entropy_online_gb300", "csrc")
    h = hashlib.sha256()
    for f in ATTN_SOURCES:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()


def attention_bytes(B: int, NH: int, T: int, D: int, out_bytes: int = 2) -> int:
    """Bytes the method must move: one read of the bf16 q, k and v, one write of
    the output (bf16 like q: 2 bytes an element; fp32: 4) and the fp32 lse."""
    return 3 * B * NH * T * D * 2 + B * NH * T * D * out_bytes + B * NH * T * 4


def attention_flops(B: int, NH: int, T: int, D: int, causal: bool, heads: int | None = None) -> float:
    """FLOPs the method must do: 2 D for each visible (query, key) pair in
    Q K^T and again in P V (T (T + 1) / 2 pairs per head under the causal
    mask, T^2 without)."""
    pairs = T * (T + 1) // 2 if causal else T * T
    return 4.0 * D * pairs * (B * NH if heads is None else heads)


def attention_desc(name, B, NH, T, D, causal):
    return (f"{name}: q, k, v bf16 [{B}, {NH}, {T}, {D}] N(0,1), "
            f"{'causal' if causal else 'no'} mask, sm_scale 1/sqrt({D}); "
            "out bf16 (allocated like q, as the page does) + fp32 lse")


def attention_oracle_sample(B, NH, T, D, causal, budget_s):
    """Time the float64 oracle on whole heads of the workload (about budget_s
    of CPU work); returns (TFLOP/s, heads, seconds)."""
    from oracle import attention_oracle as AO
    q, k, v = synthetic.make_attention_inputs(1, 4, T, D, seed=0)
    widen = lambda b: (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)  # noqa: E731
    q, k, v = widen(q)[0], widen(k)[0], widen(v)[0]
    mask = AO.causal_mask(T) if causal else None
    t0 = time.perf_counter()
    AO.attention_forward(q[:1], k[:1], v[:1], mask)
    one = max(time.perf_counter() - t0, 1e-6)
    heads = int(max(1, min(B * NH, budget_s / one)))
    reps = (heads + 3) // 4
    t0 = time.perf_counter()
    done = 0
    for _ in range(reps):
        n = min(4, heads - done)
        AO.attention_forward(q[:n], k[:n], v[:n], mask)
        done += n
    dt = time.perf_counter() - t0
    return attention_flops(B, NH, T, D, causal, heads) / dt / 1e12, heads, dt


def run_attention(args):
    import torch
    from softmax_cross_entropy_online_gb300 import api, build

    ws, rank, local = dist_env()
    B, NH, T, D, causal = ATTN_SHAPES[args.workload]
    name = args.workload
    if args.heads is not None:  # a smaller case of the same shape (profiling)
        B, NH, name = 1, args.heads, f"{args.workload}[heads={args.heads}]"
    desc = attention_desc(name, B, NH, T, D, causal)
    metric = "blockwise attention forward TFLOP/s (4 D per visible query-key pair)"
    if args.impl == "reference":
        if rank != 0:
            return 0
        vals, hs, secs = [], 0, 0.0
        for _ in range(args.warmup):
            attention_oracle_sample(B, NH, T, D, causal, 0.2)
        for _ in range(args.steps):
            v, hs, secs = attention_oracle_sample(B, NH, T, D, causal, args.cpu_budget_s / 4)
            vals.append(v)
        val = sum(vals) / len(vals)
        sample = f"{hs} of {B * NH} heads per step (float64 numpy oracle, 1 thread)"
        print(json.dumps({
            "impl": "reference", "metric": metric, "value": val, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": desc, "B": B, "NH": NH, "T": T, "D": D},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", **host_info(),
                             "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    L = api.lib()
    qb, kb, vb = synthetic.make_attention_inputs(B, NH, T, D, seed=0)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    hosts = [as_bf16(a).pin_memory() for a in (qb, kb, vb)]
    del qb, kb, vb
    q, k, v = (h.to(dev) for h in hosts)
    out = torch.empty((B, NH, T, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, NH, T), dtype=torch.float32, device=dev)
    sh = torch.cuda.current_stream(dev).cuda_stream
    scale = 1.0 / float(np.sqrt(D))
    CE_BF16 = 2

    def step():
        st = L.ce_attention_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), None, int(causal),
                                    B, NH, T, D, scale, out.data_ptr(), CE_BF16, lse.data_ptr(),
                                    sh)
        if st != 0:
            raise api.CEError(st, "ce_attention_forward")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n0 = api.ce_launch_count()
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    launches = api.ce_launch_count() - n0
    clocks = sampler.stop() if sampler else None
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    if ws > 1:
        dist.barrier()
    flops = attention_flops(B, NH, T, D, causal)
    value = ws * flops / (ms * 1e-3) / 1e12
    assert api.ce_check_errors() == 0
    peak, peak_kind = measured_tflops(burst=True)
    hbm_peak, hbm_kind = measured_peaks()
    abytes = attention_bytes(B, NH, T, D)
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = abytes / (ms * 1e-3) / 1e9
    # the bound that binds: HBM time of the algorithmic bytes against tensor
    # time of the algorithmic flops, both at the measured peaks
    hbm_bound = abytes / (hbm_peak * 1e9) >= flops / (peak * 1e12)
    tr = ATTN_NCU_TRAFFIC.get(attention_digest())
    # end to end: q, k, v from pinned host memory, the call, out and lse back
    out_host = torch.empty((B, NH, T, D), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((B, NH, T), dtype=torch.float32).pin_memory()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(2, min(args.steps, 5))
    x0.record()
    for _ in range(e2e_steps):
        for d_, h_ in zip((q, k, v), hosts):
            d_.copy_(h_, non_blocking=True)
        step()
        out_host.copy_(out, non_blocking=True)
        lse_host.copy_(lse, non_blocking=True)
    x1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(x0.elapsed_time(x1) / e2e_steps, dev)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cv, hs, secs = attention_oracle_sample(B, NH, T, D, causal, args.cpu_budget_s)
        cpu = {"value": cv, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", **host_info(),
               "sample": f"{hs} of {B * NH} heads in float64 numpy ({secs:.1f} s on 1 host "
                         "thread)"}
    if rank == 0:
        print(json.dumps({
            "metric": metric, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": desc, "B": B, "NH": NH, "T": T, "D": D, "causal": causal,
                       "l2": f"inputs (3 x {B * NH * T * D * 2 / 1e6:.0f} MB) "
                             + ("larger than L2" if 3 * B * NH * T * D * 2 > 129e6 else
                                "within L2")},
            "roofline": ({"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                          "frac": gbs / hbm_peak, "peak_source": hbm_kind,
                          "algorithmic_bytes": abytes}
                         if hbm_bound else
                         {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                          "frac": tflops / peak, "peak_source": peak_kind})
            | {"traffic": None if tr is None else tr["bytes_per_launch"],
               "tensor": {"achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                          "frac": tflops / peak, "peak_source": peak_kind},
               "kernel": f"attention_fwd_kernel<{D}>", "ms_per_launch": ms},
            "e2e": {"value": ws * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": 3 * B * NH * T * D * 2,
                    "d2h_bytes_per_step": B * NH * T * (D * 2 + 4), "ms_per_step": e2e_ms},
            "cpu_baseline": cpu, "gpu_launches": launches, "clocks": clocks}), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="f32_32768x4096",
                    choices=sorted(synthetic.WORKLOADS) + sorted(LINEAR_SHAPES)
                    + sorted(ATTN_SHAPES))
    ap.add_argument("--max-resident-gb", type=float, default=64.0)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=1024)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-workloads", action="store_true",
                    help="time only the headline workload (no fp16/bf16/small side records)")
    ap.add_argument("--no-linear-side", action="store_true",
                    help="leave the fused linear + CE step out of the side records")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of back-to-back calls during which the clocks are sampled")
    ap.add_argument("--rows", type=int, default=None,
                    help="override the workload's row count (smaller cases for profiling)")
    ap.add_argument("--vocab", type=int, default=None,
                    help="linear + CE workload: override V (smaller cases for profiling)")
    ap.add_argument("--schedule", choices=["lean", "fused"], default="lean",
                    help="linear + CE workload: the lean schedule (no logits stored, the "
                         "default) or the fused one (fp32 logits chunks)")
    ap.add_argument("--heads", type=int, default=None,
                    help="attention workloads: run B = 1 with this many heads instead")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps, always
    if args.workload in ATTN_SHAPES:
        return run_attention(args)
    if args.workload in LINEAR_SHAPES:
        if args.impl == "reference":
            return run_linear_reference(args)
        return run_linear(args)
    w = synthetic.WORKLOADS[args.workload]
    if args.rows is not None:
        w = dataclasses.replace(w, M=args.rows, name=f"{w.name}[rows={args.rows}]")
    if args.impl == "reference":
        return run_reference(args, w)
    return run_native(args, w)


if __name__ == "__main__":
    sys.exit(main())
