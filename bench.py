#!/usr/bin/env python3
"""Benchmark of libapsp (blocked Floyd-Warshall APSP) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload ba16384]

One step = one full solve (all rounds of phases 1-3) of the workload's n x n
matrix, already resident in device memory.  Before each step the input is
restored from a pristine device copy; the restore is not timed.  The matrix
(1 GiB at n = 16384) is far larger than L2, so no flush is needed.  Metric:
relaxations per second, n^3 / solve time.

Prints one JSON line (rank 0).  Under torchrun with N > 1 every rank solves
its own replica (replicas only: the path has no exchange step on one GPU).
The throughput is summed over ranks and the time is the maximum over ranks.

--impl reference times the CPU oracle (the untiled triple loop, all host
cores) on a bounded sample of the same workload: the first few k-steps of
Floyd-Warshall on the full matrix.

--algo johnson measures the sparse path instead: Johnson's APSP with one
Delta-stepping search per source (min_graph_gb300.solve_sparse) on the same
int32 matrix, with the same n^3 / time unit so the two methods compare
directly.  Its roofline is the search kernel's arc stream (8 bytes per
packed arc and 20 per vertex range, per source) against the L2 read
bandwidth measured in the same run; the CPU baseline and the reference arm
time the oracle's binary-heap Dijkstra from a sample of sources.

--algo sssp measures the grid-wide single-source Delta-stepping search
(min_graph_gb300.sssp) on an R-MAT graph of 2^scale vertices and 32 arcs per
vertex, as the Delta-stepping page does: one step is one search from a
seeded random source, and the metric is traversed edges per second (m /
search time).  Its roofline is HBM: 8 bytes per arc and 16 per vertex per
search against the measured copy bandwidth.  The CPU baseline and the
reference arm time the oracle's CSR Dijkstra from one source.

--algo ooc measures the out-of-core solver (min_graph_gb300.solve_ooc): the
workload's matrix in pinned host memory, streamed through the GPU in K x K
super-blocks (--block).  A step is one whole blocking call, copies included,
so value and e2e are the same figure; the input is restored on the host
before each step, outside the timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import graphgen  # noqa: E402

METRIC = "APSP relaxations/sec (n³/time) and % of GB300 INT32 add-min peak, 1 GPU"
UNIT = "relaxations/s"
OOC_METRIC = METRIC.replace(", 1 GPU", ", out-of-core from host memory, 1 GPU")
TB = 128
NOMINAL_INT32_LANES = 128  # INT32 lanes per SM per clock (nominal, one add-min per lane)
SMALL_MAX_N = 512  # n at or below which the library solves in one launch of a thread-block cluster
SMALL_BLOCK = 32   # that kernel's block edge


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ba16384", choices=sorted(graphgen.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--threads", type=int, default=0, help="host threads for the oracle (0: all cores)")
    ap.add_argument("--algo", choices=["fw", "johnson", "sssp", "ooc"], default="fw")
    ap.add_argument("--block", type=int, default=4096, help="super-block K for --algo ooc (0: from the budget)")
    ap.add_argument("--device-bytes", type=int, default=0, help="device budget for --algo ooc (0: 70%% of free)")
    ap.add_argument("--scale", type=int, default=22, help="R-MAT scale for --algo sssp")
    ap.add_argument("--delta", type=int, default=0, help="Delta for --algo johnson (0: the library's default)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(dist, x: float, device) -> float:
    """The largest x over all ranks (x itself without a process group): the
    timed region of a multi-rank run is the slowest rank's."""
    if dist is None:
        return float(x)
    import torch

    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world: int, steps: int, work_per_step: float, seconds: float) -> float:
    """Whole-job throughput: every rank does `steps` steps of `work_per_step`
    units (replicas), in the slowest rank's `seconds`."""
    return world * steps * work_per_step / seconds


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except OSError:
        return {}


# ------------------------------------------------------------------ clocks

# NVML clock-event reason bits (nvml.h) that the timing rules watch
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown"}


class _Nvml:
    """Read-only NVML queries through ctypes: the SM clock, its maximum and
    the active clock-event reasons of one GPU (no setting is changed)."""

    CLOCK_SM = 1  # NVML_CLOCK_SM

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            self.lib.nvmlShutdown()
            raise OSError("no NVML handle for this GPU")
        try:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self):
        clk, rs = self.ct.c_uint(0), self.ct.c_ulonglong(0)
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, self.ct.byref(clk)) != 0:
            return None
        if self.reasons_fn(self.h, self.ct.byref(rs)) != 0:
            return None
        return clk.value, rs.value

    def max_sm(self):
        mx = self.ct.c_uint(0)
        return mx.value if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM, self.ct.byref(mx)) == 0 else None

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs.
    In-process NVML every 0.2 ms (one sample right before and one right
    after the region as well), so that timed regions of a few milliseconds
    are covered; nvidia-smi every 200 ms where NVML cannot be loaded."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None
        self.nvml = None
        self.thread = None
        self.samples = []
        self.stop = False

    def _loop(self):
        while not self.stop:
            x = self.nvml.sample()
            if x is not None:
                self.samples.append(x)
            time.sleep(0.0002)

    def __enter__(self):
        try:
            self.nvml = _Nvml(self.gpu)
        except (OSError, AttributeError):
            self.nvml = None
        if self.nvml is not None:
            import threading
            x = self.nvml.sample()
            if x is not None:
                self.samples.append(x)
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()
            time.sleep(0.02)  # running steadily before the timed region starts
            return self
        try:
            self.out = open(f"/tmp/apsp_clocks_{os.getpid()}.csv", "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.02)  # started before the timed region
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop = True
            self.thread.join(timeout=5)
            x = self.nvml.sample()
            if x is not None:
                self.samples.append(x)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.out is not None:
            self.out.close()

    def summary(self):
        if self.nvml is not None:
            mx = self.nvml.max_sm()
            self.nvml.close()
            if not self.samples:
                return None
            reasons = sorted({name for _, r in self.samples for bit, name in NVML_REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(float(c) for c, _ in self.samples),
                    "sm_max_mhz": float(mx) if mx is not None else None,
                    "samples": len(self.samples), "reasons": reasons, "source": "nvml, every 0.2 ms"}
        if self.proc is None or self.out is None:
            return None
        rows = []
        try:
            with open(self.out.name) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
            os.unlink(self.out.name)
        except OSError:
            return None
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "samples": len(rows), "reasons": reasons, "source": "nvidia-smi, every 200 ms"}


# ------------------------------------------------------------------ CPU side

FW_SAMPLE_RELAX = 4e10  # relaxations per CPU sample: the whole solve when n^3 fits, else n^2 per k-step
FW_SAMPLE_K0 = 256       # k-steps a partial sample starts after (computed once, untimed)


def fw_sample_plan(n: int):
    """(k0, S): a CPU sample of an n-vertex Floyd-Warshall times k-steps
    k0 .. k0+S-1.  The whole solve (0, n) when n^3 <= FW_SAMPLE_RELAX; else
    S = that budget / n^2 steps starting after the first FW_SAMPLE_K0, whose
    state is computed once, untimed.  Fixed counts, so every sample of a
    workload times the same steps on the same matrix states."""
    if float(n) ** 3 <= FW_SAMPLE_RELAX:
        return 0, n
    S = max(1, min(n, int(round(FW_SAMPLE_RELAX / (float(n) * n)))))
    return max(0, min(FW_SAMPLE_K0, n - S)), S


L2_FLUSH_BYTES = 256 << 20  # larger than the 129 MB L2


def fw_needs_flush(n: int, itemsize: int) -> bool:
    """Inputs smaller than the flush buffer are timed after an L2 flush."""
    return n * n * itemsize < L2_FLUSH_BYTES


def fw_config(workload: str, n: int, w: np.ndarray, world: int) -> dict:
    """The `config` of the Floyd-Warshall lines, shared verbatim by both arms."""
    nbytes = n * n * w.itemsize
    if fw_needs_flush(n, w.itemsize):
        l2 = (f"input {nbytes / 2**20:.2f} MiB < L2: restored from a device copy, then L2 flushed by "
              f"writing a {L2_FLUSH_BYTES >> 20} MiB buffer, before each step, outside the timed events")
    else:
        l2 = (f"input {nbytes / 2**30:.2f} GiB > L2; restored from a device copy before each step, "
              "outside the timed events")
    return {"workload": workload, "n": n, "graph": graphgen.describe(workload), "l2": l2,
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def fw_sample_state(w: np.ndarray, k0: int, threads: int) -> np.ndarray:
    """The oracle's matrix after its first k0 k-steps (int32 clamped to INF;
    fp32 as fp64), untimed: the starting state of every partial sample."""
    import oracle

    is_i32 = w.dtype == np.int32
    d = (np.array(np.minimum(w, graphgen.INF_I32), dtype=np.int32, copy=True) if is_i32
         else np.array(w, dtype=np.float64, copy=True))
    if k0 > 0:
        (oracle.default().fw_i32_steps if is_i32 else oracle.default().fw_f64_steps)(d, 0, k0, threads=threads)
    return d


def time_fw_sample(state: np.ndarray, k0: int, ksteps: int, threads: int):
    """One CPU sample: the oracle's untiled Floyd-Warshall (OpenMP over rows)
    runs k-steps k0 .. k0+ksteps-1 on a fresh copy of `state`.  Returns
    (seconds, relaxations in the metric's unit, mean fraction of rows the
    sampled steps process).

    The oracle skips row i of step k while D[i][k] is INF (no path i ~> k
    through earlier vertices yet).  A whole solve counts n^3, the metric's
    definition.  A partial sample counts the relaxations the oracle executed
    (n per processed row): past the first few hundred k-steps of these
    connected graphs nearly every row is processed, so that rate estimates a
    whole solve's n^3 rate.  Rows are counted outside the timed calls."""
    import oracle

    d = np.array(state, copy=True)
    is_i32 = d.dtype == np.int32
    steps = oracle.default().fw_i32_steps if is_i32 else oracle.default().fw_f64_steps
    n = d.shape[0]
    dt, rows = 0.0, 0
    for k in range(k0, k0 + ksteps):
        col = d[:, k]
        rows += int(np.count_nonzero(col < graphgen.INF_I32) if is_i32 else np.count_nonzero(np.isfinite(col)))
        t0 = time.perf_counter()
        steps(d, k, k + 1, threads=threads)
        dt += time.perf_counter() - t0
    units = float(n) ** 3 if (k0 == 0 and ksteps == n) else float(rows) * n
    return dt, units, rows / (ksteps * float(n))


def fw_sample_text(workload: str, n: int, k0: int, ksteps: int, is_i32: bool, dense: float, threads: int,
                   seconds: float) -> str:
    what = ("the whole solve" if (k0 == 0 and ksteps == n)
            else f"k-steps {k0}..{k0 + ksteps - 1} of {n} (from the state after the first {k0}, computed once, untimed)")
    head = (f"{what} of the oracle's untiled Floyd-Warshall ({'int32' if is_i32 else 'fp64'}, OpenMP over rows) "
            f"on the full n={n} {workload} matrix, each sample from a fresh copy; {seconds:.3g} s timed, "
            f"{threads} threads")
    if k0 == 0 and ksteps == n:
        return head + "; value = n^3 / time"
    return (head + f"; the sampled steps processed {dense:.1%} of their rows (the oracle skips row i of "
            "step k while D[i][k] is INF); value = relaxations executed per second, which estimates a whole "
            "solve's n^3 rate since past its first few hundred k-steps a whole solve of this connected graph "
            "processes nearly every row")


def reference_arm(args, rank, ooc: bool = False):
    """--impl reference: the oracle as it stands, on the host cores.  Each
    step is one sample (fw_sample_plan) from the same starting state, so every
    step times the same work."""
    if rank != 0:
        return
    import oracle

    w = graphgen.make(args.workload)
    n = w.shape[0]
    is_i32 = w.dtype == np.int32
    thr = args.threads or oracle.default_threads()
    k0, ks = fw_sample_plan(n)
    state = fw_sample_state(w, k0, thr)
    times, relax, dense = [], [], []
    for step in range(args.warmup + args.steps):
        dt, rx, fr = time_fw_sample(state, k0, ks, thr)
        if step >= args.warmup:
            times.append(dt)
            relax.append(rx)
            dense.append(fr)
    tot = sum(times)
    value = sum(relax) / tot
    sample = fw_sample_text(args.workload, n, k0, ks, is_i32, float(np.mean(dense)), thr, tot)
    line = {
        "impl": "reference", "metric": OOC_METRIC if ooc else METRIC, "value": value, "unit": UNIT,
        "n_gpus": 1 if ooc else args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32" if is_i32 else "f32",
        "data": "synthetic",
        "config": ooc_config(args, n, args.block or None) if ooc else fw_config(args.workload, n, w, args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU side

def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("fw_kernels.cuh", "fw_fused.cuh", "fw_cluster.cuh", "fw_launch_impl.cuh", "mm_core.cuh", "tma.cuh"):
        with open(os.path.join(ROOT, "min_graph_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def phase3_traffic(n: int):
    """DRAM bytes per phase-3 launch from the committed ncu summary, scaled by
    tiles; None when the kernel source changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "fw_phase3_persistent_er8192_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except OSError:
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None
    nb = -(-n // TB)
    return rec["dram_bytes_per_tile"] * (nb - 1) ** 2 / 1e9  # GB per launch


def fused_traffic(n: int):
    """DRAM bytes per fw_round_fused launch from the committed ncu summary,
    scaled by work items; None when the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "fw_round_fused_er8192_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except OSError:
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None
    nb = -(-n // TB)
    return rec["dram_bytes_per_item"] * nb * nb / 1e9  # GB per (full lookahead) launch


def ours(args, rank, world, local):
    import torch

    import min_graph_gb300 as apsp

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    cfg = graphgen.CONFIGS[args.workload]
    n = cfg["n"]
    w = graphgen.make(args.workload)
    dtype = torch.int32 if w.dtype == np.int32 else torch.float32
    pristine = torch.from_numpy(w).to(dev)
    work = torch.empty_like(pristine)
    stream = torch.cuda.current_stream(dev)

    def step_solve():
        apsp.solve(work, stream=stream)

    nb = -(-n // TB)
    small_path = n <= SMALL_MAX_N and os.environ.get("APSP_SMALL", "1") != "0"
    fused_schedule = os.environ.get("APSP_FUSED", "1") != "0"
    launches_per_solve = (1 if small_path else (nb + 1) if fused_schedule
                          else nb + (2 * nb if nb > 1 else 0))
    # The tile-product core's relaxation rate on this GPU, measured now by
    # the issue-rate probe (libapsp_peak: the library's own inner loop on a
    # shared-memory slab, one 256-thread block per SM): the achievable peak
    # beside the nominal one.
    import min_graph_gb300.peak as peak

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    probe_variant = 8 if dtype == torch.int32 else 13  # the core phase 3 runs (fused add-min / packed fp32)
    probe = peak.measure(probe_variant, sms, 256, 8192)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    flush = (torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
             if fw_needs_flush(n, w.itemsize) else None)

    def step(k, timed):
        work.copy_(pristine)  # restore the input (outside the events)
        if flush is not None:
            flush.fill_(k)  # evict the input and the workspace from L2
        if timed:
            starts[k].record(stream)
        step_solve()
        if timed:
            ends[k].record(stream)

    # warm-up: the timed loop's own sequence, after the probe, so that the
    # first timed step finds the GPU in the state the others do
    for k in range(args.warmup):
        step(k, False)
    apsp.stream_check(stream)
    barrier()
    with ClockSampler(local) as clocks:
        for k in range(args.steps):
            step(k, True)
        barrier()
    apsp.stream_check(stream)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # A separate, instrumented pass (not part of the headline): CUDA events
    # around every launch, which splits a solve into its phases.  The events
    # between launches hold back the overlap of consecutive launches, so
    # these launch times are slightly longer than the headline's.
    apsp.phase_timing_read()
    apsp.phase_timing_enable(True)
    for _ in range(min(2, args.steps)):
        work.copy_(pristine)
        step_solve()
    torch.cuda.synchronize()
    apsp.phase_timing_enable(False)
    apsp.stream_check(stream)
    phase_ms, phase_cnt = apsp.phase_timing_read()
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(dist, total_ms, dev)
    relax_per_step = float(n) ** 3
    value = whole_job_value(world, args.steps, relax_per_step, total_ms * 1e-3)

    # correctness spot check of the timed result: four oracle rows
    check = None
    if rank == 0:
        import oracle

        src = np.array([0, n // 3, (2 * n) // 3, n - 1], dtype=np.int32)
        got = work[src.tolist(), :].cpu().numpy()
        if dtype == torch.int32:
            ref = oracle.dijkstra_i32(w, src)
            check = bool(np.array_equal(got, ref))
        else:
            ref = oracle.dijkstra_f32(w, src)
            fin = np.isfinite(ref)
            check = bool(np.array_equal(np.isfinite(got), fin) and
                         np.all(np.abs(got[fin] - ref[fin]) <= 1e-5 * np.abs(ref[fin])))

    # end to end through the host-buffer C-ABI calls (pinned memory).  The
    # headline: the K steps as one batched call, each step's matrix uploaded
    # from the pinned input and its result downloaded into a pinned output,
    # copies overlapped with the neighbouring steps' solves.  Beside it: K
    # single calls, each copying in, solving and copying out in turn.
    e2e = None
    if not args.no_e2e:
        host_src = torch.from_numpy(w)
        pinned = torch.empty_like(host_src).pin_memory()
        pinned.copy_(host_src)
        outs = [torch.empty_like(host_src).pin_memory() for _ in range(2)]
        apsp.solve_host_batch([pinned, pinned], outs)  # warm-up (allocates the staging buffers)
        barrier()
        t0 = time.perf_counter()
        apsp.solve_host_batch([pinned] * args.steps, [outs[b % 2] for b in range(args.steps)])
        batch_total = max_over_ranks(dist, time.perf_counter() - t0, dev)
        e2e_ok = bool(torch.equal(outs[(args.steps - 1) % 2][:4], work[:4].cpu()))
        single_times = []
        for _ in range(args.steps):
            outs[0].copy_(host_src)
            barrier()
            t0 = time.perf_counter()
            apsp.solve_host(outs[0])
            single_times.append(time.perf_counter() - t0)
        single_total = max_over_ranks(dist, sum(single_times), dev)
        nbytes = n * n * w.itemsize
        e2e = {"value": whole_job_value(world, args.steps, relax_per_step, batch_total), "unit": UNIT,
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
               "ms_per_step": batch_total / args.steps * 1e3,
               "api": "apsp_solve_host_batch (copies overlapped with neighbouring steps' solves)",
               "result_matches_device_solve": e2e_ok,
               "single_call": {"value": whole_job_value(world, args.steps, relax_per_step, single_total),
                               "ms_per_step": single_total / args.steps * 1e3, "api": "apsp_solve_host"}}

    # roofline of the dominant kernel (phase 3): algorithmic relaxations per
    # launch / average launch time, against SMs x 128 lanes x clock
    pk = peaks()
    clk = clocks.summary()
    f_max = (clk or {}).get("sm_max_mhz") or pk.get("sm_max_mhz", 2070.0)
    f_load = (clk or {}).get("sm_mhz")
    f_gemm = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")
    fused = phase_cnt[0] == 0 and phase_cnt[2] > 0
    inst_launches = phase_cnt[2]
    inst_ms = phase_ms[2] / inst_launches if inst_launches else None
    npad = nb * TB
    if small_path:
        # one launch of the one-cluster kernel: all (32 ceil(n/32))^3
        # relaxations of the 32-wide blocked solve
        kernel = "fw_cluster_small"
        p3_relax = float(SMALL_BLOCK * -(-n // SMALL_BLOCK)) ** 3
        p3_launches = args.steps
        p3_ms = sum(step_ms) / p3_launches
        launch_basis = "timed solves' CUDA events (one launch per solve)"
    elif fused:
        # round-fused schedule: all of a solve's npad^3 relaxations (phases 1-3)
        # run in its nb + 1 launches of fw_round_fused, which take the whole
        # solve; the average launch is the timed solves' time over their
        # launches (the short gaps between launches included)
        kernel = "fw_round_fused"
        p3_relax = float(npad) ** 3 / (nb + 1)
        p3_launches = args.steps * (nb + 1)
        p3_ms = sum(step_ms) / p3_launches
        launch_basis = "timed solves' CUDA events / launches (gaps between launches included)"
    else:
        # three-kernel schedule: phase 3's own launches, from the
        # instrumented pass's per-launch events
        p3_launches, p3_ms = inst_launches, inst_ms
        launch_basis = "per-launch CUDA events of the instrumented pass"
        kernel = ("fw_phase3_minplus" if os.environ.get("APSP_PHASE3") == "cpasync"
                  else "fw_phase3_persistent")
        p3_relax = float(nb - 1) ** 2 * TB ** 3 if nb > 1 else 0.0
    ops_per_relax = 1 if dtype == torch.int32 else 2
    peak_tops = sms * NOMINAL_INT32_LANES * f_max * 1e6 / ops_per_relax / 1e12
    roof = None
    if p3_ms:
        achieved = p3_relax / (p3_ms * 1e-3) / 1e12
        traffic = phase3_traffic(n) if not fused else fused_traffic(n)
        measured_tops = sms * probe["relax_per_clk_sm"] * f_max * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak_tops, "unit": "Trelax/s",
                "frac": achieved / peak_tops, "traffic": traffic,
                "traffic_unit": "GB per launch (DRAM read + write, scaled from the committed ncu capture)",
                "peak_measured_addmin": measured_tops,
                "frac_of_measured_addmin": achieved / measured_tops,
                "kernel": kernel, "peak_basis":
                    f"{sms} SMs x {NOMINAL_INT32_LANES} INT32 lanes x {f_max:.0f} MHz"
                    + (" / 2 ops per fp32 relaxation" if ops_per_relax == 2 else ""),
                "frac_at_load_clock": (achieved / (peak_tops * f_load / f_max)) if f_load else None,
                # the peak at the median SM clock that MEASURED_PEAKS.json saw
                # under a power-capped bf16 GEMM; this kernel's own clock is
                # sampled above (clocks.sm_mhz), and `frac` uses the maximum
                "peak_at_gemm_load_clock": (peak_tops * f_gemm / f_max) if f_gemm else None,
                "frac_at_gemm_load_clock": (achieved / (peak_tops * f_gemm / f_max)) if f_gemm else None,
                "gemm_load_clock_mhz": f_gemm,
                "peak_measured_basis": f"{sms} SMs x {probe['relax_per_clk_sm']:.2f} relaxations/clk/SM "
                                       f"(issue-rate probe in this run: {probe['what']}) x {f_max:.0f} MHz",
                "probe": probe,
                "avg_launch_ms": p3_ms, "launches": p3_launches, "avg_launch_basis": launch_basis,
                "instrumented_pass": {"avg_launch_ms": inst_ms, "launches": inst_launches,
                                      "phase_ms": phase_ms, "phase_launches": phase_cnt},
                "phase_share": [m / sum(phase_ms) for m in phase_ms] if sum(phase_ms) > 0 else None}
        if not fused and phase_cnt[0] > 0 and phase_cnt[1] > 0:
            # the three-kernel schedule times phases 1 and 2 apart: their HBM
            # rates, algorithmic bytes per launch (phase 1: the primary tile
            # read and written; phase 2: each of the 2(nb-1) panel tiles read,
            # written back and written to the workspace panel)
            hbm = peaks().get("hbm_gbs") or 6800.0
            tile = TB * TB * w.itemsize
            p1_ms = phase_ms[0] / phase_cnt[0]
            p2_ms = phase_ms[1] / phase_cnt[1]
            p1_gbs = 2 * tile / (p1_ms * 1e-3) / 1e9
            p2_gbs = 2 * (nb - 1) * 3 * tile / (p2_ms * 1e-3) / 1e9
            roof["phases_1_2"] = {
                "phase1": {"ms_per_launch": p1_ms, "GB/s": p1_gbs, "frac_hbm": p1_gbs / hbm},
                "phase2": {"ms_per_launch": p2_ms, "GB/s": p2_gbs, "frac_hbm": p2_gbs / hbm},
                "hbm_peak_gbs": hbm}
        roof["solve_hbm_GBps"] = 2.0 * w.itemsize * float(n) * n * nb / (total_ms / args.steps * 1e-3) / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_subprocess(args, steps=4, warmup=1)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32" if dtype == torch.int32 else "f32",
            "data": "synthetic",
            "config": fw_config(args.workload, n, w, world),
            "pct_int32_addmin_peak": (roof["frac"] * 100) if roof else None,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * launches_per_solve,
            "clocks": clk, "check_rows_vs_oracle": check,
            "step_ms": step_ms,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------ Johnson arm

JOHNSON_METRIC = "APSP n³/time (Floyd-Warshall-equivalent relaxations/s), Johnson + Delta-stepping, 1 GPU"


def arc_count(w: np.ndarray) -> int:
    n = w.shape[0]
    return int(np.count_nonzero(w < graphgen.INF_I32) - np.count_nonzero(np.diag(w) < graphgen.INF_I32))


def cpu_dijkstra_sample(w: np.ndarray, target_s: float):
    """Time the oracle's binary-heap Dijkstra (all host cores) from seeded
    sources, growing the batch until one call takes about target_s seconds.
    Returns (n^3-equivalent relax/s, sources, seconds, threads)."""
    import oracle

    n = w.shape[0]
    thr = oracle.default_threads()
    rng = np.random.default_rng(7)
    k = min(n, 4 * thr)
    while True:
        src = rng.choice(n, k, replace=False).astype(np.int32)
        t0 = time.perf_counter()
        oracle.dijkstra_i32(w, src, threads=thr)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or k >= n:
            return float(n) ** 2 * k / dt, k, dt, thr
        k = min(n, max(k + 1, int(k * target_s / max(dt, 1e-3))))


def johnson_config(args, n: int, m: int, world: int) -> dict:
    """The `config` of the Johnson lines, shared verbatim by both arms."""
    return {"workload": args.workload, "n": n, "m": m, "graph": graphgen.describe(args.workload),
            "algo": "johnson", "delta": args.delta or "library default",
            "l2": f"input {n * n * 4 / 2**30:.2f} GiB; restored from a device copy before each "
                  "step, outside the timed events; the output rows go to HBM",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def cpu_baseline_subprocess(args, steps: int, warmup: int):
    """A cpu_baseline from the reference arm of the same --algo and workload,
    run as a fresh process (no CUDA context or torch thread pools in it)."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--algo", args.algo,
           "--workload", args.workload, "--scale", str(args.scale), "--block", str(args.block),
           "--steps", str(steps), "--warmup", str(warmup), "--threads", str(args.threads)]
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True, env=env)
    if p.returncode != 0:
        raise RuntimeError("CPU baseline run failed:\n" + p.stderr[-2000:])
    return json.loads(p.stdout.strip().splitlines()[-1])["cpu_baseline"]


def reference_johnson(args, rank):
    if rank != 0:
        return
    w = graphgen.make(args.workload)
    if w.dtype != np.int32:
        raise SystemExit("--algo johnson needs an int32 workload")
    n = w.shape[0]
    vals, secs, ks = [], [], []
    for step in range(args.warmup + args.steps):
        v, k, dt, thr = cpu_dijkstra_sample(w, 2.5)
        if step >= args.warmup:
            vals.append(v)
            secs.append(dt)
            ks.append(k)
    value = sum(float(n) ** 2 * k for k in ks) / sum(secs)
    sample = (f"binary-heap Dijkstra (the oracle's per-source search) from about {int(np.mean(ks))} "
              f"seeded sources of the n={n} {args.workload} graph per step (~2.5 s, {thr} threads), "
              f"scaled to n sources; {sum(secs):.1f} s timed")
    line = {
        "impl": "reference", "metric": JOHNSON_METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sum(secs) / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": johnson_config(args, n, arc_count(w), args.gpus),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ours_johnson(args, rank, world, local):
    import torch

    import min_graph_gb300 as apsp
    import min_graph_gb300.peak as peak

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    w = graphgen.make(args.workload)
    if w.dtype != np.int32:
        raise SystemExit("--algo johnson needs an int32 workload")
    n = w.shape[0]
    m = arc_count(w)
    pristine = torch.from_numpy(w).to(dev)
    work = torch.empty_like(pristine)
    stream = torch.cuda.current_stream(dev)
    l2 = peak.l2_read()  # measured L2 read bandwidth, the roofline's denominator

    for _ in range(args.warmup):
        work.copy_(pristine)
        apsp.solve_sparse(work, delta=args.delta, stream=stream)
    apsp.sparse_timing_read()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clocks:
        apsp.sparse_timing_enable(True)
        for k in range(args.steps):
            work.copy_(pristine)  # restore the input (outside the events)
            starts[k].record(stream)
            apsp.solve_sparse(work, delta=args.delta, stream=stream)
            ends[k].record(stream)
        barrier()
        apsp.sparse_timing_enable(False)
    search_ms, searches, kernels = apsp.sparse_timing_read()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(dist, total_ms, dev)
    value = whole_job_value(world, args.steps, float(n) ** 3, total_ms * 1e-3)

    check = None
    if rank == 0:
        import oracle

        src = np.array([0, n // 3, (2 * n) // 3, n - 1], dtype=np.int32)
        check = bool(np.array_equal(work[src.tolist(), :].cpu().numpy(), oracle.dijkstra_i32(w, src)))

    # end to end: each step uploads the dense matrix from pinned host memory,
    # solves it and downloads the result.  The copies run on a copy stream
    # into and out of two device buffers, so step b + 1's upload and step
    # b - 1's download overlap the solve of step b (as the batched host
    # entry point of the dense solver does).
    e2e = None
    if not args.no_e2e:
        host_src = torch.from_numpy(w)
        pinned = torch.empty_like(host_src).pin_memory()
        pinned.copy_(host_src)
        outs = [torch.empty_like(host_src).pin_memory() for _ in range(2)]
        bufs = [torch.empty_like(pristine) for _ in range(2)]
        cs = torch.cuda.Stream(dev)

        def pipelined(count):
            up = [torch.cuda.Event() for _ in range(2)]
            done = [torch.cuda.Event() for _ in range(2)]

            def upload(b):
                with torch.cuda.stream(cs):
                    bufs[b % 2].copy_(pinned, non_blocking=True)
                    up[b % 2].record(cs)

            upload(0)
            if count > 1:
                upload(1)
            for b in range(count):
                k = b % 2
                stream.wait_event(up[k])
                apsp.solve_sparse(bufs[k], delta=args.delta, stream=stream)  # returns when solved
                done[k].record(stream)
                cs.wait_event(done[k])
                with torch.cuda.stream(cs):
                    outs[k].copy_(bufs[k], non_blocking=True)  # then step b + 2's upload reuses bufs[k]
                if b + 2 < count:
                    upload(b + 2)
            cs.synchronize()
            stream.synchronize()

        pipelined(2)  # warm-up
        barrier()
        t0 = time.perf_counter()
        pipelined(args.steps)
        e2e_total = max_over_ranks(dist, time.perf_counter() - t0, dev)
        nbytes = n * n * 4
        e2e = {"value": whole_job_value(world, args.steps, float(n) ** 3, e2e_total), "unit": UNIT,
               "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
               "ms_per_step": e2e_total / args.steps * 1e3,
               "api": "apsp_solve_sparse_i32 on device buffers; copies on a second stream overlap the neighbouring steps' solves",
               "result_matches_device_solve": bool(torch.equal(outs[(args.steps - 1) % 2][:4], work[:4].cpu()))}

    clk = clocks.summary()
    roof = None
    if searches:
        avg = search_ms / searches
        algo_bytes = float(n) * (8.0 * m + 20.0 * n)  # per search launch: every source reads each arc and range once
        achieved = algo_bytes / (avg * 1e-3) / 1e9
        roof = {"bound": "l2", "achieved": achieved, "peak": l2["gbs"], "unit": "GB/s",
                "frac": achieved / l2["gbs"], "traffic": None,
                "kernel": "sssp_delta_kernel", "avg_launch_ms": avg, "launches": searches,
                "algorithmic_bytes_per_launch": algo_bytes,
                "peak_basis": f"L2 read probe in this run ({l2['bytes'] >> 20} MiB buffer, "
                              f"{l2['blocks']} x {l2['threads']} threads, {l2['passes']} passes)",
                "search_share": search_ms / total_ms if total_ms > 0 else None,
                "arc_relaxations_per_s": float(n) * m / (avg * 1e-3)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_subprocess(args, steps=4, warmup=1)

    if rank == 0:
        line = {
            "metric": JOHNSON_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": johnson_config(args, n, m, world),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels, "clocks": clk, "check_rows_vs_oracle": check, "step_ms": step_ms,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------ single-source arm

SSSP_METRIC = "SSSP traversed edges/s (m/time), grid-wide Delta-stepping on R-MAT, 1 GPU"


def sssp_sources(n: int, count: int, row_ptr: np.ndarray) -> np.ndarray:
    """Seeded random sources with at least one out-arc (a source without one
    traverses nothing)."""
    rng = np.random.default_rng(17)
    deg = np.diff(row_ptr)
    out = []
    while len(out) < count:
        v = int(rng.integers(0, n))
        if deg[v] > 0:
            out.append(v)
    return np.array(out, dtype=np.int32)


def sssp_config(args, n: int, m: int, graph_bytes: int, world: int) -> dict:
    """The `config` of the single-source lines, shared verbatim by both arms."""
    return {"workload": f"rmat{args.scale}", "n": n, "m": m, "graph": graphgen.describe_rmat(args.scale),
            "algo": "sssp", "delta": args.delta or "library default",
            "l2": f"graph {graph_bytes / 2**30:.2f} GiB resident; one seeded random source per step",
            "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"}


def reference_sssp(args, rank):
    if rank != 0:
        return
    import oracle

    row_ptr, col, w = graphgen.rmat_csr(args.scale)
    n, m = row_ptr.size - 1, int(row_ptr[-1])
    src = sssp_sources(n, args.warmup + args.steps, row_ptr)
    secs = []
    for q, s in enumerate(src):
        t0 = time.perf_counter()
        oracle.dijkstra_csr_i32(row_ptr, col, w, [int(s)], threads=1)
        if q >= args.warmup:
            secs.append(time.perf_counter() - t0)
    value = m * len(secs) / sum(secs)
    sample = f"the oracle's binary-heap Dijkstra on the CSR graph, one source per step, 1 thread"
    line = {
        "impl": "reference", "metric": SSSP_METRIC, "value": value, "unit": "TEPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sum(secs) / len(secs) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": sssp_config(args, n, m, int(row_ptr.nbytes + col.nbytes + w.nbytes), args.gpus),
        "cpu_baseline": {"value": value, "unit": "TEPS", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TEPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def ours_sssp(args, rank, world, local):
    import torch

    import min_graph_gb300 as apsp

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    row_ptr, col, w = graphgen.rmat_csr(args.scale)
    n, m = row_ptr.size - 1, int(row_ptr[-1])
    stream = torch.cuda.current_stream(dev)
    # the graph is prepared once (checked and partitioned against Delta), as
    # the page builds its CSR once; each step is one search on it
    graph = apsp.SsspGraph(*[torch.from_numpy(a).to(dev) for a in (row_ptr, col, w)], delta=args.delta)
    delta_used = graph.info()[2]
    out = torch.empty(n, dtype=torch.int32, device=dev)
    src = sssp_sources(n, args.warmup + args.steps, row_ptr)
    for s in src[:args.warmup]:
        graph.search(int(s), out=out, stream=stream)
    apsp.sparse_timing_read()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier()
    with ClockSampler(local) as clocks:
        apsp.sparse_timing_enable(True)
        for k, s in enumerate(src[args.warmup:]):
            starts[k].record(stream)
            graph.search(int(s), out=out, stream=stream)
            ends[k].record(stream)
        barrier()
        apsp.sparse_timing_enable(False)
    search_ms, searches, kernels = apsp.sparse_timing_read()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(step_ms)
    total_ms = max_over_ranks(dist, total_ms, dev)
    value = whole_job_value(world, args.steps, m, total_ms * 1e-3)

    check = None
    if rank == 0:
        import oracle

        last = int(src[-1])
        check = bool(np.array_equal(out.cpu().numpy(), oracle.dijkstra_csr_i32(row_ptr, col, w, [last])[0]))

    e2e = None
    if not args.no_e2e:
        # the graph goes to the device once (it is the input of every search);
        # per step: the source index is the whole input, the distances come back
        host_out = torch.empty(n, dtype=torch.int32).pin_memory()
        times = []
        for it, s in enumerate(src[:args.steps + 1]):
            barrier()
            t0 = time.perf_counter()
            graph.search(int(s), out=out, stream=stream)
            host_out.copy_(out, non_blocking=True)
            torch.cuda.current_stream(dev).synchronize()
            if it > 0:
                times.append(time.perf_counter() - t0)
        e2e_total = max_over_ranks(dist, sum(times), dev)
        e2e = {"value": whole_job_value(world, args.steps, m, e2e_total), "unit": "TEPS", "h2d_bytes_per_step": 4,
               "d2h_bytes_per_step": n * 4, "ms_per_step": e2e_total / args.steps * 1e3,
               "graph_h2d_bytes_once": int(row_ptr.nbytes + col.nbytes + w.nbytes)}

    clk = clocks.summary()
    pk = peaks()
    hbm = pk.get("hbm_gbs") or pk.get("hbm_GBps") or 6800.0
    roof = None
    if searches:
        avg = search_ms / searches
        algo_bytes = 8.0 * m + 16.0 * n
        achieved = algo_bytes / (avg * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": None, "kernel": "sssp_grid_kernel", "avg_launch_ms": avg, "launches": searches,
                "algorithmic_bytes_per_launch": algo_bytes,
                "peak_basis": "MEASURED_PEAKS.json hbm_gbs" if pk.get("hbm_gbs") else "fallback 6.8 TB/s",
                "search_share": search_ms / total_ms if total_ms > 0 else None}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle

        t0 = time.perf_counter()
        oracle.dijkstra_csr_i32(row_ptr, col, w, [int(src[0])], threads=1)
        dt = time.perf_counter() - t0
        cpu = {"value": m / dt, "unit": "TEPS", "cores": 1, "kind": "oracle",
               "sample": f"the oracle's binary-heap Dijkstra from one source ({dt:.1f} s, 1 thread)"}

    if rank == 0:
        line = {
            "metric": SSSP_METRIC, "value": value, "unit": "TEPS", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": sssp_config(args, n, m, int(row_ptr.nbytes + col.nbytes + w.nbytes), world),
            "delta_used": delta_used,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels, "clocks": clk, "check_vs_oracle": check, "step_ms": step_ms,
        }
        print(json.dumps(line), flush=True)
    graph.close()
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------------------ out-of-core arm

def ooc_config(args, n: int, K) -> dict:
    """The `config` of the out-of-core lines, shared verbatim by both arms."""
    return {"workload": args.workload, "n": n, "graph": graphgen.describe(args.workload), "algo": "ooc",
            "block": K, "super_rounds": (-(-n // K) if K else None),
            "host": "pinned; restored before each step, outside the timing", "parallelism": "1 GPU"}


def ours_ooc(args, rank, world, local):
    """One host matrix streamed through one GPU: under torchrun only rank 0
    runs it (the other ranks exit without work)."""
    import torch

    import min_graph_gb300 as apsp

    if rank != 0:
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = graphgen.make(args.workload)
    n = w.shape[0]
    src = torch.from_numpy(w)
    host = torch.empty_like(src).pin_memory()
    K = args.block or apsp.ooc_block(n, args.device_bytes or 0)
    for _ in range(args.warmup):
        host.copy_(src)
        apsp.solve_ooc(host, device_bytes=args.device_bytes, block=args.block)
    times = []
    with ClockSampler(local) as clocks:
        for _ in range(args.steps):
            host.copy_(src)  # restore the input (outside the timed region)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            apsp.solve_ooc(host, device_bytes=args.device_bytes, block=args.block)
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps * float(n) ** 3 / total
    check = None
    if rank == 0:
        import oracle

        rows = np.array([0, n // 3, (2 * n) // 3, n - 1], dtype=np.int32)
        got = host.numpy()[rows]
        if w.dtype == np.int32:
            check = bool(np.array_equal(got, oracle.dijkstra_i32(w, rows)))
        else:
            ref = oracle.dijkstra_f32(w, rows)
            fin = np.isfinite(ref)
            check = bool(np.array_equal(np.isfinite(got), fin) and
                         np.all(np.abs(got[fin] - ref[fin]) <= 1e-5 * np.abs(ref[fin])))
    props = torch.cuda.get_device_properties(dev)
    clk = clocks.summary()
    f_max = (clk or {}).get("sm_max_mhz") or peaks().get("sm_max_mhz", 2070.0)
    ops = 1 if w.dtype == np.int32 else 2
    peak_tops = props.multi_processor_count * NOMINAL_INT32_LANES * f_max * 1e6 / ops / 1e12
    nR = -(-n // K) if K else None
    nbytes = n * n * w.itemsize
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_subprocess(args, steps=4, warmup=1)
    line = {
        "metric": OOC_METRIC, "value": value, "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int32" if w.dtype == np.int32 else "f32", "data": "synthetic",
        "config": ooc_config(args, n, K),
        "roofline": {"bound": "alu", "achieved": value / 1e12, "peak": peak_tops, "unit": "Trelax/s",
                     "frac": value / 1e12 / peak_tops, "traffic": None, "kernel": "whole call (minplus_accum_kernel "
                     "and the in-core solver, copies overlapped)"},
        "cpu_baseline": cpu,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": int(nbytes * (nR or 1)),
                "d2h_bytes_per_step": int(nbytes * (nR or 1)),
                "note": "the call itself is end to end: about one crossing of the matrix each way per super-round"},
        "clocks": clk, "check_rows_vs_oracle": check, "step_s": times,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.algo == "ooc":
        if args.impl == "reference":
            reference_arm(args, rank, ooc=True)
        else:
            ours_ooc(args, rank, world, local)
        return
    if args.algo == "sssp":
        if args.impl == "reference":
            reference_sssp(args, rank)
        else:
            ours_sssp(args, rank, world, local)
        return
    if args.algo == "johnson":
        if args.impl == "reference":
            reference_johnson(args, rank)
        else:
            ours_johnson(args, rank, world, local)
        return
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    ours(args, rank, world, local)


if __name__ == "__main__":
    main()
