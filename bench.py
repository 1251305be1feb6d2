#!/usr/bin/env python3
"""RMSNorm forward benchmark: achieved HBM GB/s on one GB300 (and per rank
under torchrun), with the roofline fraction, the end-to-end figure through the
C ABI from host buffers, SM clocks during the timed region, and the fp64 CPU
oracle timed on the host cores as a reported baseline.

A step is one call of the C ABI's rmsnorm_fwd over one [M, N] batch (the
whole forward: row load, sum of squares, rsqrt, rstd store, scale, store).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle as the reference arm

Algorithmic bytes per step: 2*M*N (x read) + 2*M*N (y written) + 2*N (w read)
+ 4*M (rstd written); GB/s = bytes / seconds / 1e9 (the GB/s formula of the
skillmd "RMSNorm Kernel Optimization" page, with the weight and rstd added).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import threading
import time
from typing import NamedTuple

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "RMSNorm fwd achieved HBM GB/s and % of GB300 peak (1 GPU), per M×N×dtype"
DCODE = {"bf16": 0, "fp16": 1, "fp32": 2}  # rmsnorm_dtype_t
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ["common.cuh", "async_copy.cuh", "cluster.cuh", "launch.h", "kernels_warp.cu",
                  "kernels_cta.cu", "kernels_tma.cu", "kernels_cluster.cu", "kernels_generic.cu",
                  "kernels_bwd.cu", "api.cu", "host_pipeline.cu"]


# ---------------------------------------------------------------- host-side helpers

def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=None, help="named workload (default: the 16384x512 bf16 one)")
    p.add_argument("--e2e-steps", type=int, default=400)
    p.add_argument("--chunk-rows", type=int, default=0,
                   help="rows per chunk of the host-buffer path (0: the library's default)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-workload", action="store_true",
                   help="skip the per-workload entries (every named workload, both launch modes)")
    p.add_argument("--variant", default="auto", help="force a kernel variant (ablation)")
    p.add_argument("--lanes-per-row", type=int, default=0)
    p.add_argument("--stages", type=int, default=0)
    p.add_argument("--rows-per-stage", type=int, default=0)
    p.add_argument("--max-ctas", type=int, default=0)
    p.add_argument("--strict-order", action="store_true",
                   help="time without RMSNORM_FLAG_EARLY_LOADS (no overlap between steps)")
    p.add_argument("--blocked", action="store_true", help="contiguous row block per CTA")
    p.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    p.add_argument("--cluster-size", type=int, default=0)
    p.add_argument("--l2-prefetch", type=int, default=0,
                   help="L2 prefetch distance (rmsnorm_options_t.l2_prefetch; 0 = planner's choice)")
    p.add_argument("--prewait-prefetch", type=int, default=0,
                   help="rows/chunks prefetched before the PDL wait "
                        "(rmsnorm_options_t.prewait_prefetch; 0 = planner's choice, -1 = none)")
    p.add_argument("--ablation", action="store_true",
                   help="time a matrix of kernel variants and knobs per workload, one JSON line each")
    p.add_argument("--backward", action="store_true",
                   help="time the backward (dx, dw) on the workload instead of the forward")
    p.add_argument("--launch-only", type=int, default=0, metavar="N",
                   help="no timing: N direct calls of the planned forward over the rotating pool "
                        "(early loads unless --strict-order), for profiler captures of steady-state "
                        "launches; prints the plan")
    return p.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(value: float) -> float:
    """Max of a host float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def whole_job_gbs(bytes_per_rank_step: int, steps: int, world: int, max_seconds: float) -> float:
    """Weak scaling: every rank moves its own batch each step; the job's time is the slowest rank's."""
    return bytes_per_rank_step * steps * world / max_seconds / 1e9


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Source files behind each kernel variant (its translation unit and the headers
# it includes); a traffic figure stays valid while these and the launch plan do.
VARIANT_SOURCES = {
    "warp": ["kernels_warp.cu"], "cta": ["kernels_cta.cu"], "tma": ["kernels_tma.cu"],
    "cluster": ["cluster.cuh", "kernels_cluster.cu"], "generic": ["kernels_generic.cu"],
}
COMMON_SOURCES = ["common.cuh", "async_copy.cuh", "launch.h"]


def kernel_hash(variant: str | None = None) -> str:
    """sha256 prefix of a variant's kernel sources (all sources when None)."""
    names = KERNEL_SOURCES if variant is None else COMMON_SOURCES + VARIANT_SOURCES[variant]
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "memory_bound_normalization_fwd_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PLAN_KEYS = ("variant", "threads", "grid", "lanes_per_row", "vecs_per_lane", "rows_per_stage",
             "stages", "smem_bytes", "cluster_size", "l2_prefetch", "prewait_prefetch")


def load_traffic(workload: str, plan: dict, profiles_dir: str | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of the timed kernel (its `kernel_hash` line matches the
    variant's source hash) with the same launch plan (its `plan` line), else None.
    A summary may hold several entries (one per launch plan, e.g. both launch
    modes); each starts at its own `kernel_hash` line."""
    path = os.path.join(profiles_dir or os.path.join(ROOT, "profiles"), f"traffic_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    want = kernel_hash(plan["variant"])
    for seg in re.split(r"(?=kernel_hash:)", text)[1:]:
        m_hash = re.search(r"kernel_hash:\s*`?([0-9a-f]+)", seg)
        m_bytes = re.search(r"traffic_bytes_per_launch:\s*`?([0-9]+)", seg)
        m_plan = re.search(r"plan:\s*`(\{.*?\})`", seg)
        if not (m_hash and m_bytes and m_plan) or m_hash.group(1) != want:
            continue
        recorded = json.loads(m_plan.group(1))
        if all(recorded.get(k) == plan.get(k) for k in PLAN_KEYS):
            return int(m_bytes.group(1))
    return None


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                [exe, f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[3], parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        # Samples under load: SM clock above idle; the first/last samples bracket the region.
        sm = [r[0] for r in rows]
        busy = [r for r in rows if r[0] >= 0.5 * max(sm)] or rows
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in busy:
            for name, v in zip(names[1:], r[3][1:]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "samples_under_load": len(busy)}


# ---------------------------------------------------------------- timing harness

class Timed(NamedTuple):
    """One timed region: max-over-ranks seconds, steps it ran, seconds per step
    (this rank), clock samples, how it was launched, graph replays it held."""
    max_s: float
    steps: int
    per_step_s: float
    clocks: dict | None
    launch: str
    replays: int


class PoolBench:
    """Inputs resident in HBM in a rotating pool of buffer sets (>= 3x L2, so no
    step reads another step's lines from L2), steps issued as a CUDA graph of
    C-ABI calls, timed with CUDA events on the launching stream."""

    def __init__(self, wl, x_bits, w_bits, dev):
        import torch
        from memory_bound_normalization_fwd_gb300 import binding as B
        from memory_bound_normalization_fwd_gb300 import workloads as W
        self.wl, self.dev = wl, dev
        self.dcode = DCODE[wl.dtype]
        self.x_host = W.to_torch(x_bits, wl.dtype)
        self.w_dev = W.to_torch(w_bits, wl.dtype).to(dev)
        self.set_bytes = 2 * W.ELEM_BYTES[wl.dtype] * wl.M * wl.N + 4 * wl.M
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.pool = max(2, -(-3 * self.l2 // self.set_bytes))
        self.xs = [self.x_host.to(dev) for _ in range(self.pool)]
        self.ys = [torch.empty_like(self.xs[0]) for _ in range(self.pool)]
        self.rs = [torch.empty(wl.M, dtype=torch.float32, device=dev) for _ in range(self.pool)]
        self.stream = torch.cuda.Stream(dev)

    def _graph_time(self, step, K: int, Wm: int, clock_gpu=None, min_ms: float = 2.0):
        """Time K steps as the GPU runs them, at any K.

        Exactly K calls (rotating through the pool) are captured into one CUDA
        graph (several such graphs over successive slices of the pool when it
        holds more than K buffer sets). After Wm untimed direct calls and untimed
        replays, the timed region is R back-to-back replays between two CUDA
        events on the launching stream, R chosen (the same on every rank) so
        that the region lasts at least ``min_ms``; the per-step time is the
        region's time over R*K. A timed region of direct host calls would time
        the host's launch rate instead of the kernels."""
        import torch
        stream = self.stream
        with torch.cuda.stream(stream):
            for k in range(max(3, min(Wm, 64))):
                step(k)
        stream.synchronize()
        # When the pool holds more buffer sets than K, one graph of K calls would
        # cycle through only K of them (and a small workload would then stay in
        # L2): graphs g = 0, 1, ... each take the next K sets, and replays go
        # round-robin over them, so consecutive replays still walk the whole pool.
        n_graphs = max(1, -(-self.pool // K))
        graphs = []
        for g in range(n_graphs):
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
                for k in range(K):
                    step(g * K + k)
            graphs.append(graph)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for r in range(max(n_graphs, -(-Wm // K))):
                graphs[r % n_graphs].replay()
        torch.cuda.synchronize()
        # Replays per timed region, from one timed probe replay (max over ranks,
        # so every rank runs the same count), rounded up to whole pool cycles.
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            graphs[0].replay()
            b.record(stream)
        torch.cuda.synchronize()
        reps = int(max_over_ranks(float(max(1, -(-min_ms // max(a.elapsed_time(b), 1e-3))))))
        reps = -(-reps // n_graphs) * n_graphs
        barrier()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(clock_gpu) if clock_gpu is not None else None
        if sampler:
            sampler.__enter__()
        try:
            torch.cuda.synchronize()
            barrier()
            with torch.cuda.stream(stream):
                start.record(stream)
                for r in range(reps):
                    graphs[r % n_graphs].replay()
                end.record(stream)
            torch.cuda.synchronize()
            barrier()
        finally:
            if sampler:
                sampler.__exit__(None, None, None)
        ms = start.elapsed_time(end)
        steps = reps * K
        launch = (f"CUDA graph of {K} ABI calls (rotating the pool"
                  + (f"; {n_graphs} such graphs over successive pool slices, replayed in turn"
                     if n_graphs > 1 else "")
                  + f"), {reps} replays back to back in the timed region ({steps} steps)")
        return Timed(max_over_ranks(ms / 1e3), steps, ms / 1e3 / steps,
                     sampler.summary() if sampler else None, launch, reps)

    def trials(self, opts, n_trials: int = 20, min_ms: float = 2.0):
        """GB/s of `n_trials` separately timed windows (each at least `min_ms` of
        graph replays, CUDA events around each window), after the main timed
        region: (median, min, max, steps per window)."""
        import statistics as st
        import torch
        from memory_bound_normalization_fwd_gb300 import binding as B
        wl, stream, sh = self.wl, self.stream, self.stream.cuda_stream

        def step(k: int):
            i = k % self.pool
            rc = B.rmsnorm_fwd_ex(self.xs[i].data_ptr(), self.w_dev.data_ptr(), self.ys[i].data_ptr(),
                                  self.rs[i].data_ptr(), wl.M, wl.N, wl.eps, wl.offset, self.dcode,
                                  opts, sh)
            if rc != 0:
                raise RuntimeError(B.rmsnorm_last_error())
        per_graph = self.pool * max(1, 384 // self.pool)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for k in range(per_graph):
                step(k)
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        # replays per window: enough for min_ms, from a timed probe replay
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize()
        reps = max(1, int(min_ms / max(a.elapsed_time(b), 1e-3)) + 1)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_trials + 1)]
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for t in range(n_trials):
                for _ in range(reps):
                    graph.replay()
                evs[t + 1].record(stream)
        torch.cuda.synchronize()
        steps = reps * per_graph
        gbs = [wl.algorithmic_bytes * steps / (evs[t].elapsed_time(evs[t + 1]) / 1e3) / 1e9
               for t in range(n_trials)]
        return st.median(gbs), min(gbs), max(gbs), steps

    def timed(self, opts, K: int, Wm: int, clock_gpu=None, min_ms: float = 2.0) -> Timed:
        """K steps of rmsnorm_fwd_ex with `opts`, timed as `_graph_time` times them."""
        from memory_bound_normalization_fwd_gb300 import binding as B
        wl, sh = self.wl, self.stream.cuda_stream

        def step(k: int):
            i = k % self.pool
            rc = B.rmsnorm_fwd_ex(self.xs[i].data_ptr(), self.w_dev.data_ptr(), self.ys[i].data_ptr(),
                                  self.rs[i].data_ptr(), wl.M, wl.N, wl.eps, wl.offset, self.dcode,
                                  opts, sh)
            if rc != 0:
                raise RuntimeError(B.rmsnorm_last_error())
        return self._graph_time(step, K, Wm, clock_gpu, min_ms)

    def copy_timed(self, K: int, Wm: int, min_ms: float = 2.0) -> Timed:
        """A plain device copy of x into y at the same size, same pool, same graph shape."""
        def step(k: int):
            i = k % self.pool
            self.ys[i].copy_(self.xs[i])
        return self._graph_time(step, K, Wm, None, min_ms)


def agree(a_bits, b_bits, dtype: str) -> bool:
    """Two runs' outputs are the same bits, or, where the two launches reduce a
    row in a different order, within one unit in the last place (16-bit
    formats) or 64 (fp32, whose last place is 2^13 times finer)."""
    import numpy as np
    if np.array_equal(a_bits, b_bits):
        return True
    wide = dtype == "fp32"
    sign = np.int64(0x80000000 if wide else 0x8000)

    def ordinal(b):
        b = b.astype(np.int64)
        return np.where(b & sign, -(b & (sign - 1)), b)
    return int(np.abs(ordinal(a_bits) - ordinal(b_bits)).max()) <= (64 if wide else 1)


# ---------------------------------------------------------------- CPU oracle legs

def run_oracle_threaded(x, w, wl, rows: int, threads: int):
    """The oracle over the first `rows` rows, split into contiguous blocks over
    `threads` Python threads (ctypes releases the GIL in the C call). Returns seconds."""
    import numpy as np
    import oracle
    y = np.empty((rows, wl.N), dtype=oracle.bits_dtype(wl.dtype))
    r = np.empty(rows, dtype=np.float64)
    xs = np.ascontiguousarray(x[:rows])
    bounds = [rows * i // threads for i in range(threads + 1)]
    oracle.lib()
    ts = [threading.Thread(target=oracle.rmsnorm_fwd_into,
                           args=(xs, w, y, r, wl.eps, wl.offset, wl.dtype, bounds[i], bounds[i + 1]))
          for i in range(threads) if bounds[i + 1] > bounds[i]]
    t0 = time.perf_counter()
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return time.perf_counter() - t0


def cpu_baseline(x, w, wl, repeats: int = 3):
    cores = os.cpu_count() or 1
    secs = [run_oracle_threaded(x, w, wl, wl.M, cores) for _ in range(repeats)]
    t = statistics.median(secs)
    # One thread, on a row sample of about a tenth of a second of work.
    probe = min(wl.M, max(1, 256 * 512 // wl.N))
    t1 = run_oracle_threaded(x, w, wl, probe, 1)
    rows1 = int(min(wl.M, max(probe, probe * 0.1 / max(t1, 1e-6))))
    t1 = statistics.median(run_oracle_threaded(x, w, wl, rows1, 1) for _ in range(repeats))
    eb = 4 if wl.dtype == "fp32" else 2
    bytes1 = 2 * eb * rows1 * wl.N + eb * wl.N + 4 * rows1
    return {"value": round(wl.algorithmic_bytes / t / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "single_thread": round(bytes1 / t1 / 1e9, 4),
            "sample": f"whole {wl.M}x{wl.N} {wl.dtype} batch, {repeats} runs, median "
                      f"({t:.3f} s each, fp64 C oracle, {cores} threads over row blocks); "
                      f"single_thread: {rows1} rows on one thread, median of {repeats}"}


# ---------------------------------------------------------------- our arm

def bench_ours(args, wl, rank, world, local_rank):
    import numpy as np
    import torch
    from memory_bound_normalization_fwd_gb300 import binding as B
    from memory_bound_normalization_fwd_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dcode = DCODE[wl.dtype]
    eb = W.ELEM_BYTES[wl.dtype]
    x_bits, w_bits = W.generate(wl)
    pb = PoolBench(wl, x_bits, w_bits, dev)
    x_host, w_dev, xs, ys, rs = pb.x_host, pb.w_dev, pb.xs, pb.ys, pb.rs
    pool, set_bytes, l2, stream, sh = pb.pool, pb.set_bytes, pb.l2, pb.stream, pb.stream.cuda_stream
    timed = pb.timed

    def make_opts(early: bool, early_weights: bool = False):
        return B.make_options(variant=args.variant, lanes_per_row=args.lanes_per_row,
                              stages=args.stages, rows_per_stage=args.rows_per_stage,
                              max_ctas=args.max_ctas, early_loads=early, blocked=args.blocked,
                              pdl=not args.no_pdl, cluster_size=args.cluster_size,
                              early_weights=early_weights, l2_prefetch=args.l2_prefetch,
                              prewait_prefetch=args.prewait_prefetch)

    # Main measurement. The steps are independent batches (x and w are written
    # by no step), which meets the precondition of RMSNORM_FLAG_EARLY_LOADS:
    # step k+1 may start loading while step k finishes; every store stays in
    # stream order. --strict-order measures without the flag.
    early = not args.strict_order
    opts = make_opts(early)
    plan = B.rmsnorm_plan_info(wl.M, wl.N, dcode, xs[0].data_ptr(), w_dev.data_ptr(),
                               ys[0].data_ptr(), opts)
    K, Wm = args.steps, max(3, args.warmup)
    # The timed region lasts at least half a second, so that the clock sampler
    # sees it under load.
    main = timed(opts, K, Wm, torch.cuda.current_device() if world == 1 else local_rank,
                 min_ms=500.0)
    value = whole_job_gbs(wl.algorithmic_bytes, main.steps, world, main.max_s)
    per_launch_s = main.per_step_s

    # The same workload under strict stream order (every access waits for the
    # previous step): the figure that applies to a dependent chain of layers,
    # where each launch reads the previous kernel's output.
    strict = None
    if early:
        sopts = make_opts(False)
        splan = B.rmsnorm_plan_info(wl.M, wl.N, dcode, xs[0].data_ptr(), w_dev.data_ptr(),
                                    ys[0].data_ptr(), sopts)
        # Weights resident (as in inference), x the previous step's output: the
        # strict chain with only w read early.
        tw = timed(make_opts(False, True), K, Wm, min_ms=100.0)
        ts = timed(sopts, K, Wm, min_ms=100.0)
        strict = {"value": round(whole_job_gbs(wl.algorithmic_bytes, ts.steps, world, ts.max_s), 2),
                  "unit": "GB/s", "steps": ts.steps, "launch": ts.launch,
                  "frac": None, "plan": splan,
                  "early_weights": round(whole_job_gbs(wl.algorithmic_bytes, tw.steps, world,
                                                       tw.max_s), 2),
                  "note": "no RMSNORM_FLAG_EARLY_LOADS: each launch reads x only after the "
                          "previous step completes (the case of a dependent chain of layers); "
                          "early_weights: the same with RMSNORM_FLAG_EARLY_WEIGHTS (w read "
                          "before the wait, x after)"}
    # Twenty separately timed windows of the headline configuration (after the
    # timed region above, which alone gives `value`): median, min, max.
    t_med, t_min, t_max, t_steps = pb.trials(make_opts(early))
    opts = make_opts(False)  # the end-to-end leg keeps strict order (copies precede each call)

    # End to end through the public host-buffer call: per step, rmsnorm_fwd_host
    # moves pinned host x to the device in chunks, normalises each chunk in a
    # device ring and copies y and rstd back to pinned host memory (the two
    # copy directions overlapping), all inside the timed region.
    x_pin = x_host.pin_memory()
    y_pin = torch.empty(x_host.shape, dtype=x_host.dtype).pin_memory()
    r_pin = torch.empty(wl.M, dtype=torch.float32).pin_memory()
    Ke = max(20, min(args.e2e_steps, K))
    ws_bytes = B.rmsnorm_fwd_host_workspace_size(wl.M, wl.N, dcode, args.chunk_rows)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def e2e_step():
        rc = B.rmsnorm_fwd_host(x_pin.data_ptr(), w_dev.data_ptr(), y_pin.data_ptr(),
                                r_pin.data_ptr(), wl.M, wl.N, wl.eps, wl.offset, dcode,
                                args.chunk_rows, ws.data_ptr(), ws_bytes, opts, sh)
        if rc != 0:
            raise RuntimeError(B.rmsnorm_last_error())

    def time_steps(step, n):
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
        torch.cuda.synchronize()
        barrier()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(n):
                step()
            end.record(stream)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(start.elapsed_time(end) / 1e3)

    e2e_s = time_steps(e2e_step, Ke)
    # Same answer as the device-resident run under strict order, the last one
    # timed on the pool (pool set 1 holds the same x).
    j = 1 % pool
    if not agree(W.from_torch(y_pin), W.from_torch(ys[j]), wl.dtype):
        raise RuntimeError("end-to-end output differs from the device-resident output")

    # For comparison: the same bytes moved serially on one stream (x in, the
    # device call, y and rstd out), as a caller without the host path would.
    x_e, y_e, r_e = xs[0], ys[0], rs[0]

    def serial_step():
        x_e.copy_(x_pin, non_blocking=True)
        rc = B.rmsnorm_fwd_ex(x_e.data_ptr(), w_dev.data_ptr(), y_e.data_ptr(), r_e.data_ptr(),
                              wl.M, wl.N, wl.eps, wl.offset, dcode, opts, sh)
        if rc != 0:
            raise RuntimeError(B.rmsnorm_last_error())
        y_pin.copy_(y_e, non_blocking=True)
        r_pin.copy_(r_e, non_blocking=True)

    serial_s = time_steps(serial_step, Ke)

    # The same call with RMSNORM_FLAG_HOST_DIRECT: one kernel reads x and writes
    # y and rstd in the pinned host buffers itself (no ring, no copy engines).
    dopts = B.make_options(host_direct=True)

    def direct_step():
        rc = B.rmsnorm_fwd_host(x_pin.data_ptr(), w_dev.data_ptr(), y_pin.data_ptr(),
                                r_pin.data_ptr(), wl.M, wl.N, wl.eps, wl.offset, dcode, 0, 0, 0,
                                dopts, sh)
        if rc != 0:
            raise RuntimeError(B.rmsnorm_last_error())

    direct_s = time_steps(direct_step, Ke)
    if not agree(W.from_torch(y_pin), W.from_torch(ys[j]), wl.dtype):
        raise RuntimeError("host-direct output differs from the device-resident output")

    # Context: a plain device copy of x into y (torch) of the same size, same pool
    # and graph shape: the ceiling a kernel moving these bytes meets at this size.
    # (Last, since it overwrites the pool's y buffers.)
    tc = pb.copy_timed(K, 3, min_ms=100.0)
    copy_gbs = 2 * pb.x_host.element_size() * wl.M * wl.N * tc.steps / tc.max_s / 1e9
    ring_rows = min(wl.M, args.chunk_rows or max(1, (4 << 20) // (eb * wl.N)))

    peak, peak_src = load_peaks()
    achieved = wl.algorithmic_bytes / per_launch_s / 1e9
    traffic = load_traffic(wl.name, plan)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": round(main.max_s * 1e3 / main.steps, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded torch CPU generator; see workloads.py)",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "eps": wl.eps, "offset": wl.offset,
                   "x": f"N(0,{wl.x_std}^2)" + (f" + {wl.outlier_p} outliers N(0,{wl.outlier_std}^2)"
                                                if wl.outlier_p else ""),
                   "bytes_per_step": wl.algorithmic_bytes,
                   "l2": f"rotating pool of {pool} buffer sets ({pool * set_bytes / 1e6:.0f} MB) "
                         f"> 3x L2 ({l2 / 1e6:.0f} MB); no flush needed",
                   "launch": main.launch,
                   "launch_order": ("early loads (RMSNORM_FLAG_EARLY_LOADS): steps are independent "
                                    "batches, so step k+1 may start loading x while step k "
                                    "finishes; all stores stay in stream order"
                                    + ("; this plan uses the pre-wait L2 prefetch instead (x read "
                                       "after the wait, its first chunks asked into L2 before it)"
                                       if plan.get("prewait_prefetch") else "")) if early
                                   else "strict stream order",
                   "plan": plan},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured"
                     else "fallback 6.8 TB/s", "algorithmic_bytes": wl.algorithmic_bytes,
                     "kernel_hash": kernel_hash(plan["variant"])},
        "e2e": {"value": round(whole_job_gbs(wl.algorithmic_bytes, Ke, world, e2e_s), 2),
                "unit": "GB/s", "h2d_bytes_per_step": eb * wl.M * wl.N,
                "d2h_bytes_per_step": eb * wl.M * wl.N + 4 * wl.M, "steps": Ke,
                "ms_per_step": round(e2e_s * 1e3 / Ke, 4),
                "path": (f"rmsnorm_fwd_host: pinned host x -> device ring in chunks of {ring_rows} "
                         f"rows (4 slots) on a copy-in stream, kernel in place per chunk, y and rstd -> pinned host on "
                         f"a second stream, copy directions overlapping"),
                "serial_one_stream": round(whole_job_gbs(wl.algorithmic_bytes, Ke, world,
                                                         serial_s), 2),
                "host_direct": round(whole_job_gbs(wl.algorithmic_bytes, Ke, world, direct_s), 2)},
        "context": {"device_copy_same_size_gbs": round(copy_gbs, 1),
                    "note": "torch copy of x into y, same pool and graph shape (x and y bytes only)"},
        "trials": {"n": 20, "steps_each": t_steps, "median": round(t_med, 2), "min": round(t_min, 2),
                   "max": round(t_max, 2), "unit": "GB/s",
                   "note": "separately timed windows after the timed region; value is the timed region"},
        "timed_region": {"steps": main.steps, "graph_replays": main.replays,
                         "seconds": round(main.max_s, 6),
                         "note": f"the --steps {K} ABI calls captured as a CUDA graph and "
                                 f"replayed {main.replays} times back to back between CUDA events "
                                 "(see config.launch); ms_per_step = region time / steps run"},
        "gpu_launches": main.steps,  # one kernel per rmsnorm_fwd_ex call
        "clocks": main.clocks,
    }
    if strict is not None:
        strict["frac"] = round(strict["value"] / peak, 4)
        line["strict_order"] = strict
    if world == 1 and not args.no_per_workload:
        del pb, xs, ys, rs
        torch.cuda.empty_cache()
        line["per_workload"] = per_workload(args, dev, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x_bits, w_bits, wl)
    return line


def per_workload(args, dev, peak: float) -> dict:
    """Every named workload (the metric is per M x N x dtype), in both launch
    modes, timed as the headline is (a CUDA graph of ABI calls over a rotating
    pool >= 3x L2, replayed back to back, here for at least 100 ms) except that
    the graphs hold a fixed 200 calls whatever --steps is: these entries
    describe the workloads, and a short graph would add its launch boundary
    every few steps. Each
    entry: GB/s, fraction of the peak, the plan, and the DRAM traffic per
    launch from the committed ncu summary when it matches the current kernel
    sources and plan (else null)."""
    import torch
    from memory_bound_normalization_fwd_gb300 import binding as B
    from memory_bound_normalization_fwd_gb300 import workloads as W
    out = {}
    for name, wl in W.WORKLOADS.items():
        x_bits, w_bits = W.generate(wl)
        pb = PoolBench(wl, x_bits, w_bits, dev)
        K = 200
        entry = {"M": wl.M, "N": wl.N, "dtype": wl.dtype, "bytes_per_step": wl.algorithmic_bytes,
                 "pool_sets": pb.pool}
        for mode, early in (("early_loads", True), ("strict", False)):
            opts = B.make_options(early_loads=early)
            plan = B.rmsnorm_plan_info(wl.M, wl.N, pb.dcode, pb.xs[0].data_ptr(),
                                       pb.w_dev.data_ptr(), pb.ys[0].data_ptr(), opts)
            t = pb.timed(opts, K, 3, min_ms=100.0)
            gbs = wl.algorithmic_bytes / t.per_step_s / 1e9
            entry[mode] = {"gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                           "us_per_step": round(t.per_step_s * 1e6, 3), "steps": t.steps,
                           "graph_calls": K, "plan": plan,
                           "traffic": load_traffic(name, plan)}
        out[name] = entry
        del pb
        torch.cuda.empty_cache()
    return out


def launch_only_backward(args, wl) -> dict:
    """N direct rmsnorm_bwd calls over a rotating pool of x, dy and dx sets
    (early loads unless --strict-order), the plan bench_backward times;
    nothing is timed."""
    import torch
    from memory_bound_normalization_fwd_gb300 import binding as B
    from memory_bound_normalization_fwd_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    dcode = DCODE[wl.dtype]
    x_bits, w_bits = W.generate(wl)
    dy_bits, _ = W.generate(W.custom(wl.M, wl.N, wl.dtype, seed=99))
    x0, dy0 = W.to_torch(x_bits, wl.dtype).to(dev), W.to_torch(dy_bits, wl.dtype).to(dev)
    w = W.to_torch(w_bits, wl.dtype).to(dev)
    r0 = torch.empty(wl.M, dtype=torch.float32, device=dev)
    B.fwd(x0, w, eps=wl.eps, offset=wl.offset, y=torch.empty_like(x0), rstd=r0)
    eb = W.ELEM_BYTES[wl.dtype]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool = max(2, -(-3 * l2 // (3 * eb * wl.M * wl.N + 4 * wl.M)))
    xs = [x0.clone() for _ in range(pool)]
    dys = [dy0.clone() for _ in range(pool)]
    dxs = [torch.empty_like(x0) for _ in range(pool)]
    dw = torch.empty(wl.N, dtype=torch.float32, device=dev)
    opts = B.make_options(variant=args.variant, max_ctas=args.max_ctas,
                          lanes_per_row=args.lanes_per_row, rows_per_stage=args.rows_per_stage,
                          stages=args.stages, early_loads=not args.strict_order)
    nbytes = B.rmsnorm_bwd_workspace_size(wl.M, wl.N, dcode, opts)
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream().cuda_stream
    for k in range(args.launch_only):
        i = k % pool
        rc = B.rmsnorm_bwd(xs[i].data_ptr(), w.data_ptr(), r0.data_ptr(), dys[i].data_ptr(),
                           dxs[i].data_ptr(), dw.data_ptr(), wl.M, wl.N, wl.offset, dcode,
                           ws.data_ptr(), ws.numel() * 4, opts, s)
        if rc != 0:
            raise RuntimeError(B.rmsnorm_last_error())
    torch.cuda.synchronize()
    return {"launch_only_backward": wl.name, "launches": args.launch_only, "pool_sets": pool,
            "launch_order": "strict" if args.strict_order else "early loads",
            "plan": B.rmsnorm_bwd_plan_info(wl.M, wl.N, dcode, opts)}


def launch_only(args, wl) -> dict:
    """N direct rmsnorm_fwd_ex calls over the rotating pool, the plan bench_ours
    times for this workload and launch mode; nothing is timed."""
    import torch
    from memory_bound_normalization_fwd_gb300 import binding as B
    from memory_bound_normalization_fwd_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    x_bits, w_bits = W.generate(wl)
    pb = PoolBench(wl, x_bits, w_bits, dev)
    opts = B.make_options(variant=args.variant, lanes_per_row=args.lanes_per_row,
                          stages=args.stages, rows_per_stage=args.rows_per_stage,
                          max_ctas=args.max_ctas, early_loads=not args.strict_order,
                          blocked=args.blocked, pdl=not args.no_pdl,
                          cluster_size=args.cluster_size, l2_prefetch=args.l2_prefetch,
                          prewait_prefetch=args.prewait_prefetch)
    plan = B.rmsnorm_plan_info(wl.M, wl.N, pb.dcode, pb.xs[0].data_ptr(), pb.w_dev.data_ptr(),
                               pb.ys[0].data_ptr(), opts)
    with torch.cuda.stream(pb.stream):
        for k in range(args.launch_only):
            i = k % pb.pool
            rc = B.rmsnorm_fwd_ex(pb.xs[i].data_ptr(), pb.w_dev.data_ptr(), pb.ys[i].data_ptr(),
                                  pb.rs[i].data_ptr(), wl.M, wl.N, wl.eps, wl.offset, pb.dcode,
                                  opts, pb.stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(B.rmsnorm_last_error())
    torch.cuda.synchronize()
    return {"launch_only": wl.name, "launches": args.launch_only, "pool_sets": pb.pool,
            "launch_order": "strict" if args.strict_order else "early loads", "plan": plan,
            "kernel_hash": kernel_hash(plan["variant"])}


# ---------------------------------------------------------------- ablation matrix

def ablation_configs(wl):
    """Kernel variants and knobs to compare on one workload (the pages' knobs:
    TMA staging on or off, prefetch depth, rows per warp, registers and
    occupancy; plus launch overlap, the pre-wait prefetch and row order)."""
    eb = 4 if wl.dtype == "fp32" else 2
    nvec, row = wl.N * eb // 16, eb * wl.N
    cfgs = [dict(), dict(early_loads=True), dict(early_weights=True), dict(pdl=False),
            dict(blocked=True)]
    # Pre-wait L2 prefetch off (the plans the planner takes without it), and
    # its depth per kernel.
    cfgs += [dict(prewait_prefetch=-1), dict(early_loads=True, prewait_prefetch=-1)]
    for PW in (1, 2, 3):
        cfgs.append(dict(variant="tma", prewait_prefetch=PW))
        if nvec <= 128:
            cfgs.append(dict(variant="warp", prewait_prefetch=PW))
    if nvec <= 128:
        for G in (8, 16, 32):
            for D in (1, 2, 4):
                if (nvec + G - 1) // G <= 4:
                    cfgs.append(dict(variant="warp", lanes_per_row=G, stages=D))
    for T in (64, 128, 256, 512, 1024):
        if T // 2 < nvec <= 4 * T:
            cfgs.append(dict(variant="cta", lanes_per_row=T))
    for kb in (8, 16, 32):
        R = max(1, kb * 1024 // row)
        for S in (1, 2, 3, 4):
            if S * R * row <= 200 * 1024:
                for early in (False, True):
                    cfgs.append(dict(variant="tma", rows_per_stage=R, stages=S, early_loads=early))
    for early in (False, True):  # TMA stores: y leaves by cp.async.bulk from the stage
        cfgs.append(dict(variant="tma", bulk_store=True, early_loads=early))
    if nvec >= 512:
        for C in (2, 4):
            cfgs.append(dict(variant="cluster", cluster_size=C, early_loads=True))
    cfgs.append(dict(variant="generic"))
    return cfgs


def run_ablation(args, names):
    import torch
    from memory_bound_normalization_fwd_gb300 import binding as B
    from memory_bound_normalization_fwd_gb300 import workloads as W
    peak, _ = load_peaks()
    dev = torch.device("cuda", 0)
    for name in names:
        wl = W.get(name)
        x_bits, w_bits = W.generate(wl)
        pb = PoolBench(wl, x_bits, w_bits, dev)
        K = args.steps if wl.M * wl.N < (1 << 26) else max(200, args.steps // 20)
        t = pb.copy_timed(K, 3, min_ms=100.0)
        print(json.dumps({"ablation": name, "config": "device copy x -> y (torch)",
                          "gbs": round(2 * pb.x_host.element_size() * wl.M * wl.N * t.steps
                                       / t.max_s / 1e9, 1)}), flush=True)
        for cfg in ablation_configs(wl):
            opts = B.make_options(**cfg)
            try:
                plan = B.rmsnorm_plan_info(wl.M, wl.N, pb.dcode, pb.xs[0].data_ptr(),
                                           pb.w_dev.data_ptr(), pb.ys[0].data_ptr(), opts)
            except B.RMSNormError:
                continue
            t = pb.timed(opts, K, 3, min_ms=100.0)
            gbs = wl.algorithmic_bytes * t.steps / t.max_s / 1e9
            print(json.dumps({"ablation": name, "config": cfg, "gbs": round(gbs, 1),
                              "frac": round(gbs / peak, 4), "plan": plan}), flush=True)
        del pb
        torch.cuda.empty_cache()


# ---------------------------------------------------------------- backward

def bench_backward(args, wl):
    """Throughput of rmsnorm_bwd on the workload: algorithmic bytes per step =
    x, dy read and dx written (3 e M N, e bytes per element) + rstd read (4 M)
    + w read (e N) + dw written (4 N); the dw partials in the workspace are not
    counted."""
    import torch
    from memory_bound_normalization_fwd_gb300 import binding as B
    from memory_bound_normalization_fwd_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    dcode = DCODE[wl.dtype]
    eb = W.ELEM_BYTES[wl.dtype]
    x_bits, w_bits = W.generate(wl)
    dy_bits, _ = W.generate(W.custom(wl.M, wl.N, wl.dtype, seed=99))
    x0, dy0 = W.to_torch(x_bits, wl.dtype).to(dev), W.to_torch(dy_bits, wl.dtype).to(dev)
    w = W.to_torch(w_bits, wl.dtype).to(dev)
    r0 = torch.empty(wl.M, dtype=torch.float32, device=dev)
    B.fwd(x0, w, eps=wl.eps, offset=wl.offset, y=torch.empty_like(x0), rstd=r0)
    set_bytes = 3 * eb * wl.M * wl.N + 4 * wl.M
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool = max(2, -(-3 * l2 // set_bytes))
    xs = [x0.clone() for _ in range(pool)]
    dys = [dy0.clone() for _ in range(pool)]
    dxs = [torch.empty_like(x0) for _ in range(pool)]
    rs = [r0.clone() for _ in range(pool)]
    dw = torch.empty(wl.N, dtype=torch.float32, device=dev)

    def make(early):
        return B.make_options(variant=args.variant, max_ctas=args.max_ctas,
                              lanes_per_row=args.lanes_per_row, l2_prefetch=args.l2_prefetch,
                              prewait_prefetch=args.prewait_prefetch,
                              rows_per_stage=args.rows_per_stage, stages=args.stages,
                              early_loads=early)
    nbytes = B.rmsnorm_bwd_workspace_size(wl.M, wl.N, dcode, make(False))
    ws = torch.empty(nbytes // 4 + 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    sh = stream.cuda_stream
    step_bytes = 3 * eb * wl.M * wl.N + 4 * wl.M + eb * wl.N + 4 * wl.N
    peak, _ = load_peaks()

    def run(opts):
        def step(k):
            i = k % pool
            rc = B.rmsnorm_bwd(xs[i].data_ptr(), w.data_ptr(), rs[i].data_ptr(), dys[i].data_ptr(),
                               dxs[i].data_ptr(), dw.data_ptr(), wl.M, wl.N, wl.offset, dcode,
                               ws.data_ptr(), ws.numel() * 4, opts, sh)
            if rc != 0:
                raise RuntimeError(B.rmsnorm_last_error())

        with torch.cuda.stream(stream):
            for k in range(8):
                step(k)
        torch.cuda.synchronize()
        per = pool * max(1, 128 // pool)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for k in range(per):
                step(k)
        K = max(per, args.steps // per * per)
        with torch.cuda.stream(stream):
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(K // per):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        sec = a.elapsed_time(b) / 1e3
        return step_bytes * K / sec / 1e9, K, sec

    gbs, K, sec = run(make(False))
    gbs_e, _, sec_e = run(make(True))
    return {"backward": wl.name, "value": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak, 4),
            "steps": K, "ms_per_step": round(sec * 1e3 / K, 5), "bytes_per_step": step_bytes,
            "early_loads": {"value": round(gbs_e, 1), "frac": round(gbs_e / peak, 4),
                            "ms_per_step": round(sec_e * 1e3 / K, 5),
                            "note": "RMSNORM_FLAG_EARLY_LOADS: x, w and rstd of the first rows read "
                                    "before the previous step completes (steps are independent)"},
            "workspace_bytes": nbytes, "variant": args.variant, "max_ctas": args.max_ctas,
            "rows_per_stage": args.rows_per_stage, "stages": args.stages,
            "plan": B.rmsnorm_bwd_plan_info(wl.M, wl.N, dcode, make(False)),
            "l2": f"rotating pool of {pool} sets ({pool * set_bytes / 1e6:.0f} MB) > 3x L2"}


# ---------------------------------------------------------------- reference arm (the oracle)

def bench_reference(args, wl):
    from memory_bound_normalization_fwd_gb300 import workloads as W
    cores = os.cpu_count() or 1
    x, w = W.generate(wl)
    # Calibrate the rate, then size each step so the whole run takes about a minute.
    probe = min(wl.M, 64 * cores)
    t = run_oracle_threaded(x, w, wl, probe, cores)
    rows_per_s = probe / max(t, 1e-6)
    total = args.steps + max(3, args.warmup)
    rows = int(max(cores, min(wl.M, rows_per_s * 60.0 / total)))
    eb = 4 if wl.dtype == "fp32" else 2
    step_bytes = 2 * eb * rows * wl.N + eb * wl.N + 4 * rows
    for _ in range(max(3, args.warmup) if total * rows / rows_per_s < 120 else 3):
        run_oracle_threaded(x, w, wl, rows, cores)
    secs = sum(run_oracle_threaded(x, w, wl, rows, cores) for _ in range(args.steps))
    value = step_bytes * args.steps / secs / 1e9
    sample = f"first {rows} of {wl.M} rows per step ({wl.N} columns, {wl.dtype}), fp64 C oracle"
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(secs * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic (seeded torch CPU generator; see workloads.py)",
        "config": {"workload": wl.name, "M": wl.M, "N": wl.N, "eps": wl.eps, "offset": wl.offset,
                   "bytes_per_step": step_bytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    from memory_bound_normalization_fwd_gb300 import workloads as W
    wl = W.get(args.workload or W.BENCH_WORKLOAD)
    rank, world, local_rank = dist_env()

    if args.ablation:
        run_ablation(args, [args.workload] if args.workload else list(W.WORKLOADS))
        return 0

    if args.launch_only:
        fn = launch_only_backward if args.backward else launch_only
        print(json.dumps(fn(args, wl)), flush=True)
        return 0

    if args.backward:
        for name in ([args.workload] if args.workload else list(W.WORKLOADS)):
            print(json.dumps(bench_backward(args, W.get(name))), flush=True)
        return 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(bench_reference(args, wl)), flush=True)
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    try:
        line = bench_ours(args, wl, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
