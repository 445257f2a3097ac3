"""Benchmark of the quantized projection path on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one fused gate/up SwiGLU projection of the 8B-shaped layer
(X fp16 [2048, 4096], Wg and Wu Q4_0 [14336, 4096], Y fp16 [2048, 14336]),
the workload the headline metric is quoted on.  Inputs are resident in HBM
and rotate through 4 distinct copies (332 MB > L2) so each step reads cold
weights.  Prints one JSON line (rank 0).

Extra keys: "roofline" of the SwiGLU kernel (tensor bound, against the
measured dense bf16/fp16 peak), "m1" (the same weights at M = 1 through the
streaming GEMV, GB/s against measured HBM bandwidth), "e2e" (the public API
with pinned host X and Y copied every step), "cpu_baseline" (the CPU oracle
on a bounded row sample), "clocks" (nvidia-smi sampled during the timed
region) and "gpu_launches".

--impl reference times the CPU oracle (the only reference implementation
of this path; the pages ship no runnable code) on bounded row samples of the
same workload.

Multi-GPU: the projection has no exchange step, so N ranks run N independent
replicas (weak scaling); the only collectives are the timing barrier and the
max-over-ranks reduction.
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
sys.path.insert(0, ROOT)

METRIC = "quantized prefill GEMM TFLOP/s & % roofline (8B SwiGLU, M=2048); M=1 GB/s"
WORKLOAD = "8b_swiglu_q4_0_m2048"
M_, N_, K_ = 2048, 14336, 4096
ROTATE = 4
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["swiglu_block_quantized_gb300/csrc/tc_proj.cuh",
                  "swiglu_block_quantized_gb300/csrc/codec.cuh",
                  "swiglu_block_quantized_gb300/csrc/common.cuh"]
GEMV_SOURCES = ["swiglu_block_quantized_gb300/csrc/gemv.cuh",
                "swiglu_block_quantized_gb300/csrc/codec.cuh",
                "swiglu_block_quantized_gb300/csrc/common.cuh"]


# ---------------------------------------------------------------- helpers

def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(name, sources):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", name + ".json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_hash") != source_hash(sources):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi in loop mode; keeps (time, sm_mhz, max_mhz, reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.rows, self.proc = index, [], None

    def start(self):
        try:  # -lms 50: a few samples inside even a short timed region
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 6:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or [r for (_, r) in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2 + i].lower() == "active"})

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return None


def dist_setup(ngpus):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return ws, rank, local


def reduce_max(value, ws):
    """Max of a float over ranks (the only collective of the benchmark)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- oracle legs

def oracle_sample(X, Wg, Wu, rows):
    import oracle
    import synth
    t0 = time.perf_counter()
    oracle.swiglu(X, Wg, Wu, synth.Q4_0, M_, N_, K_, rows=rows)
    return time.perf_counter() - t0


def cpu_baseline(X, Wg, Wu, target_s=12.0):
    """Oracle on a row sample sized to about target_s seconds of wall time
    (grown until the measured time reaches most of the target: a small
    sample underestimates the oracle's rate)."""
    import numpy as np
    n = 8
    while True:
        rows = sorted(set(np.linspace(0, M_ - 1, n).astype(int).tolist()))
        t = oracle_sample(X, Wg, Wu, rows)
        if t >= 0.6 * target_s or len(rows) >= M_:
            break
        n = int(min(M_, max(2 * n, n * target_s / max(t, 1e-3))))
    flops = 2.0 * 2.0 * len(rows) * N_ * K_
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle", "cpu_model": cpu_model(),
            "sample": "%d of %d activation rows of the workload (all %d outputs per row), %.1f s"
                      % (len(rows), M_, N_, t)}


def make_inputs(seed=2):
    import synth
    X = synth.activations(M_, K_, seed=seed)
    Wg = synth.weights(synth.Q4_0, N_, K_, seed=seed, name="Wg")
    Wu = synth.weights(synth.Q4_0, N_, K_, seed=seed, name="Wu")
    return X, Wg, Wu


def run_reference(args, ws, rank):
    if rank != 0:
        return
    X, Wg, Wu = make_inputs()
    rows_per_step = 8
    import numpy as np
    rng = np.random.default_rng(0)
    for _ in range(args.warmup):
        oracle_sample(X, Wg, Wu, sorted(rng.choice(M_, rows_per_step, replace=False).tolist()))
    times = [oracle_sample(X, Wg, Wu, sorted(rng.choice(M_, rows_per_step, replace=False).tolist()))
             for _ in range(args.steps)]
    t = sum(times)
    flops = 2.0 * 2.0 * rows_per_step * N_ * K_ * args.steps
    value = flops / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": M_, "N": N_, "K": K_, "codec": "Q4_0",
                   "step": "CPU oracle on %d random activation rows (all outputs)" % rows_per_step},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": "%d activation rows per step" % rows_per_step},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our arm

def run_ours(args, ws, rank, local):
    import numpy as np
    import torch

    import swiglu_block_quantized_gb300 as m

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    m.build()
    m.load()
    X, Wg, Wu = make_inputs()
    do_cpu = rank == 0 and ws == 1 and not args.no_cpu_baseline
    cpu = cpu_baseline(X, Wg, Wu, args.cpu_seconds) if do_cpu else None

    xs = [torch.from_numpy(X).to(dev) for _ in range(ROTATE)]
    wgs = [torch.from_numpy(Wg).to(dev) for _ in range(ROTATE)]
    wus = [torch.from_numpy(Wu).to(dev) for _ in range(ROTATE)]
    ys = [torch.empty((M_, N_), dtype=torch.float16, device=dev) for _ in range(ROTATE)]
    stream = torch.cuda.current_stream()

    def step(i):
        j = i % ROTATE
        m.swiglu(xs[j], wgs[j], wus[j], m.Q4_0, N_, K_, out=ys[j])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert m.check_device_status() == m.OK

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(ws)
    elapsed_ms = e0.elapsed_time(e1)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    assert m.check_device_status() == m.OK
    elapsed_ms = reduce_max(elapsed_ms, ws)

    flops_step = 2.0 * 2.0 * M_ * N_ * K_
    value = flops_step * args.steps * ws / (elapsed_ms * 1e-3) / 1e12
    per_launch_ms = elapsed_ms / args.steps
    pk, pk_src = peaks()
    achieved = flops_step / (per_launch_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / pk["bf16_tflops"],
                "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
                "traffic": recorded_traffic("tc_swiglu_q4_0_8b_m2048", KERNEL_SOURCES),
                "peak_source": "%s dense bf16 burst (fp16 dense rate is the same)" % pk_src,
                "kernel": "tc_proj_kernel<Q4_0, swiglu, NX=256>"}

    # ---- M = 1: the same weights through the streaming GEMV (HBM bound)
    x1 = [torch.from_numpy(X[:1].copy()).to(dev) for _ in range(ROTATE)]
    y1 = [torch.empty((1, N_), dtype=torch.float16, device=dev) for _ in range(ROTATE)]
    reps = 64   # launches per captured graph (a Python loop would starve a 10 us kernel)
    for i in range(10):
        m.swiglu(x1[i % ROTATE], wgs[i % ROTATE], wus[i % ROTATE], m.Q4_0, N_, K_, out=y1[i % ROTATE])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(reps):
            j = i % ROTATE
            m.swiglu(x1[j], wgs[j], wus[j], m.Q4_0, N_, K_, out=y1[j])
    graph.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    m1_ms = e0.elapsed_time(e1) / reps
    m1_bytes = 2 * m.weight_bytes(m.Q4_0, N_, K_) + K_ * 2 + N_ * 2
    m1_gbs = m1_bytes / (m1_ms * 1e-3) / 1e9
    m1 = {"workload": "8b_swiglu_q4_0_m1", "value": m1_gbs, "unit": "GB/s", "us_per_launch": 1e3 * m1_ms,
          "timing": "CUDA graph of %d back-to-back launches over %d weight copies" % (reps, ROTATE),
          "bytes_per_launch": m1_bytes, "peak": pk["hbm_gbs"], "frac": m1_gbs / pk["hbm_gbs"],
          "peak_source": "%s HBM copy bandwidth" % pk_src,
          "traffic": recorded_traffic("gemv_swiglu_q4_0_8b_m1", GEMV_SOURCES)}

    # ---- end to end through the public API: pinned host X in, Y out each
    # step (m4q_project_host: row chunks copied in, projected and copied back,
    # the copies of a chunk overlapping the kernels of its neighbours)
    xh = torch.from_numpy(X).pin_memory()
    yh = torch.empty((M_, N_), dtype=torch.float16).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    chunk = args.e2e_chunk_rows

    def e2e_step(j):
        m.project_host(xh, wgs[j], m.Q4_0, N_, K_, wu=wus[j], out=yh, x_dev=xs[j], y_dev=ys[j], chunk_rows=chunk)
    for i in range(2):
        e2e_step(i % ROTATE)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i % ROTATE)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), ws) / e2e_steps
    e2e = {"value": flops_step * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
           "h2d_bytes_per_step": X.nbytes, "d2h_bytes_per_step": M_ * N_ * 2,
           "call": "m4q_project_host (chunk_rows %d; 0 = library default)" % chunk,
           "weights": "resident in HBM (model parameters)"}

    # The extra tables are measured after the headline; a failure in one of
    # them is reported in its key (and on stderr) instead of losing the line.
    mlx4 = guarded(measure_mlx4, m, X, dev, steps=max(20, min(args.steps, 200)))
    attention = guarded(measure_attention, m, dev)
    configs = None if args.no_configs else guarded(measure_configs, m, dev, peaks()[0], do_cpu, (wgs[0], wus[0]))

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_launch_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16",
        "data": "synthetic (seeded; LLaMA-8B-shaped MLP, Q4_0 recipe)",
        "config": {"workload": WORKLOAD, "M": M_, "N": N_, "K": K_, "codec": "Q4_0",
                   "accumulate": "fp32", "output": "fp16",
                   "l2": "inputs rotate through %d distinct copies (%.0f MB > L2)"
                         % (ROTATE, ROTATE * (X.nbytes + Wg.nbytes + Wu.nbytes + M_ * N_ * 2) / 1e6),
                   "parallelism": "replicas" if ws > 1 else "single"},
        "roofline": roofline, "m1": m1, "e2e": e2e, "mlx4": mlx4, "attention": attention, "configs": configs,
        "cpu_baseline": cpu, "clocks": clocks,
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


def guarded(fn, *a, **kw):
    try:
        return fn(*a, **kw)
    except Exception as exc:  # reported, not hidden: the key carries the error
        import traceback
        traceback.print_exc()
        return {"error": "%s: %s" % (type(exc).__name__, exc)}


# ---------------------------------------------------------------- every workload

def proj_flops(kind, M, N, K):
    return (4.0 if kind == "swiglu" else 2.0) * M * N * K


def proj_bytes(m, kind, codec, M, N, K):
    """Algorithmic bytes of one projection: packed weights (both for the
    gated form), X read once, Y written once."""
    return (2 if kind == "swiglu" else 1) * m.weight_bytes(codec, N, K) + 2 * M * K + 2 * M * N


def roofline_of(flops, nbytes, pk):
    """(roofline time in s, bound): the slower of the FLOPs at the dense fp16
    tensor peak and the bytes at the HBM copy bandwidth."""
    t_f = flops / (pk["bf16_tflops"] * 1e12)
    t_b = nbytes / (pk["hbm_gbs"] * 1e9)
    return (t_f, "tensor") if t_f >= t_b else (t_b, "hbm")


class GraphTimer:
    """Mean device time of one call: CUDA events around replays of a CUDA
    graph that issues the calls back to back, cycling through `calls` (one
    closure per copy of the inputs, so consecutive launches read different
    memory).  Replays are repeated until about 3 ms of device time is timed."""

    def __init__(self, stream):
        import torch
        self.torch, self.stream = torch, stream
        self.e0 = torch.cuda.Event(enable_timing=True)
        self.e1 = torch.cuda.Event(enable_timing=True)

    def __call__(self, calls, min_calls=40):
        torch = self.torch
        for c in calls[:3]:
            c()   # first launches outside the capture (per-kernel attributes)
        torch.cuda.synchronize()
        reps = len(calls) * max(1, -(-min_calls // len(calls)))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                calls[i % len(calls)]()
        g.replay()
        torch.cuda.synchronize()
        self.e0.record(self.stream)
        g.replay()
        self.e1.record(self.stream)
        torch.cuda.synchronize()
        one = self.e0.elapsed_time(self.e1)
        n = max(1, min(50, int(3.0 / max(one, 1e-3))))
        self.e0.record(self.stream)
        for _ in range(n):
            g.replay()
        self.e1.record(self.stream)
        torch.cuda.synchronize()
        del g
        return self.e0.elapsed_time(self.e1) / (n * reps), reps * n


def copies_for(set_bytes, l2_bytes, most=300):
    """Distinct copies of a launch's inputs and outputs so that the copies
    together exceed twice the L2: each launch then reads cold memory (the
    tiny workload, bound by launch latency, stops at `most` copies)."""
    return int(max(2, min(most, -(-2 * l2_bytes // max(set_bytes, 1)))))


def oracle_rate(kind, X, W, Wu, codec, M, N, K, threads, target_s=1.5):
    """The CPU oracle's TFLOP/s on a row sample of one projection, grown until
    it takes about target_s seconds (or covers every row)."""
    import numpy as np

    import oracle
    n = min(M, 4)
    while True:
        rows = sorted(set(np.linspace(0, M - 1, n).astype(int).tolist()))
        t0 = time.perf_counter()
        if kind == "swiglu":
            oracle.swiglu(X, W, Wu, codec, M, N, K, rows=rows, nthreads=threads)
        else:
            oracle.gemm(X, W, codec, M, N, K, rows=rows, nthreads=threads)
        t = time.perf_counter() - t0
        if t >= 0.6 * target_s or len(rows) >= M:
            break
        n = int(min(M, max(2 * n, n * target_s / max(t, 1e-4))))
    return {"value": proj_flops(kind, len(rows), N, K) / t / 1e12, "unit": "TFLOP/s", "threads": threads,
            "kind": "oracle", "sample": "%d of %d activation rows, all %d outputs, %.2f s" % (len(rows), M, N, t)}


def measure_configs(m, dev, pk, do_cpu, c2w=None):
    """Every workload the pages' tables measure, one GPU: the tiny Q4_0 GEMM,
    the 1B projections in Q4_0 and Q8_0, the Q2_0 sweep over M, and the 1B
    layer set per projection and per layer at M in {1, 128, 512, 2048}.  Each
    entry: time per launch, TFLOP/s, GB/s of algorithmic bytes, and the
    fraction of its roofline (the slower of FLOPs at the dense fp16 peak and
    bytes at HBM bandwidth, both measured).  Inputs and outputs rotate
    through copies larger than twice the L2, so every launch reads cold
    memory; launches are issued from CUDA graphs."""
    import torch

    import synth
    stream = torch.cuda.current_stream()
    timer = GraphTimer(stream)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cpu_threads = os.cpu_count() or 1
    out = {}

    def upload(a):
        return torch.from_numpy(a).to(dev)

    def entry(name, kind, codec, M, N, K, x, w, wu, flops=None, nbytes=None, calls=None, note=None):
        nbytes = nbytes if nbytes is not None else proj_bytes(m, kind, codec, M, N, K)
        flops = flops if flops is not None else proj_flops(kind, M, N, K)
        if calls is None:
            ncopy = copies_for(nbytes, l2)
            xs = [x] + [x.clone() for _ in range(ncopy - 1)]
            ws = [w] + [w.clone() for _ in range(ncopy - 1)]
            wus = [wu] + [wu.clone() for _ in range(ncopy - 1)] if wu is not None else None
            ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _ in range(ncopy)]
            if kind == "swiglu":
                calls = [lambda i=i: m.swiglu(xs[i], ws[i], wus[i], codec, N, K, out=ys[i]) for i in range(ncopy)]
            else:
                calls = [lambda i=i: m.gemm(xs[i], ws[i], codec, N, K, out=ys[i]) for i in range(ncopy)]
        ms, launches = timer(calls)
        t_roof, bound = roofline_of(flops, nbytes, pk)
        e = {"M": M, "N": N, "K": K, "codec": synth.CODEC_NAMES[codec] if codec is not None else "mixed",
             "kind": kind, "us_per_launch": 1e3 * ms, "tflops": flops / (ms * 1e-3) / 1e12,
             "gbs": nbytes / (ms * 1e-3) / 1e9, "flops": flops, "bytes": nbytes, "bound": bound,
             "roofline_us": 1e6 * t_roof, "frac": t_roof / (ms * 1e-3),
             "timing": "CUDA graph, %d launches cycling through %d copies of inputs and outputs (%.0f MB; L2 %.0f MB)"
                       % (launches, len(calls), len(calls) * nbytes / 1e6, l2 / 1e6)}
        if note:
            e["note"] = note
        out[name] = e
        return e

    # C0: the tiny Q4_0 GEMM (a correctness case; bound by launch latency)
    M, N, K = 64, 256, 256
    X0 = synth.activations(M, K, seed=0)
    W0 = synth.weights(synth.Q4_0, N, K, seed=0)
    e = entry("c0_tiny_q4_0_m64", "gemm", synth.Q4_0, M, N, K, upload(X0), upload(W0), None)
    e["bound"] = "launch latency (roofline %.3f us)" % e["roofline_us"]
    if do_cpu:
        e["cpu_baseline"] = [oracle_rate("gemm", X0, W0, None, synth.Q4_0, M, N, K, 1),
                             oracle_rate("gemm", X0, W0, None, synth.Q4_0, M, N, K, cpu_threads)]

    # C1: the 1B projection 2048 x 8192 x 2048 in Q4_0 and Q8_0
    M, N, K = 2048, 8192, 2048
    X1 = synth.activations(M, K, seed=1)
    for codec in (synth.Q4_0, synth.Q8_0):
        W1 = synth.weights(codec, N, K, seed=1)
        e = entry("c1_1b_proj_%s_m2048" % synth.CODEC_NAMES[codec].lower(), "gemm", codec, M, N, K,
                  upload(X1), upload(W1), None)
        if do_cpu:
            e["cpu_baseline"] = [oracle_rate("gemm", X1, W1, None, codec, M, N, K, 1),
                                 oracle_rate("gemm", X1, W1, None, codec, M, N, K, cpu_threads)]

    # C2 over M: the 8B fused gate/up below the headline's M = 2048 (the
    # GEMV for M <= 16, the small-M tcgen05 kernel up to 128, the prefill
    # kernel above), on the headline's weights
    if c2w is not None:
        N2, K2 = 14336, 4096
        for M in (1, 16, 64, 128, 512):
            X2 = synth.activations(M, K2, seed=2)
            entry("c2_8b_swiglu_q4_0_m%d" % M, "swiglu", synth.Q4_0, M, N2, K2, upload(X2), c2w[0], c2w[1])

    # C3: the Q2_0 ternary 4096 x 4096 over M
    N = K = 4096
    W3 = synth.weights(synth.Q2_0, N, K, seed=3)
    w3 = upload(W3)
    for M in (1, 16, 512, 2048):
        X3 = synth.activations(M, K, seed=3)
        e = entry("c3_q2_0_m%d" % M, "gemm", synth.Q2_0, M, N, K, upload(X3), w3, None)
        if do_cpu and M == 2048:
            e["cpu_baseline"] = [oracle_rate("gemm", X3, W3, None, synth.Q2_0, M, N, K, cpu_threads)]

    # C4: the 1B layer set, per projection and per layer (one graph of the
    # layer's launches: q, k, v, o, gate/up, down; and with q/k/v fused into
    # one head-major projection)
    layer = synth.llama1b_layer(1)
    wts = {}
    for i, (name, kind, codec, _, n, k) in enumerate(layer):
        if kind == "swiglu":
            wts[name] = (upload(synth.weights(codec, n, k, seed=40 + i, name="Wg")),
                         upload(synth.weights(codec, n, k, seed=40 + i, name="Wu")))
        else:
            wts[name] = (upload(synth.weights(codec, n, k, seed=40 + i)), None)
    wqkv = torch.cat([wts["q"][0], wts["k"][0], wts["v"][0]]).contiguous()
    for M in (1, 128, 512, 2048):
        xs_in = {}
        lay_flops = lay_bytes = 0.0
        per = {}
        for i, (name, kind, codec, _, n, k) in enumerate(layer):
            x = xs_in.setdefault(k, upload(synth.activations(M, k, seed=60 + k)))
            e = entry("c4_1b_layer_m%d_%s" % (M, name), kind, codec, M, n, k, x, wts[name][0], wts[name][1])
            per[name] = e
            lay_flops += e["flops"]
            lay_bytes += e["bytes"]
        # whole layer as one chain of launches per copy of its activations
        ncopy = copies_for(lay_bytes, l2)
        sets = []
        for c in range(ncopy):
            d = {"x": xs_in[2048].clone() if c else xs_in[2048],
                 "ao": xs_in[2048].clone(),   # stands in for the attention output (o's input)
                 "h": torch.empty((M, 8192), dtype=torch.float16, device=dev),
                 "q": torch.empty((M, 2048), dtype=torch.float16, device=dev),
                 "k": torch.empty((M, 512), dtype=torch.float16, device=dev),
                 "v": torch.empty((M, 512), dtype=torch.float16, device=dev),
                 "qkv": torch.empty((48, M, 64), dtype=torch.float16, device=dev),
                 "o": torch.empty((M, 2048), dtype=torch.float16, device=dev),
                 "y": torch.empty((M, 2048), dtype=torch.float16, device=dev)}
            if c:
                d["w"] = {nm: (a.clone(), b.clone() if b is not None else None) for nm, (a, b) in wts.items()}
                d["wqkv"] = wqkv.clone()
            else:
                d["w"], d["wqkv"] = wts, wqkv
            sets.append(d)

        def layer_call(d, fused):
            w = d["w"]
            if fused:
                m.gemm_heads(d["x"], d["wqkv"], synth.Q8_0, 3072, 2048, 64, out=d["qkv"])
            else:
                m.gemm(d["x"], w["q"][0], synth.Q8_0, 2048, 2048, out=d["q"])
                m.gemm(d["x"], w["k"][0], synth.Q8_0, 512, 2048, out=d["k"])
                m.gemm(d["x"], w["v"][0], synth.Q8_0, 512, 2048, out=d["v"])
            m.gemm(d["ao"], w["o"][0], synth.Q8_0, 2048, 2048, out=d["o"])
            m.swiglu(d["x"], w["gate_up"][0], w["gate_up"][1], synth.Q4_0, 8192, 2048, out=d["h"])
            m.gemm(d["h"], w["down"][0], synth.Q4_0, 2048, 8192, out=d["y"])

        for fused in (False, True):
            calls = [lambda d=d, f=fused: layer_call(d, f) for d in sets]
            name = "c4_1b_layer_m%d_%s" % (M, "layer_fused_qkv" if fused else "layer")
            e = entry(name, "layer", None, M, 2048, 2048, None, None, None, flops=lay_flops, nbytes=lay_bytes,
                      calls=calls, note="%s, one graph of %d launches per layer"
                      % ("q/k/v as one head-major projection" if fused else "q, k, v, o, gate/up, down",
                         4 if fused else 6))
            e["sum_of_projections_us"] = sum(v["us_per_launch"] for v in per.values())
        del sets
        torch.cuda.empty_cache()
    assert m.check_device_status() == m.OK
    return out


def measure_mlx4(m, X, dev, steps):
    """The same layer on MLX 4-bit affine weights (the format of the pages'
    MLX comparison): M = 2048 TFLOP/s and M = 1 GB/s, timed like the
    headline (cold weights rotating through copies; CUDA events)."""
    import torch

    import synth
    # ROTATE distinct weight sets (4 x 73 MB > L2), so each launch reads cold weights
    wg = [torch.from_numpy(synth.weights(synth.MLX4, N_, K_, seed=2 + r, name="Wg")).to(dev) for r in range(ROTATE)]
    wu = [torch.from_numpy(synth.weights(synth.MLX4, N_, K_, seed=2 + r, name="Wu")).to(dev) for r in range(ROTATE)]
    x = torch.from_numpy(X).to(dev)
    y = torch.empty((M_, N_), dtype=torch.float16, device=dev)
    x1 = torch.from_numpy(X[:1].copy()).to(dev)
    y1 = torch.empty((1, N_), dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(4):
        m.swiglu(x, wg[i % ROTATE], wu[i % ROTATE], m.MLX4, N_, K_, out=y)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        m.swiglu(x, wg[i % ROTATE], wu[i % ROTATE], m.MLX4, N_, K_, out=y)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    reps = 64
    graph = torch.cuda.CUDAGraph()
    for i in range(4):
        m.swiglu(x1, wg[i % ROTATE], wu[i % ROTATE], m.MLX4, N_, K_, out=y1)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        for i in range(reps):
            m.swiglu(x1, wg[i % ROTATE], wu[i % ROTATE], m.MLX4, N_, K_, out=y1)
    graph.replay()
    torch.cuda.synchronize()
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    m1_ms = e0.elapsed_time(e1) / reps
    assert m.check_device_status() == m.OK
    m1_bytes = 2 * m.weight_bytes(m.MLX4, N_, K_) + K_ * 2 + N_ * 2
    pk, _ = peaks()
    tflops = 4.0 * M_ * N_ * K_ / (ms * 1e-3) / 1e12
    gbs = m1_bytes / (m1_ms * 1e-3) / 1e9
    return {"workload": "8b_swiglu_mlx4_m2048", "codec": "MLX4 (w = q*s + b, 32-weight groups, 20-byte blocks)",
            "value": tflops, "unit": "TFLOP/s", "ms_per_launch": ms, "steps": steps,
            "frac": tflops / pk["bf16_tflops"],
            "m1": {"workload": "8b_swiglu_mlx4_m1", "value": gbs, "unit": "GB/s", "us_per_launch": 1e3 * m1_ms,
                   "bytes_per_launch": m1_bytes, "frac": gbs / pk["hbm_gbs"]}}


def measure_attention(m, dev, reps=20):
    """Attention of the 8B layer (H = 32, 8 KV heads, D = 128) over an fp16
    and a Q8_0 KV cache: causal prefill M = T = 2048 (TFLOP/s, causal FLOPs
    4 H D sum_i (i + 1)) and one decode token over T = 32768 (GB/s of KV
    cache read).  CUDA events around a graph of `reps` launches."""
    import torch

    import synth
    H, Hkv, D = 32, 8, 128
    out = {}
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pk, _ = peaks()

    def timed(fn):
        # `reps` launches captured in one CUDA graph, so host-side launch
        # cost (a 10-50 us kernel here) does not enter the device time
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(reps):
                fn()
        graph.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    for name, codec in (("q8_0", synth.Q8_0), ("f16", synth.KV_F16)):
        M = T = 2048
        q = torch.from_numpy(synth.queries(H, M, D, seed=1)).to(dev)
        k = torch.from_numpy(synth.kv_cache(codec, Hkv, T, D, seed=2, name="K")).to(dev)
        v = torch.from_numpy(synth.kv_cache(codec, Hkv, T, D, seed=2, name="V")).to(dev)
        o = torch.empty((M, H * D), dtype=torch.float16, device=dev)
        ms = timed(lambda: m.attention(q, k, v, codec, Hkv, T, q_offset=0, out=o))
        flops = 4.0 * H * D * (M * (M + 1) / 2)
        out["prefill_" + name] = {"workload": "8b_attention_causal_m2048_t2048_%s" % name,
                                  "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_launch": ms,
                                  "frac": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
                                  "path": ("tcgen05 attn_tc_kernel" if name == "f16" else
                                           "Q8_0 caches decoded to fp16 in the workspace, then attn_tc_kernel "
                                           "(both launches timed)")}
        # a prefill chunk: 512 new queries over a 4096-token context
        Mc, Tc = 512, 4096
        qc = torch.from_numpy(synth.queries(H, Mc, D, seed=5)).to(dev)
        kcc = torch.from_numpy(synth.kv_cache(codec, Hkv, Tc, D, seed=6, name="K")).to(dev)
        vcc = torch.from_numpy(synth.kv_cache(codec, Hkv, Tc, D, seed=6, name="V")).to(dev)
        oc = torch.empty((Mc, H * D), dtype=torch.float16, device=dev)
        ms = timed(lambda: m.attention(qc, kcc, vcc, codec, Hkv, Tc, q_offset=Tc - Mc, out=oc))
        flops = 4.0 * H * D * sum(Tc - Mc + i + 1 for i in range(Mc))
        out["chunk_" + name] = {"workload": "8b_attention_causal_m512_t4096_%s" % name,
                                "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_launch": ms,
                                "frac": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"]}
        del qc, kcc, vcc, oc
        T = 32768
        q1 = torch.from_numpy(synth.queries(H, 1, D, seed=3)).to(dev)
        kc = [torch.from_numpy(synth.kv_cache(codec, Hkv, T, D, seed=4 + r, name="K")).to(dev) for r in range(2)]
        vc = [torch.from_numpy(synth.kv_cache(codec, Hkv, T, D, seed=4 + r, name="V")).to(dev) for r in range(2)]
        o1 = torch.empty((1, H * D), dtype=torch.float16, device=dev)
        ws = torch.empty(max(1, m.load().m4q_attention_workspace_bytes(H, Hkv, 1, T, D)), dtype=torch.uint8,
                         device=dev)
        it = [0]

        def dec():
            j = it[0] % 2
            it[0] += 1
            m.attention(q1, kc[j], vc[j], codec, Hkv, T, out=o1, workspace=ws)
        ms = timed(dec)
        kv_bytes = 2 * kc[0].numel() * kc[0].element_size()
        out["decode_" + name] = {"workload": "8b_attention_decode_t32768_%s" % name,
                                 "value": kv_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "us_per_launch": 1e3 * ms,
                                 "kv_bytes": kv_bytes, "frac": kv_bytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                 "l2": "two cache copies alternate (%.0f MB each)" % (kv_bytes / 1e6)}
    assert m.check_device_status() == m.OK
    return out


def run_profile_case(case, local):
    """A few launches of one kernel on the full workload, for ncu captures."""
    import torch

    import swiglu_block_quantized_gb300 as m
    torch.cuda.set_device(local)
    m.build()
    if case.startswith("attn_"):
        import synth
        H, Hkv, D = 32, 8, 128
        codec = synth.Q8_0 if case.endswith("q8_0") else synth.KV_F16
        M, T = (2048, 2048) if "prefill" in case else (1, 32768)
        q = torch.from_numpy(synth.queries(H, M, D, seed=1)).cuda()
        k = torch.from_numpy(synth.kv_cache(codec, Hkv, T, D, seed=2, name="K")).cuda()
        v = torch.from_numpy(synth.kv_cache(codec, Hkv, T, D, seed=2, name="V")).cuda()
        for _ in range(3):
            m.attention(q, k, v, codec, Hkv, T, q_offset=T - M)
        torch.cuda.synchronize()
        assert m.check_device_status() == m.OK
        print("profile case %s: 3 launches done" % case)
        return
    if case.startswith("gemm_"):
        # gemm_<codec>_<n>x<k>_m<M>: one projection of the workload table
        import synth
        _, cname, shape, mtag = case.split("_")
        codec = {"q4": synth.Q4_0, "q8": synth.Q8_0, "q2": synth.Q2_0}[cname]
        N, K = (int(v) for v in shape.split("x"))
        M = int(mtag[1:])
        x = torch.from_numpy(synth.activations(M, K, seed=1)).cuda()
        w = torch.from_numpy(synth.weights(codec, N, K, seed=1)).cuda()
        y = torch.empty((M, N), dtype=torch.float16, device="cuda")
        for _ in range(3):
            m.gemm(x, w, codec, N, K, out=y)
        torch.cuda.synchronize()
        assert m.check_device_status() == m.OK
        print("profile case %s: 3 launches done" % case)
        return
    X, Wg, Wu = make_inputs()
    codec = m.Q4_0
    if "mlx4" in case:
        import synth
        codec = m.MLX4
        Wg = synth.weights(synth.MLX4, N_, K_, seed=2, name="Wg")
        Wu = synth.weights(synth.MLX4, N_, K_, seed=2, name="Wu")
    if case.endswith("_m1"):
        X = X[:1].copy()
    elif case.endswith("_m64"):
        X = X[:64].copy()
    x = torch.from_numpy(X).cuda()
    wg, wu = torch.from_numpy(Wg).cuda(), torch.from_numpy(Wu).cuda()
    y = torch.empty((X.shape[0], N_), dtype=torch.float16, device="cuda")
    for _ in range(3):
        m.swiglu(x, wg, wu, codec, N_, K_, out=y)
    torch.cuda.synchronize()
    assert m.check_device_status() == m.OK
    print("profile case %s: 3 launches done" % case)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--e2e-chunk-rows", type=int, default=0,
                    help="rows per chunk of the end-to-end call (0: the library default)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload table (every BASELINE workload, timed after the headline)")
    ap.add_argument("--profile-case", default=None,
                    choices=["swiglu_m2048", "swiglu_m1", "swiglu_m64", "swiglu_mlx4_m2048", "swiglu_mlx4_m1",
                             "attn_prefill_q8_0", "attn_decode_q8_0", "attn_prefill_f16", "attn_decode_f16",
                             "gemm_q4_8192x2048_m2048", "gemm_q8_8192x2048_m2048", "gemm_q2_4096x4096_m1",
                             "gemm_q2_4096x4096_m16", "gemm_q2_4096x4096_m2048", "gemm_q8_512x2048_m128",
                             "gemm_q4_2048x8192_m128"],
                    help="only run 3 launches of one case (for ncu)")
    args = ap.parse_args(argv)
    if args.profile_case:
        run_profile_case(args.profile_case, int(os.environ.get("LOCAL_RANK", "0")))
        return
    if args.warmup < 3:
        args.warmup = 3
    ws, rank, local = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
