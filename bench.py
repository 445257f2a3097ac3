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
            "kind": "oracle",
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

    # ---- end to end through the public API: pinned host X in, Y out each step
    xh = torch.from_numpy(X).pin_memory()
    yh = torch.empty((M_, N_), dtype=torch.float16).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    xd, yd = xs[0], ys[0]
    for _ in range(2):
        xd.copy_(xh, non_blocking=True)
        m.swiglu(xd, wgs[0], wus[0], m.Q4_0, N_, K_, out=yd)
        yh.copy_(yd, non_blocking=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(e2e_steps):
        j = i % ROTATE
        xs[j].copy_(xh, non_blocking=True)
        m.swiglu(xs[j], wgs[j], wus[j], m.Q4_0, N_, K_, out=ys[j])
        yh.copy_(ys[j], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = reduce_max(e0.elapsed_time(e1), ws) / e2e_steps
    e2e = {"value": flops_step * ws / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": X.nbytes, "d2h_bytes_per_step": M_ * N_ * 2,
           "weights": "resident in HBM (model parameters)"}

    mlx4 = measure_mlx4(m, X, dev, steps=max(20, min(args.steps, 200)))
    attention = measure_attention(m, dev)

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
        "roofline": roofline, "m1": m1, "e2e": e2e, "mlx4": mlx4, "attention": attention,
        "cpu_baseline": cpu, "clocks": clocks,
        "gpu_launches": args.steps,
    }
    print(json.dumps(line), flush=True)


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
                                  "value": flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_launch": ms}
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
    ap.add_argument("--profile-case", default=None,
                    choices=["swiglu_m2048", "swiglu_m1", "swiglu_m64", "swiglu_mlx4_m2048", "swiglu_mlx4_m1",
                             "attn_prefill_q8_0", "attn_decode_q8_0", "attn_prefill_f16", "attn_decode_f16"],
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
