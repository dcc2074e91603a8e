"""Benchmark of the W4A16 group-128 linear layer on one GB300 (or N replicas).

Default workload (one JSON line): the full Llama-3-8B decode-step linear
stream -- 32 decoder layers of qkv 4096->6144, o_proj 4096->4096, gate_up
4096->28672 and down 14336->4096, plus lm_head 4096->128256: 129 GEMMs and
7 504 658 432 streamed weights per decode step -- swept over the batch sizes
B in {1, 4, 16, 64, 128, 256, 270, 384, 512, 1024} that map the
memory-bound-to-compute-bound crossover.  One bench step is one decode step
at every B of the sweep (1290 GEMMs: the whole hot path -- weight + scale
stream, register decode, tensor products, split-K reduction, bf16
epilogue).  Synthetic seeded inputs with the shapes and value distributions
of that workload; the 129 distinct weight sets (3.87 GB) exceed L2, so every
GEMM streams its weights from HBM.

``value`` is the time of one sweep step in µs; ``per_batch`` gives, for every
B, the decode step's µs, TB/s, TFLOP/s, its roofline (bound, fraction of the
measured peak) and the measured time above max(memory, math) -- the
dequantisation cost the two-term decode-step model predicts, where it stops
hiding.  Other workloads (``--workload``) print the same kind of line for the
decoder-layer set, the prefill, single-step and zero-point shapes.

``--impl reference`` times the CPU oracle (the slow definition the library is
checked against) on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("W4A16 decode GEMM µs/step & TB/s (small B), TFLOP/s (large B); "
          "% roofline on 1 GB300")
LAYER = [("qkv", 4096, 6144), ("o_proj", 4096, 4096), ("gate_up", 4096, 28672),
         ("down", 14336, 4096)]
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024
FORCE = -1  # kernel path forced from the command line (-1: the library's choice)
SWEEP_BATCHES = (1, 4, 16, 64, 128, 256, 270, 384, 512, 1024)
LM_HEAD = ("lm_head", 4096, 128256)


# --------------------------------------------------------------- workloads

def workload(name: str, batch: int | None, shape: str | None = None):
    """List of (label, B, K, N, zero_points, outlier_frac) GEMMs forming one step."""
    if name == "decode_layer":
        return [(f"{lbl}_B{B}", B, K, N, False, 0.0)
                for B in (1, 2, 4, 8, 16) for lbl, K, N in LAYER]
    if name == "single":
        K, N = (int(v) for v in (shape or "4096x4096").split("x"))
        return [(f"linear_{K}x{N}", batch or 1, K, N, False, 0.0)]
    if name == "decode_step":
        B = batch or 1
        return [(f"{lbl}_L{i}", B, K, N, False, 0.0) for i in range(32) for lbl, K, N in LAYER] + \
            [("lm_head", B, 4096, 128256, False, 0.0)]
    if name == "prefill":
        return [(lbl, batch or 2048, K, N, False, 0.01) for lbl, K, N in LAYER if lbl != "o_proj"]
    if name == "zp70b":
        B = batch or 1
        return [(f"{lbl}_B{B}", B, K, N, True, 0.0) for lbl, K, N in
                (("qkv", 8192, 10240), ("gate_up", 8192, 57344), ("down", 28672, 8192))]
    raise SystemExit(f"unknown workload {name}")


def step_bytes_flops(gemms):
    from weight_only_int4_gemm_gb300 import model
    b = sum(model.linear_bytes(B, K, N, zp) for _, B, K, N, zp, _ in gemms)
    f = sum(model.linear_flops(B, K, N) for _, B, K, N, _, _ in gemms)
    return b, f


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        hbm = d.get("hbm_gbs")
        tf = d.get("bf16_tflops")
        tfs = d.get("bf16_tflops_sustained", tf)
        if hbm and tf:
            return float(hbm), float(tf), float(tfs), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash(names):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_int4_gemm_gb300", "csrc")
    for n in names:
        with open(os.path.join(csrc, n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_COMMON = ["dequant.cuh", "epilogue.cuh", "fmt16.cuh", "checks.cuh", "launch.cuh"]
KERNEL_FILES = {"skinny": ["skinny.cu"] + _COMMON,
                "skinny_kernel": ["skinny.cu"] + _COMMON,
                "tcgen05": ["tc_gemm.cu", "tc_wide.cu", "tc_ptx.cuh"] + _COMMON,
                "tc_kernel": ["tc_gemm.cu", "tc_ptx.cuh"] + _COMMON,
                "wide_kernel": ["tc_wide.cu", "tc_ptx.cuh"] + _COMMON}


def traffic_from_profiles(kernel: str, workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(KERNEL_FILES[kernel])
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and \
                parts[1] == workload_name and parts[2] == want:
            return float(parts[3])
    return None


# --------------------------------------------------------------- clocks

class ClockSampler:
    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = device_index

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 8:
                self.samples.append(f)
        return False

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for s in self.samples for n, v in zip(names, s[4:8]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.samples)}


# --------------------------------------------------------------- GPU arm

def copy_index(gemms, uses, n_copies):
    """For step k, GEMM i uses copy (k * uses + occurrence) % n_copies of its
    layer, so two uses of one copy are n_copies uses of that layer apart."""
    occ, seen = [], {}
    for _, B, K, N, zp, _ in gemms:
        key = (K, N, zp)
        occ.append(seen.get(key, 0))
        seen[key] = seen.get(key, 0) + 1
    return lambda k, i, key: (k * uses[key] + occ[i]) % n_copies


def build_buffers(gemms, copies_for, device):
    """Packed weights (several copies when needed to defeat L2), scales, x, y."""
    import torch

    import weight_only_int4_gemm_gb300 as w
    from weight_only_int4_gemm_gb300 import inputs

    layers = {}
    for label, B, K, N, zp, outl in gemms:
        key = (K, N, zp)
        if key not in layers:
            reps = []
            for c in range(copies_for(key)):
                qw, sc, qz = inputs.make_weights(K, N, seed=7 * K + 13 * N + 1_000_003 * c + zp,
                                                 zero_points=zp, device=device)
                reps.append((w.w4a16_pack(qw, qz), sc))
                del qw, qz
            layers[key] = reps
    acts = {}
    for i, (label, B, K, N, zp, outl) in enumerate(gemms):
        acts[i] = (inputs.make_activations(B, K, seed=10_000 + i, outlier_frac=outl, device=device),
                   torch.empty((B, N), dtype=torch.bfloat16, device=device))
    torch.cuda.synchronize()
    return layers, acts


def run_gpu(args, gemms, rank, world, device):
    import torch

    import weight_only_int4_gemm_gb300 as w

    per_copy = {}
    for _, B, K, N, zp, _ in gemms:
        per_copy[(K, N, zp)] = w.w4a16_packed_bytes(K, N, zp) + (K // 128) * N * 2
    distinct_bytes = sum(per_copy.values())
    uses = {}
    for _, B, K, N, zp, _ in gemms:
        uses[(K, N, zp)] = uses.get((K, N, zp), 0) + 1
    # copies so that the bytes streamed between two uses of one copy exceed 4x L2
    if distinct_bytes * max(uses.values()) >= 4 * L2_BYTES and max(uses.values()) == 1:
        n_copies = 1
    else:
        n_copies = max(2, -(-4 * L2_BYTES // max(1, distinct_bytes)) + 1)
    layers, acts = build_buffers(gemms, lambda key: n_copies, device)

    ws = torch.zeros(max(w.w4a16_workspace_bytes(B, K, N) for _, B, K, N, _, _ in gemms) + 256,
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)
    paths = [w.w4a16_select_path(B, K, N) if FORCE < 0 else FORCE for _, B, K, N, _, _ in gemms]

    counter = {"i": 0}
    pick = copy_index(gemms, uses, n_copies)

    def one_step():
        # every GEMM uses the next copy of its layer's weights (round robin)
        for i, (label, B, K, N, zp, _) in enumerate(gemms):
            packed, sc = layers[(K, N, zp)][pick(counter["i"], i, (K, N, zp))]
            x, y = acts[i]
            w.w4a16_gemm(x, packed, sc, zp, N, out=y, workspace=ws, stream=stream, path=FORCE)
        counter["i"] += 1

    # capture one CUDA graph per copy rotation so launch overhead stays off the clock
    graphs = []
    with torch.cuda.stream(stream):
        for _ in range(3):
            one_step()
    stream.synchronize()
    n_graphs = n_copies
    for g in range(n_graphs):
        counter["i"] = g
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            one_step()
        graphs.append(graph)
    stream.synchronize()

    def replay(k):
        graphs[k % n_graphs].replay()

    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            replay(k)
    stream.synchronize()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(device.index or 0) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for k in range(args.steps):
                replay(k)
            stop.record(stream)
        stop.synchronize()
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    ms = start.elapsed_time(stop)
    assert w.w4a16_device_status() == 0, "device-side wait timed out during the bench"
    # per-step distribution: events around each of up to 200 further replays
    n_dist = min(args.steps, 200)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_dist + 1)]
    with torch.cuda.stream(stream):
        evs[0].record(stream)
        for k in range(n_dist):
            replay(k)
            evs[k + 1].record(stream)
    evs[-1].synchronize()
    per_step = sorted(evs[k].elapsed_time(evs[k + 1]) for k in range(n_dist))
    step_pct = {"p10_ms": per_step[int(0.1 * (n_dist - 1))],
                "p50_ms": per_step[int(0.5 * (n_dist - 1))],
                "p90_ms": per_step[int(0.9 * (n_dist - 1))], "replays": n_dist}

    if args.per_gemm:
        per_gemm_table(gemms, layers, ws, stream, device, load_peaks()[0], path=FORCE)
    # end to end through the public API with host buffers
    e2e = run_e2e(args, gemms, layers, device, ws, pick, n_copies)
    return ms, clk.summary(), paths, n_copies, e2e, step_pct


def per_gemm_table(gemms, layers, ws, stream, device, hbm_gbs, reps=200, path=-1,
                   tflops=None):
    """Each distinct (B, K, N) alone, in a CUDA graph of `reps` launches that
    rotate over the weight copies; prints one line per GEMM to stderr, with the
    roofline fraction against the burst peaks (a kernel timed alone)."""
    import torch

    import weight_only_int4_gemm_gb300 as w
    from weight_only_int4_gemm_gb300 import model

    seen = set()
    for i, (label, B, K, N, zp, _) in enumerate(gemms):
        if (B, K, N, zp) in seen:
            continue
        seen.add((B, K, N, zp))
        reps_list = layers[(K, N, zp)]
        x = torch.randn((B, K), device=device).to(torch.bfloat16)
        y = torch.empty((B, N), dtype=torch.bfloat16, device=device)
        with torch.cuda.stream(stream):
            for r in range(3):
                packed, sc = reps_list[r % len(reps_list)]
                w.w4a16_gemm(x, packed, sc, zp, N, out=y, workspace=ws, stream=stream, path=path)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                packed, sc = reps_list[r % len(reps_list)]
                w.w4a16_gemm(x, packed, sc, zp, N, out=y, workspace=ws, stream=stream, path=path)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / reps
        byts = model.linear_bytes(B, K, N, zp)
        fl = model.linear_flops(B, K, N)
        pname = w.w4a16_kernel_name(B, K, N) if path < 0 else w.PATH_NAMES[path]
        tf = tflops or load_peaks()[1]
        roof = max(byts / (hbm_gbs * 1e3), fl / (tf * 1e6))  # µs
        print(f"per-gemm B={B:5d} K={K:6d} N={N:6d} zp={int(zp)} kernel={pname:12s} "
              f"{us:9.2f} us  {byts / us / 1e3:8.1f} GB/s ({byts / us / 1e3 / hbm_gbs * 100:5.1f}% hbm)  "
              f"{fl / us / 1e6:8.1f} TFLOP/s ({fl / us / 1e6 / tf * 100:5.1f}% bf16 burst)  "
              f"roofline frac {roof / us:5.3f}", file=sys.stderr, flush=True)


def run_e2e(args, gemms, layers, device, ws, pick, n_copies):
    """End to end through the public API with host buffers: every step copies
    all of its inputs from one pinned host buffer to the device, runs the step's
    GEMMs through ``w4a16_gemm`` and copies all outputs back to one pinned host
    buffer.  Timed twice: replaying CUDA graphs of that sequence (one per weight
    rotation, as a serving loop would; the copies happen on every replay), and
    eagerly (one Python call per GEMM).  Returns both."""
    import torch

    import weight_only_int4_gemm_gb300 as w
    from weight_only_int4_gemm_gb300 import inputs

    x_sizes = [B * K for _, B, K, _, _, _ in gemms]
    y_sizes = [B * N for _, B, _, N, _, _ in gemms]
    host_x = torch.empty(sum(x_sizes), dtype=torch.bfloat16).pin_memory()
    host_y = torch.empty(sum(y_sizes), dtype=torch.bfloat16).pin_memory()
    off = 0
    for i, (label, B, K, N, zp, outl) in enumerate(gemms):
        host_x[off:off + x_sizes[i]] = inputs.make_activations(
            B, K, seed=20_000 + i, outlier_frac=outl).reshape(-1)
        off += x_sizes[i]
    dev_x = torch.empty_like(host_x, device=device)
    dev_y = torch.empty_like(host_y, device=device)
    xs, ys, ox, oy = [], [], 0, 0
    for i, (label, B, K, N, zp, _) in enumerate(gemms):
        xs.append(dev_x[ox:ox + x_sizes[i]].view(B, K))
        ys.append(dev_y[oy:oy + y_sizes[i]].view(B, N))
        ox += x_sizes[i]
        oy += y_sizes[i]
    h2d, d2h = host_x.numel() * 2, host_y.numel() * 2
    steps = max(3, min(args.steps, args.e2e_steps))
    stream = torch.cuda.Stream(device)

    def step(k):
        dev_x.copy_(host_x, non_blocking=True)
        for i, (label, B, K, N, zp, _) in enumerate(gemms):
            packed, sc = layers[(K, N, zp)][pick(k, i, (K, N, zp))]
            w.w4a16_gemm(xs[i], packed, sc, zp, N, out=ys[i], workspace=ws, stream=stream,
                         path=FORCE)
        host_y.copy_(dev_y, non_blocking=True)

    def timed(run):
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            start.record(stream)
            for k in range(steps):
                run(k)
            stop.record(stream)
        stop.synchronize()
        return start.elapsed_time(stop)

    with torch.cuda.stream(stream):
        for k in range(3):
            step(k)
    stream.synchronize()
    eager_ms = timed(step)
    graphs = []
    for g in range(n_copies):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step(g)
        graphs.append(graph)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for k in range(3):
            graphs[k % n_copies].replay()
    stream.synchronize()
    graph_ms = timed(lambda k: graphs[k % n_copies].replay())
    return graph_ms, eager_ms, steps, h2d, d2h


# --------------------------------------------------------------- oracle arm

class OracleSampler:
    """Times the CPU oracle on a column sample of every GEMM of one step and
    extrapolates to the whole step (the oracle's cost is linear in columns:
    each column is dequantised once and dotted with every row)."""

    def __init__(self, gemms):
        import numpy as np

        import oracle
        from weight_only_int4_gemm_gb300 import inputs

        def bits(t):
            t = t.contiguous()
            return t.view(__import__("torch").int16).numpy().view(np.uint16) \
                if str(t.dtype) == "torch.bfloat16" else t.numpy().view(np.uint32)

        self.MAX_COLS = 16384
        self.np, self.oracle, self.gemms = np, oracle, gemms
        self.probs = []
        for i, (label, B, K, N, zp, outl) in enumerate(gemms):
            qw, sc, qz = inputs.make_weights(K, min(N, self.MAX_COLS), seed=i, zero_points=zp)
            x = inputs.make_activations(B, K, seed=30_000 + i, outlier_frac=outl)
            self.probs.append((bits(x), bits(qw), bits(sc), None if qz is None else bits(qz), N))
        self.cols = 1

    def step(self) -> float:
        est = 0.0
        c = self.np.arange(self.cols, dtype=self.np.int32)
        for x, qw, sc, qz, N in self.probs:
            t1 = time.perf_counter()
            self.oracle.gemm(x, qw, sc, qz, cols=c)
            est += (time.perf_counter() - t1) * N / self.cols
        return est

    def calibrate(self, seconds_per_step: float):
        """Grow the column sample (1 .. 16384) until one sampled step costs about
        ``seconds_per_step`` of CPU time."""
        while self.cols < self.MAX_COLS:
            t0 = time.perf_counter()
            self.step()
            if time.perf_counter() - t0 >= seconds_per_step:
                break
            self.cols *= 2

    def describe(self, steps: int, seconds: float) -> str:
        return (f"{self.cols} column(s) of each of the {len(self.gemms)} GEMMs of one step "
                f"(all rows, all K), timed and scaled by N/columns; {steps} sampled step(s), "
                f"{seconds:.1f} s of CPU work")


def reduce_times_over_ranks(ms: float, e2e_step_ms: float, world: int, device=None):
    """Replicas run independently; the job takes as long as the slowest rank,
    so both timings are reduced with MAX over ranks (no data-path collective)."""
    if world <= 1:
        return ms, e2e_step_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms, e2e_step_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0]), float(t[1])


def aggregate_value(bytes_per_step: int, world: int, step_s: float) -> float:
    """Whole-job TB/s: every replica streams its own step's bytes."""
    return bytes_per_step * world / step_s / 1e12


# --------------------------------------------------------------- decode-step sweep

def sweep_layers():
    """The 129 GEMM shapes of one Llama-3-8B decode step, in execution order."""
    return [(f"{lbl}_L{i}", K, N) for i in range(32) for lbl, K, N in LAYER] + [LM_HEAD]


def sweep_roofline(byts: float, flops: float, t_s: float, hbm: float, tflops: float):
    """Bound, achieved, fraction and the time above max(memory, math)."""
    t_mem = byts / (hbm * 1e9)
    t_math = flops / (tflops * 1e12)
    if t_mem >= t_math:
        r = {"bound": "hbm", "achieved": byts / t_s / 1e9, "peak": hbm, "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": flops / t_s / 1e12, "peak": tflops,
             "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["memory_us"] = t_mem * 1e6
    r["math_us"] = t_math * 1e6
    r["above_roofline_us"] = (t_s - max(t_mem, t_math)) * 1e6
    return r


class SweepOracleSampler:
    """Times the CPU oracle on a column sample of every distinct (B, K, N) of the
    sweep and extrapolates to the whole sweep step (the oracle's cost is linear
    in columns: each column is dequantised once and dotted with every row)."""

    def __init__(self, batches):
        import numpy as np

        import oracle
        from weight_only_int4_gemm_gb300 import inputs
        self.np, self.oracle = np, oracle
        self.MAX_COLS = 4096
        counts = {}
        for _, K, N in sweep_layers():
            counts[(K, N)] = counts.get((K, N), 0) + 1
        self.probs = []
        for B in batches:
            for i, ((K, N), cnt) in enumerate(sorted(counts.items())):
                qw, sc, _ = inputs.make_weights(K, min(N, self.MAX_COLS), seed=i)
                x = inputs.make_activations(B, K, seed=30_000 + 7 * B + i)
                self.probs.append((B, x.view(__import__("torch").int16).numpy().view(np.uint16),
                                   qw.numpy().view(np.uint32),
                                   sc.view(__import__("torch").int16).numpy().view(np.uint16),
                                   N, cnt))
        self.cols = 1

    def step(self) -> float:
        est = 0.0
        c = self.np.arange(self.cols, dtype=self.np.int32)
        for B, x, qw, sc, N, cnt in self.probs:
            t1 = time.perf_counter()
            self.oracle.gemm(x, qw, sc, None, cols=c)
            est += (time.perf_counter() - t1) * N / self.cols * cnt
        return est

    def calibrate(self, seconds_per_step: float):
        while self.cols < self.MAX_COLS:
            t0 = time.perf_counter()
            self.step()
            if time.perf_counter() - t0 >= seconds_per_step:
                break
            self.cols *= 2

    def describe(self, steps: int, seconds: float) -> str:
        return (f"{self.cols} column(s) of each of the {len(self.probs)} distinct (B, K, N) "
                f"GEMMs of the sweep (all rows, all K), timed and extrapolated by N/columns "
                f"and by the GEMM's count per decode step (32 layers, 1 lm_head); {steps} "
                f"sampled step(s), {seconds:.1f} s of CPU work")


def kernel_name(w, B, K, N):
    return w.w4a16_kernel_name(B, K, N) if FORCE < 0 else w.PATH_NAMES[FORCE]


def run_sweep(args, rank, world, device):
    """Config 3: one decode step at every B of the sweep, as one CUDA graph per B."""
    import torch

    import weight_only_int4_gemm_gb300 as w
    from weight_only_int4_gemm_gb300 import inputs, model

    batches = [args.batch] if args.batch else list(SWEEP_BATCHES)
    shapes = sweep_layers()
    hbm, tf_burst, tf_sust, peak_src = load_peaks()
    # 129 distinct weight sets (3.87 GB > L2): every GEMM streams from HBM
    weights = []
    for i, (lbl, K, N) in enumerate(shapes):
        qw, sc, _ = inputs.make_weights(K, N, seed=1_000 + i, device=device)
        weights.append((w.w4a16_pack(qw), sc))
        del qw
    ws = torch.zeros(max(w.w4a16_workspace_bytes(B, K, N) for B in batches
                         for _, K, N in shapes) + 256, dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)
    per_b = []
    for B in batches:
        x_tot = sum(B * K for _, K, _ in shapes)
        y_tot = sum(B * N for _, _, N in shapes)
        dev_x = torch.empty(x_tot, dtype=torch.bfloat16, device=device)
        dev_y = torch.empty(y_tot, dtype=torch.bfloat16, device=device)
        xs, ys, ox, oy = [], [], 0, 0
        for i, (lbl, K, N) in enumerate(shapes):
            xs.append(dev_x[ox:ox + B * K].view(B, K))
            ys.append(dev_y[oy:oy + B * N].view(B, N))
            xs[-1].copy_(inputs.make_activations(B, K, seed=10_000 + 7 * B + i, device=device))
            ox += B * K
            oy += B * N
        byts = sum(model.linear_bytes(B, K, N) for _, K, N in shapes)
        flops = sum(model.linear_flops(B, K, N) for _, K, N in shapes)
        kern = kernel_name(w, B, 4096, 4096)
        per_b.append({"B": B, "dev_x": dev_x, "dev_y": dev_y, "xs": xs, "ys": ys,
                      "bytes": byts, "flops": flops, "kernel": kern})

    def decode_step(e):
        for i, (lbl, K, N) in enumerate(shapes):
            packed, sc = weights[i]
            w.w4a16_gemm(e["xs"][i], packed, sc, False, N, out=e["ys"][i], workspace=ws,
                         stream=stream, path=FORCE)

    with torch.cuda.stream(stream):
        for e in per_b:
            decode_step(e)
    stream.synchronize()
    for e in per_b:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            decode_step(e)
        e["graph"] = g
    stream.synchronize()

    def sweep_step(evs=None):
        for j, e in enumerate(per_b):
            if evs is not None:
                evs[j].record(stream)
            e["graph"].replay()
        if evs is not None:
            evs[-1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            sweep_step()
    stream.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(device)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(per_b) + 1)]
           for _ in range(args.steps)]
    with ClockSampler(device.index or 0) as clk:
        with torch.cuda.stream(stream):
            for k in range(args.steps):
                sweep_step(evs[k])
        evs[-1][-1].synchronize()
    torch.cuda.synchronize(device)
    if world > 1:
        dist.barrier()
    assert w.w4a16_device_status() == 0, "device-side wait timed out during the bench"
    ms_total = evs[0][0].elapsed_time(evs[-1][-1])
    for j, e in enumerate(per_b):
        times = sorted(evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps))
        e["ms"] = sum(times) / len(times)
        e["p50_ms"] = times[len(times) // 2]
        e["p10_ms"] = times[(len(times) - 1) // 10]
        e["p90_ms"] = times[len(times) - 1 - (len(times) - 1) // 10]

    # end to end through the public API with host buffers: per B, one H2D
    # copy of all of the decode step's activations from pinned host memory,
    # the step's 129 w4a16_gemm calls and one D2H copy of all of its outputs,
    # captured as one CUDA graph per B and replayed once per sweep step
    h2d = d2h = 0
    for e in per_b:
        e["host_x"] = e["dev_x"].cpu().pin_memory()
        e["host_y"] = torch.empty(e["dev_y"].numel(), dtype=torch.bfloat16).pin_memory()
        h2d += e["host_x"].numel() * 2
        d2h += e["host_y"].numel() * 2

    def e2e_body(e):
        e["dev_x"].copy_(e["host_x"], non_blocking=True)
        decode_step(e)
        e["host_y"].copy_(e["dev_y"], non_blocking=True)

    with torch.cuda.stream(stream):
        for e in per_b:
            e2e_body(e)
    stream.synchronize()
    for e in per_b:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_body(e)
        e["e2e_graph"] = g
    e2e_steps = max(3, min(args.steps, args.e2e_steps, 10))
    with torch.cuda.stream(stream):
        for e in per_b:
            e["e2e_graph"].replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for e in per_b:
                e["e2e_graph"].replay()
        e1.record(stream)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    assert w.w4a16_device_status() == 0, "device-side wait timed out during the bench"
    if args.per_gemm:
        seen = {}
        for i, (lbl, K, N) in enumerate(shapes):
            seen.setdefault((K, N), i)
        for e in per_b:
            gem = [(f"{shapes[i][0]}_B{e['B']}", e["B"], K, N, False, 0.0)
                   for (K, N), i in seen.items()]
            lays = {(K, N, False): [weights[i]] + [weights[j] for j, s2 in enumerate(shapes)
                                                  if (s2[1], s2[2]) == (K, N) and j != i][:5]
                    for (K, N), i in seen.items()}
            per_gemm_table(gem, lays, ws, stream, device, hbm, path=FORCE, tflops=tf_burst)
    return per_b, ms_total / args.steps, clk.summary(), e2e_ms, h2d, d2h, e2e_steps


def sweep_line(args, per_b, step_ms, clocks, e2e_ms, h2d, d2h, e2e_steps, world, device):
    import weight_only_int4_gemm_gb300 as w

    hbm, tf_burst, tf_sust, peak_src = load_peaks()
    step_ms, e2e_ms = reduce_times_over_ranks(step_ms, e2e_ms, world, device)
    rows = []
    by_kernel = {}
    for e in per_b:
        t = e["ms"] / 1e3
        r = sweep_roofline(e["bytes"], e["flops"], t, hbm, tf_sust)
        # the launch plan of each distinct shape at this batch (what ran)
        plans = {}
        for lbl, K, N in (list(LAYER) + [LM_HEAD] if FORCE == -1 else []):
            pl = w.w4a16_describe_plan(e["B"], K, N)
            plans[f"{lbl} {K}x{N}"] = (f"{pl['kernel_name']} rows {pl['batch_rows']} x "
                                       f"{pl['batch_tiles']}, K splits {pl['k_splits']}, "
                                       f"grid {pl['grid']}")
        rows.append({"B": e["B"], "kernel": e["kernel"], "plans": plans,
                     "us_per_step": e["ms"] * 1e3,
                     "p50_us": e["p50_ms"] * 1e3, "p10_us": e["p10_ms"] * 1e3,
                     "p90_us": e["p90_ms"] * 1e3, "tb_s": e["bytes"] / t / 1e12,
                     "tflops": e["flops"] / t / 1e12, "roofline": {
                         k: r[k] for k in ("bound", "achieved", "peak", "unit", "frac")},
                     "memory_us": r["memory_us"], "math_us": r["math_us"],
                     "above_roofline_us": r["above_roofline_us"],
                     "algorithmic_bytes": e["bytes"], "flops": e["flops"]})
        k = by_kernel.setdefault(e["kernel"], {"s": 0.0, "bytes": 0, "flops": 0, "launches": 0})
        k["s"] += t
        k["bytes"] += e["bytes"]
        k["flops"] += e["flops"]
        k["launches"] += len(sweep_layers())
    dom_name, dom = max(by_kernel.items(), key=lambda kv: kv[1]["s"])
    roof = sweep_roofline(dom["bytes"], dom["flops"], dom["s"], hbm, tf_sust)
    roof = {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac")}
    roof.update({"peak_source": f"{peak_src} " + ("hbm_gbs" if roof["bound"] == "hbm"
                                                  else "bf16 sustained (timed inside a long step)"),
                 "kernel": dom_name, "launches_per_step": dom["launches"],
                 "share_of_step": dom["s"] / (step_ms / 1e3),
                 "traffic": traffic_from_profiles(dom_name, "decode_sweep"),
                 "algorithmic_bytes_per_launch": dom["bytes"] / dom["launches"],
                 "flops_per_launch": dom["flops"] / dom["launches"]})
    sbytes = sum(e["bytes"] for e in per_b)
    sflops = sum(e["flops"] for e in per_b)
    launches = len(sweep_layers()) * len(per_b)
    line = {"metric": METRIC, "value": step_ms * 1e3, "unit": "µs/step",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_ms, "us_per_step": step_ms * 1e3,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; Llama-3-8B shapes, no trained weights)",
            "config": {"workload": "decode_sweep: full Llama-3-8B decode-step linear stream "
                                   "(32 layers + lm_head, 129 GEMMs) at every B of the sweep",
                       "batches": [e["B"] for e in per_b], "gemms_per_decode_step": 129,
                       "streamed_weights": sum(K * N for _, K, N in sweep_layers()),
                       "shapes_KxN": ["4096x6144", "4096x4096", "4096x28672", "14336x4096",
                                      "4096x128256"],
                       "group": 128, "zero_points": False,
                       "algorithmic_bytes_per_step": sbytes, "flops_per_step": sflops,
                       "step": "one decode step at every B of the sweep",
                       "l2": "129 distinct weight sets (3.87 GB) per decode step: inputs larger "
                             "than L2", "cuda_graph": "one graph per B",
                       "parallelism": f"replicas{world}"},
            "throughput": {"tb_s": sbytes * world / (step_ms / 1e3) / 1e12,
                           "tflops": sflops * world / (step_ms / 1e3) / 1e12},
            "per_batch": rows, "roofline": roof, "clocks": clocks,
            "gpu_launches": args.steps * launches,
            "e2e": {"value": e2e_ms * 1e3, "unit": "µs/step", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "launch": "per B, one CUDA graph of: an H2D copy of all of the decode "
                              "step's activations from pinned host memory, its 129 w4a16_gemm "
                              "calls, a D2H copy of all of its outputs"}}
    return line


# --------------------------------------------------------------- offline quantizer

FP64_NOMINAL_TFLOPS = 1.25  # GB300 dense FP64 (CUDA cores), nominal


def run_quantize(args):
    """Times the offline quantizer (round to nearest, MSE-optimal clipping) on
    one bf16 weight matrix, and the oracle on a column sample of it.  Its
    arithmetic is binary64 squared-error sums: 24 grid points x 128 weights x
    (multiply + add) per group of a column."""
    import numpy as np
    import torch

    import weight_only_int4_gemm_gb300 as w
    K, N = (int(v) for v in (args.shape or "4096x28672").split("x"))
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from __graft_entry__ import build
    build()
    g = torch.Generator().manual_seed(0)
    wt = (torch.randn((K, N), generator=g) * 0.02).to(torch.bfloat16)
    wd = wt.to(device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            w.w4a16_quantize_rtn(wd, stream=stream)
    stream.synchronize()
    steps = max(1, min(args.steps, 50))
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(steps):
                w.w4a16_quantize_rtn(wd, stream=stream)
            stop.record(stream)
        stop.synchronize()
    t = start.elapsed_time(stop) / 1e3 / steps
    in_bytes = K * N * 2
    flops64 = (K // 128) * N * 24 * 128 * 2
    line = {"metric": "W4A16 offline quantizer (RTN, MSE-optimal clipping), GB/s of bf16 weights",
            "value": in_bytes / t / 1e9, "unit": "GB/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "dtype": "bf16 in, f32 decisions, f64 error sums", "data": "synthetic N(0, 0.02)",
            "config": {"workload": "quantize", "shape_KxN": f"{K}x{N}", "group": 128, "grid": 24},
            "roofline": {"bound": "alu", "achieved": flops64 / t / 1e12,
                         "peak": FP64_NOMINAL_TFLOPS, "unit": "TFLOP/s (fp64)",
                         "frac": flops64 / t / 1e12 / FP64_NOMINAL_TFLOPS,
                         "peak_source": "nominal GB300 FP64"},
            "clocks": clk.summary(), "gpu_launches": steps}
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cols = min(N, 512)
        sub = np.ascontiguousarray(wt[:, :cols].view(torch.int16).numpy().view(np.uint16))
        t0 = time.perf_counter()
        oracle.quantize_rtn_mse(sub)
        t_cpu = (time.perf_counter() - t0) * N / cols
        line["cpu_baseline"] = {"value": in_bytes / t_cpu / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle",
                                "sample": f"{cols} of {N} columns, scaled by N/columns"}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- mixture of experts

MOE_EXPERTS, MOE_TOPK, MOE_HIDDEN, MOE_WIDTH = 128, 8, 2048, 768


def run_moe(args):
    """One mixture-of-experts layer's routed-expert GEMMs at decode: 128
    experts, top-8 routing, hidden 2048, expert width 768 -- the gate+up
    grouped GEMM (K=2048, N=2x768) and the down grouped GEMM (K=768, N=2048)
    over B tokens x 8 routed rows.  Uniform random routing (seeded); both
    GEMMs get seeded activations (the activation function between them is not
    part of this path).  Bytes: codes + scales of every expert that receives
    rows, plus x and y."""
    import numpy as np
    import torch

    import weight_only_int4_gemm_gb300 as w
    from weight_only_int4_gemm_gb300 import inputs
    tokens = args.batch or 64
    E, topk = MOE_EXPERTS, MOE_TOPK
    T = tokens * topk
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from __graft_entry__ import build
    build()
    shapes = [("gate_up", MOE_HIDDEN, 2 * MOE_WIDTH), ("down", MOE_WIDTH, MOE_HIDDEN)]
    offs = [inputs.make_routing(tokens, E, topk, seed=101 + i) for i in range(len(shapes))]
    n_copies = 2  # 2 x 311 MB of expert weights: every step streams from HBM
    weights, xs, ys, bytes_step, max_rows = [], [], [], 0, []
    for i, (lbl, K, N) in enumerate(shapes):
        reps = []
        for c in range(n_copies):
            packed, scales = [], []
            for e in range(E):
                qw, sc, _ = inputs.make_weights(K, N, seed=5000 * i + 97 * c + e, device=device)
                packed.append(w.w4a16_pack(qw))
                scales.append(sc)
            reps.append((torch.stack(packed), torch.stack(scales)))
        weights.append(reps)
        xs.append(inputs.make_activations(T, K, seed=40_000 + i, device=device))
        ys.append(torch.empty((T, N), dtype=torch.bfloat16, device=device))
        counts = offs[i][1:] - offs[i][:-1]
        active = int((counts > 0).sum())
        bytes_step += active * (K * N // 2 + (K // 128) * N * 2) + T * K * 2 + T * N * 2
        max_rows.append(int(counts.max()))
    dev_offs = [o.to(device) for o in offs]
    ws = torch.zeros(max(w.w4a16_grouped_workspace_bytes(T, E, m, K, N)
                         for m, (_, K, N) in zip(max_rows, shapes)) + 256,
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)

    def step(c, x_list=xs, y_list=ys):
        for i, (lbl, K, N) in enumerate(shapes):
            packed, scales = weights[i][c]
            w.w4a16_gemm_grouped(x_list[i], dev_offs[i], packed, scales, False, max_rows[i],
                                 out=y_list[i], workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for k in range(max(3, args.warmup)):
            step(k % n_copies)
    stream.synchronize()
    graphs = []
    for c in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(c)
        graphs.append(g)
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            graphs[k % n_copies].replay()
    stream.synchronize()
    steps = max(1, min(args.steps, 5000))
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clk:
        with torch.cuda.stream(stream):
            start.record(stream)
            for k in range(steps):
                graphs[k % n_copies].replay()
            stop.record(stream)
        stop.synchronize()
    assert w.w4a16_device_status() == 0, "device-side wait timed out during the bench"
    t = start.elapsed_time(stop) / 1e3 / steps
    hbm, _, _, peak_src = load_peaks()
    achieved = bytes_step / t / 1e9

    # end to end: host x and routing tables in, host y out, every step
    host_in = [x.cpu().pin_memory() for x in xs] + [o.pin_memory() for o in offs]
    host_out = [torch.empty_like(y, device="cpu").pin_memory() for y in ys]
    dev_in = list(xs) + dev_offs

    def e2e_step(c):
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        step(c)
        for h, d in zip(host_out, ys):
            h.copy_(d, non_blocking=True)

    with torch.cuda.stream(stream):
        for k in range(3):
            e2e_step(k % n_copies)
    stream.synchronize()
    e2e_graphs = []
    for c in range(n_copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_step(c)
        e2e_graphs.append(g)
    e_steps = max(3, min(steps, args.e2e_steps))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for k in range(e_steps):
            e2e_graphs[k % n_copies].replay()
        e1.record(stream)
    e1.synchronize()
    t_e2e = e0.elapsed_time(e1) / 1e3 / e_steps
    h2d = sum(h.numel() * h.element_size() for h in host_in)
    d2h = sum(h.numel() * h.element_size() for h in host_out)

    line = {"metric": "W4A16 mixture-of-experts layer (routed experts) µs/step & TB/s",
            "value": bytes_step / t / 1e12, "unit": "TB/s", "n_gpus": 1, "steps": steps,
            "warmup": args.warmup, "ms_per_step": t * 1e3, "us_per_step": t * 1e6,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded weights, uniform random top-8 routing)",
            "config": {"workload": "moe", "experts": E, "top_k": topk, "tokens": tokens,
                       "routed_rows": T, "hidden": MOE_HIDDEN, "expert_width": MOE_WIDTH,
                       "gemms": [f"{lbl} {K}x{N}" for lbl, K, N in shapes],
                       "max_rows": max_rows, "algorithmic_bytes_per_step": bytes_step,
                       "l2": f"expert weights rotated over {n_copies} copies (2 x 311 MB)",
                       "cuda_graph": True},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_source": f"{peak_src} hbm_gbs",
                         "kernel": "skinny (grouped)",
                         "traffic": traffic_from_profiles("skinny", "moe"),
                         "algorithmic_bytes_per_launch": bytes_step / len(shapes)},
            "clocks": clk.summary(), "gpu_launches": steps * len(shapes),
            "e2e": {"value": bytes_step / t_e2e / 1e12, "unit": "TB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": t_e2e * 1e3, "steps": e_steps}}
    if not args.no_cpu_baseline:
        import oracle
        oracle.build()
        t_cpu = 0.0
        cols_used = []
        for i, (lbl, K, N) in enumerate(shapes):
            cols = 16
            qws = [inputs.make_weights(K, cols, seed=e)[0].numpy().view(np.uint32)
                   for e in range(E)]
            scs = [inputs.make_weights(K, cols, seed=e)[1].view(torch.int16).numpy()
                   .view(np.uint16) for e in range(E)]
            xb = xs[i].cpu().view(torch.int16).numpy().view(np.uint16)
            t0 = time.perf_counter()
            oracle.gemm_grouped(xb, offs[i].numpy(), qws, scs)
            t_cpu += (time.perf_counter() - t0) * N / cols
            cols_used.append(cols)
        line["cpu_baseline"] = {"value": bytes_step / t_cpu / 1e12, "unit": "TB/s",
                                "cores": oracle.omp_threads(), "kind": "oracle",
                                "us_per_step": t_cpu * 1e6,
                                "sample": f"{cols_used} columns of each expert of the two "
                                          "grouped GEMMs (all rows, all K), scaled by N/columns"}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------- FP8 comparison

def run_fp8(args):
    """The three regimes on one GPU: one Llama-3-8B decoder layer's linear set
    at batch B as W8A8-FP8 (dynamic per-token activation quantisation + FP8
    tensor-core GEMM, per-channel weight scales), beside the same set as
    W4A16 and as plain bf16 (torch.matmul, i.e. cuBLAS).  One line per B; the
    line's value is the FP8 step time."""
    import torch

    import weight_only_int4_gemm_gb300 as w
    from weight_only_int4_gemm_gb300 import inputs
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    from __graft_entry__ import build
    build()
    hbm, tf_burst, tf_sust, peak_src = load_peaks()
    batches = [args.batch] if args.batch else [1, 16, 64, 128, 256, 512, 1024]
    n_copies = 2
    fp8_w, w4_w, bf_w = {}, {}, {}
    for lbl, K, N in LAYER:
        fp8_w[lbl], w4_w[lbl], bf_w[lbl] = [], [], []
        for c in range(n_copies):
            wt = inputs.make_dense_weight(K, N, seed=K + N + 7919 * c, device=device)
            wq, sw = w.w8a8_fp8_quantize_weight(wt)
            fp8_w[lbl].append((w.w8a8_fp8_pack_weight(wq), sw))
            del wq
            qw, sc, _ = inputs.make_weights(K, N, seed=K * 3 + N + 7919 * c, device=device)
            w4_w[lbl].append((w.w4a16_pack(qw), sc))
            bf_w[lbl].append(wt)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream(device)

    def time_graphs(step_fn, steps):
        graphs = []
        with torch.cuda.stream(stream):
            for c in range(n_copies):
                step_fn(c)
        stream.synchronize()
        for c in range(n_copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step_fn(c)
            graphs.append(g)
        with torch.cuda.stream(stream):
            for k in range(max(3, args.warmup)):
                graphs[k % n_copies].replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for k in range(steps):
                graphs[k % n_copies].replay()
            e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / steps * 1e3  # µs per step

    for B in batches:
        xs = {lbl: inputs.make_activations(B, K, seed=50 + K + N, device=device)
              for lbl, K, N in LAYER}
        xq = {lbl: (torch.empty((B, K), dtype=torch.uint8, device=device),
                    torch.empty(B, dtype=torch.float32, device=device)) for lbl, K, N in LAYER}
        ys = {lbl: torch.empty((B, N), dtype=torch.bfloat16, device=device) for lbl, K, N in LAYER}
        ws = torch.zeros(max(max(w.w8a8_fp8_workspace_bytes(B, K, N),
                                 w.w4a16_workspace_bytes(B, K, N)) for _, K, N in LAYER) + 256,
                         dtype=torch.uint8, device=device)

        def fp8_step(c):
            for lbl, K, N in LAYER:
                q, sxb = w.w8a8_fp8_quantize_act(xs[lbl], out=xq[lbl], stream=stream)
                wq, sw = fp8_w[lbl][c]
                w.w8a8_fp8_gemm(q, sxb, wq, sw, out=ys[lbl], workspace=ws, stream=stream)

        def fp8_gemm_step(c):  # activations already quantised: the GEMMs alone
            for lbl, K, N in LAYER:
                wq, sw = fp8_w[lbl][c]
                w.w8a8_fp8_gemm(xq[lbl][0], xq[lbl][1], wq, sw, out=ys[lbl], workspace=ws,
                                stream=stream)

        def w4_step(c):
            for lbl, K, N in LAYER:
                packed, sc = w4_w[lbl][c]
                w.w4a16_gemm(xs[lbl], packed, sc, False, N, out=ys[lbl], workspace=ws,
                             stream=stream)

        def bf16_step(c):
            for lbl, K, N in LAYER:
                torch.matmul(xs[lbl], bf_w[lbl][c], out=ys[lbl])

        steps = max(20, min(args.steps, 2000 if B <= 128 else 300))
        with ClockSampler(0) as clk:
            t_fp8 = time_graphs(fp8_step, steps)
        assert w.w4a16_device_status() == 0, "device-side wait timed out during the bench"
        t_fp8_gemm = time_graphs(fp8_gemm_step, steps)
        t_w4 = time_graphs(w4_step, steps)
        t_bf = time_graphs(bf16_step, steps)
        wbytes = sum(K * N + 4 * N for _, K, N in LAYER)
        abytes = sum(B * K * 2 + B * K * 2 + 4 * B + B * N * 2 for _, K, N in LAYER)
        flops = sum(2 * B * K * N for _, K, N in LAYER)
        fp8_peak = 2.0 * tf_sust
        memory_bound = (wbytes + abytes) / (hbm * 1e9) >= flops / (fp8_peak * 1e12)
        t = t_fp8 * 1e-6
        if memory_bound:
            ach = (wbytes + abytes) / t / 1e9
            roof = {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                    "frac": ach / hbm, "peak_source": f"{peak_src} hbm_gbs"}
        else:
            ach = flops / t / 1e12
            roof = {"bound": "tensor", "achieved": ach, "peak": fp8_peak, "unit": "TFLOP/s",
                    "frac": ach / fp8_peak,
                    "peak_source": f"{peak_src} bf16 sustained x 2 (nominal fp8/bf16 ratio)"}
        roof.update({"kernel": "fp8_gemm_kernel + fp8_quant_rows_kernel (whole step)",
                     "traffic": None, "algorithmic_bytes_per_step": wbytes + abytes})
        line = {"metric": "W8A8-FP8 linear set µs/step (comparison path), beside W4A16 and "
                          "bf16 cuBLAS", "value": t_fp8, "unit": "µs/step", "n_gpus": 1,
                "steps": steps, "warmup": args.warmup, "ms_per_step": t_fp8 / 1e3,
                "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
                "dtype": "e4m3 x e4m3 -> f32", "data": "synthetic (seeded; Llama-3-8B shapes)",
                "config": {"workload": "fp8", "batch": B,
                           "gemms": [f"{lbl} {K}x{N}" for lbl, K, N in LAYER],
                           "l2": f"weights rotated over {n_copies} copies", "cuda_graph": True},
                "compare": {"w4a16_us": t_w4, "bf16_cublas_us": t_bf,
                            "fp8_gemms_only_us": t_fp8_gemm,
                            "fp8_over_w4a16": t_fp8 / t_w4, "fp8_over_bf16": t_fp8 / t_bf},
                "tflops": flops / t / 1e12, "roofline": roof, "clocks": clk.summary(),
                "gpu_launches": steps * 2 * len(LAYER)}
        print(json.dumps(line), flush=True)
        del xs, xq, ys, ws


# --------------------------------------------------------------- main

def run_sweep_main(args, rank, world, local):
    """Default workload: the decode-step sweep (GPU arm, or the oracle as the
    reference arm)."""
    from weight_only_int4_gemm_gb300 import model
    batches = [args.batch] if args.batch else list(SWEEP_BATCHES)
    sbytes = sum(model.linear_bytes(B, K, N) for B in batches for _, K, N in sweep_layers())
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        sampler = SweepOracleSampler(batches)
        sampler.calibrate(min(2.0, 60.0 / (args.warmup + args.steps)))
        per_step, t_begin = [], time.perf_counter()
        for k in range(args.warmup + args.steps):
            if k > args.warmup and time.perf_counter() - t_begin > 150:
                break
            per_step.append(sampler.step())
        timed = per_step[args.warmup:] if len(per_step) > args.warmup else per_step[-1:]
        t_step = sum(timed) / len(timed)
        sample = sampler.describe(len(timed), time.perf_counter() - t_begin)
        line = {"impl": "reference", "metric": METRIC, "value": t_step * 1e6, "unit": "µs/step",
                "n_gpus": 1, "steps": len(timed), "warmup": args.warmup,
                "ms_per_step": t_step * 1e3, "us_per_step": t_step * 1e6,
                "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": "decode_sweep: full Llama-3-8B decode-step linear stream "
                                       "(32 layers + lm_head, 129 GEMMs) at every B of the sweep",
                           "batches": batches, "algorithmic_bytes_per_step": sbytes},
                "throughput": {"tb_s": sbytes / t_step / 1e12},
                "cpu_baseline": {"value": t_step * 1e6, "unit": "µs/step",
                                 "cores": oracle.omp_threads(), "kind": "oracle",
                                 "sample": sample, "extrapolated": True},
                "e2e": {"value": t_step * 1e6, "unit": "µs/step", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from __graft_entry__ import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
        build()
    per_b, step_ms, clocks, e2e_ms, h2d, d2h, e2e_steps = run_sweep(args, rank, world, device)
    line = sweep_line(args, per_b, step_ms, clocks, e2e_ms, h2d, d2h, e2e_steps, world, device)
    del per_b
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        sampler = SweepOracleSampler(batches)
        sampler.calibrate(args.cpu_budget / 4)
        t0 = time.perf_counter()
        runs = [sampler.step()]
        while time.perf_counter() - t0 < args.cpu_budget and len(runs) < 50:
            runs.append(sampler.step())
        t_cpu = statistics.median(runs)
        line["cpu_baseline"] = {"value": t_cpu * 1e6, "unit": "µs/step",
                                "cores": oracle.omp_threads(), "kind": "oracle",
                                "extrapolated": True,
                                "sample": sampler.describe(len(runs), time.perf_counter() - t0),
                                "tb_s": sbytes / t_cpu / 1e12}
        # the same oracle on one core, on a smaller column sample
        oracle.set_threads(1)
        sampler.cols = max(1, sampler.cols // 16)
        t1 = time.perf_counter()
        t_one = sampler.step()
        line["cpu_baseline"]["single_core"] = {
            "value": t_one * 1e6, "unit": "µs/step", "extrapolated": True,
            "sample": sampler.describe(1, time.perf_counter() - t1)}
        oracle.set_threads(oracle.omp_threads())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 20 for decode_sweep, 10000 otherwise)")
    ap.add_argument("--warmup", type=int, default=None,
                    help="untimed warm-up steps (default 5 for decode_sweep, 50 otherwise)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_sweep",
                    choices=["decode_sweep", "decode_layer", "single", "decode_step", "prefill",
                             "zp70b", "quantize", "moe", "fp8"])
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--shape", default=None, help="KxN for --workload single (default 4096x4096)")
    ap.add_argument("--e2e-steps", type=int, default=300)
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--force-path", choices=["skinny", "tcgen05"], default=None,
                    help="force one kernel path (ablations; default: the library's choice)")
    ap.add_argument("--per-gemm", action="store_true",
                    help="also time each distinct GEMM alone (table on stderr)")
    args = ap.parse_args()
    sweep = args.workload == "decode_sweep"
    if args.steps is None:
        args.steps = 20 if sweep else 10000
    if args.warmup is None:
        args.warmup = 5 if sweep else 50
    global FORCE
    FORCE = {"skinny": 0, "tcgen05": 1}.get(args.force_path, -1)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.workload == "quantize":
        run_quantize(args)
        return
    if args.workload == "fp8":
        if args.impl == "reference" or rank != 0:
            raise SystemExit("--workload fp8 runs our arm on one GPU only")
        run_fp8(args)
        return
    if args.workload == "moe":
        if args.impl == "reference" or rank != 0:
            raise SystemExit("--workload moe runs our arm on one GPU only")
        run_moe(args)
        return
    if sweep:
        run_sweep_main(args, rank, world, local)
        return
    gemms = workload(args.workload, args.batch, args.shape)
    sbytes, sflops = step_bytes_flops(gemms)
    hbm, tf_burst, tf_sust, peak_src = load_peaks()

    config = {"workload": args.workload, "gemms_per_step": len(gemms),
              "shapes_KxN": sorted({f"{K}x{N}" for _, _, K, N, _, _ in gemms}),
              "batches": sorted({B for _, B, _, _, _, _ in gemms}),
              "zero_points": any(g[4] for g in gemms), "group": 128,
              "algorithmic_bytes_per_step": sbytes, "flops_per_step": sflops}

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        sampler = OracleSampler(gemms)
        sampler.calibrate(min(5.0, 120.0 / (args.warmup + args.steps)))
        per_step = []
        t_begin = time.perf_counter()
        for k in range(args.warmup + args.steps):
            if k > args.warmup and time.perf_counter() - t_begin > 150:
                break
            per_step.append(sampler.step())
        timed = per_step[args.warmup:] if len(per_step) > args.warmup else per_step[-1:]
        t_step = sum(timed) / len(timed)
        sample = sampler.describe(len(timed), time.perf_counter() - t_begin)
        val = sbytes / t_step / 1e12
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TB/s",
                "n_gpus": 1, "steps": len(timed), "warmup": args.warmup,
                "ms_per_step": t_step * 1e3, "us_per_step": t_step * 1e6,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": val, "unit": "TB/s", "cores": oracle.omp_threads(),
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": val, "unit": "TB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)

    from __graft_entry__ import build
    if rank == 0 or world == 1:
        build()
    if world > 1:
        dist.barrier()
        build()

    import weight_only_int4_gemm_gb300 as w
    ms, clocks, paths, n_copies, (e2e_ms, eager_ms, e2e_steps, h2d, d2h), step_pct = \
        run_gpu(args, gemms, rank, world, device)
    ms, e2e_step_ms = reduce_times_over_ranks(ms, e2e_ms / e2e_steps, world, device)
    _, eager_step_ms = reduce_times_over_ranks(ms, eager_ms / e2e_steps, world, device)

    t_step = ms / 1e3 / args.steps
    value = aggregate_value(sbytes, world, t_step)
    # roofline for the dominant kernel: every launch of the step is one GEMM;
    # the graph replays them back to back, so the mean launch time is the
    # timed region over the launches
    from collections import Counter
    dom = Counter(paths).most_common(1)[0][0]
    dom_name = w.PATH_NAMES[dom]
    dom_idx = [i for i, p in enumerate(paths) if p == dom]
    if len(dom_idx) == len(gemms):
        dom_bytes, dom_flops = sbytes, sflops
        launch_s = t_step / len(gemms)
    else:
        dom_bytes, dom_flops = step_bytes_flops([gemms[i] for i in dom_idx])
        launch_s = t_step * len(dom_idx) / len(gemms) / len(dom_idx)  # apportioned
    per_launch_bytes = dom_bytes / len(dom_idx)
    per_launch_flops = dom_flops / len(dom_idx)
    # the bound is whichever side of the roofline the work sits on, not the kernel;
    # one GEMM timed alone is held to the burst bf16 peak, a step of many GEMMs
    # to the sustained one
    alone = args.workload == "single"
    tf_peak = tf_burst if alone else tf_sust
    memory_bound = per_launch_bytes / (hbm * 1e9) >= per_launch_flops / (tf_peak * 1e12)
    if memory_bound:
        achieved = per_launch_bytes / launch_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "peak_source": f"{peak_src} hbm_gbs"}
    else:
        achieved = per_launch_flops / launch_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tf_peak, "unit": "TFLOP/s",
                "frac": achieved / tf_peak,
                "peak_source": f"{peak_src} bf16 {'burst' if alone else 'sustained'}"}
    roof["kernel"] = dom_name
    roof["traffic"] = traffic_from_profiles(dom_name, args.workload)
    roof["algorithmic_bytes_per_launch"] = per_launch_bytes

    line = {"metric": METRIC, "value": value, "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
            "us_per_step": t_step * 1e6, "step_distribution": step_pct,
            "tflops": sflops * world / t_step / 1e12,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; Llama-3-8B shapes, no trained weights)",
            "config": dict(config, parallelism=f"replicas{world}",
                           l2=f"packed weights rotated over {n_copies} copies so each GEMM "
                              "streams from HBM (inputs larger than L2)",
                           paths=sorted({w.PATH_NAMES[p] for p in paths}),
                           cuda_graph=True),
            "roofline": roof, "clocks": clocks, "gpu_launches": args.steps * len(gemms),
            "e2e": {"value": sbytes * world / (e2e_step_ms / 1e3) / 1e12, "unit": "TB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "ms_per_step": e2e_step_ms,
                    "launch": "CUDA graph per weight rotation of: one H2D copy of the step's "
                              "inputs, the step's w4a16_gemm calls, one D2H copy of its outputs",
                    "eager": {"value": sbytes * world / (eager_step_ms / 1e3) / 1e12,
                              "ms_per_step": eager_step_ms,
                              "launch": "one Python w4a16_gemm call per GEMM, same copies"}}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        sampler = OracleSampler(gemms)
        sampler.calibrate(args.cpu_budget / 5)
        # at the column cap one sampled step may cost well under the budget:
        # repeat it until about cpu_budget seconds of oracle work are done
        t0 = time.perf_counter()
        runs = [sampler.step()]
        per = time.perf_counter() - t0
        n_runs = max(5, min(500, int(args.cpu_budget / max(per, 1e-3))))
        runs += [sampler.step() for _ in range(n_runs - 1)]
        t_cpu = statistics.median(runs)
        sample = sampler.describe(len(runs), time.perf_counter() - t0)
        line["cpu_baseline"] = {"value": sbytes / t_cpu / 1e12, "unit": "TB/s",
                                "cores": oracle.omp_threads(), "kind": "oracle", "sample": sample,
                                "us_per_step": t_cpu * 1e6}
        # the same oracle on one core, on a smaller column sample
        oracle.set_threads(1)
        sampler.cols = max(1, sampler.cols // 16)
        t1 = time.perf_counter()
        t_one = sampler.step()
        line["cpu_baseline"]["single_core"] = {
            "value": sbytes / t_one / 1e12, "unit": "TB/s", "us_per_step": t_one * 1e6,
            "sample": sampler.describe(1, time.perf_counter() - t1)}
        oracle.set_threads(oracle.omp_threads())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
