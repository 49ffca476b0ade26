#!/usr/bin/env python
"""Benchmark of the LLM.int8() decomposed matmul on B300.

Headline workload (one "step"): the 7B-like decode calls
  M in {1, 4, 16} x (K, N) in {(4096, 4096), (4096, 11008), (11008, 4096)},
X ~ N(0,1) fp16 with 0.1 % (at least 4) outlier columns, W ~ N(0, 0.02) fp16,
threshold 6.0 -- nine llmint8_matmul calls per step.  Metric: GB/s of
algorithmic bytes (Wq K*N + colScaleW 4N + outlier rows of W 2*n_o*N + X 2MK +
Y 2MN per call), against the measured HBM copy bandwidth.  Weights are held in
R replicas that rotate, so every weight matrix is evicted from L2 (126 MB)
before it is read again.

Also reported in the same JSON line: the 7B-like prefill calls (TOPS of the
whole call and of the GEMM stage against the measured dense fp16/bf16 peak),
the end-to-end number through host buffers, the CPU oracle baseline, SM clocks
sampled during the timed region, and the launch count.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from bit_quantization_matmul_row_b300 import synthetic  # noqa: E402

METRIC = "LLM.int8() matmul TOPS (prefill) & GB/s (decode) vs 1×B300 roofline"
WORKLOAD = ("7B-like decode: M in {1,4,16} x (K,N) in {(4096,4096),(4096,11008),(11008,4096)}; "
            "X ~N(0,1) fp16 with 0.1% (>=4) outlier columns of absmax U(20,60); W ~N(0,0.02) fp16; threshold 6.0")
FALLBACK_HBM = 6400.0
FALLBACK_BF16 = 1800.0
L2_BYTES = 126 * 2 ** 20


def alg_bytes(M, K, N, n_o):
    """Algorithmic bytes of one call: int8 weights, column scales, fp16 outlier rows of W, X, Y."""
    return K * N + 4 * N + 2 * n_o * N + 2 * M * K + 2 * M * N


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)),
                "measured")
    except Exception:
        return FALLBACK_HBM, FALLBACK_BF16, 1400.0, "fallback"


# ---------------------------------------------------------------------------- clocks

CLOCK_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms={period_ms}"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                self.samples.append((time.time(), float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [s for s in self.samples if t0 - 0.06 <= s[0] <= t1 + 0.06]
        note = None
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:2]
            note = "timed region shorter than the sampling period; nearest samples"
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = set()
        for s in inside:
            for name, flag in zip(names, s[3][1:]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": max(s[2] for s in inside),
               "reasons": sorted(reasons), "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ---------------------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms, world, device=None):
    """The slowest rank's time: a job of independent replicas ends when its last rank does."""
    if world <= 1:
        return float(ms)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank_step, steps, world, ms):
    """Whole-job throughput in units per second: what all ranks processed over the slowest rank's time."""
    return units_per_rank_step * steps * world / (ms * 1e-3)


# ---------------------------------------------------------------------------- CPU oracle

def cpu_oracle_time(cases_xw, n_sample_cols=None, min_seconds=10.0, max_reps=8):
    """Time the CPU oracle (A1..A5 per call, weights quantized beforehand) on the
    decode calls; optionally on the first n_sample_cols output columns only.
    Returns (bytes, seconds, reps, threads)."""
    import oracle
    oracle.build()
    prepared = []
    for (M, K, N, X, W) in cases_xw:
        Ws = W if n_sample_cols is None else np.ascontiguousarray(W[:, :n_sample_cols])
        prepared.append((M, K, Ws.shape[1], X, Ws, oracle.quantize_weight(Ws)))
    threads = oracle.default_threads()
    total_b, total_t, reps = 0, 0.0, 0
    while reps < max_reps and (total_t < min_seconds or reps == 0):
        for (M, K, N, X, Ws, wq) in prepared:
            t = time.perf_counter()
            r = oracle.llmint8_matmul(X, Ws, 6.0, wq=wq, nthreads=threads)
            total_t += time.perf_counter() - t
            total_b += alg_bytes(M, K, N, int(r["outliers"].size))
        reps += 1
    return total_b, total_t, reps, threads


# ---------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    cases = synthetic.decode_7b()
    data = []
    for c in cases:
        X, _ = c.x()
        W, _ = c.w()
        data.append((c.M, c.K, c.N, X, W))
    sample_cols = 512
    import oracle
    oracle.build()
    prepared = []
    for (M, K, N, X, W) in data:
        Ws = np.ascontiguousarray(W[:, :sample_cols])
        prepared.append((M, K, X, Ws, oracle.quantize_weight(Ws)))
    threads = oracle.default_threads()

    def step():
        b = 0
        for (M, K, X, Ws, wq) in prepared:
            r = oracle.llmint8_matmul(X, Ws, 6.0, wq=wq, nthreads=threads)
            b += alg_bytes(M, K, Ws.shape[1], int(r["outliers"].size))
        return b

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    b = 0
    for _ in range(args.steps):
        b += step()
    dt = time.perf_counter() - t
    value = b / dt / 1e9
    sample = (f"each step: the 9 decode calls (A1..A5 on the CPU oracle, weights pre-quantized) restricted "
              f"to the first {sample_cols} output columns")
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / max(args.steps, 1) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "calls_per_step": 9, "sample_cols": sample_cols},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- our arm

KERNEL_SOURCES = {  # the sources each timed kernel is compiled from
    "k_gemv_decode": ("gemv.cuh", "common.cuh"),
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(ROOT, "bit_quantization_matmul_row_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary
    (profiles/traffic.json), valid only while the kernel's sources are unchanged
    (hash match); else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        rec = json.load(open(p)).get(kernel)
        if rec and rec.get("source_sha256_16") == kernel_source_hash(kernel):
            return rec
    except Exception:
        pass
    return None


def run_ours(args, world, rank, local):
    import torch
    import torch.distributed as dist
    from bit_quantization_matmul_row_b300 import api

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    hbm_peak, bf16_peak, bf16_sust, peak_src = peaks()
    stream = torch.cuda.current_stream()

    # ---- inputs (resident in HBM), weights in R rotating replicas
    R = args.replicas
    cases = []
    for c in synthetic.decode_7b():
        X, _ = c.x()
        W, _ = c.w()
        Xd = torch.from_numpy(X).to(dev)
        Wd = torch.from_numpy(W).to(dev)
        Wq, sw = api.llmint8_quantize_weight(Wd)
        reps = [(Wq, sw, Wd)] + [(Wq.clone(), sw.clone(), Wd.clone()) for _ in range(R - 1)]
        ws = api.make_workspace(c.M, c.K, c.N, dev)
        Y = torch.empty((c.M, c.N), dtype=torch.float16, device=dev)
        cases.append(dict(c=c, X=X, Xd=Xd, reps=reps, ws=ws, Y=Y, W=W))
    torch.cuda.synchronize()
    # realised outlier counts (deterministic for these inputs) -> algorithmic bytes
    for d in cases:
        c = d["c"]
        api.llmint8_matmul(d["Xd"], c.threshold, *d["reps"][0], Y=d["Y"], workspace=d["ws"])
    torch.cuda.synchronize()
    step_bytes = 0
    for d in cases:
        c = d["c"]
        d["n_o"] = api.read_intermediates(d["ws"], c.M, c.K, c.N)["outlier_count"]
        d["bytes"] = alg_bytes(c.M, c.K, c.N, d["n_o"])
        step_bytes += d["bytes"]
    weight_set = sum(d["c"].K * d["c"].N for d in cases[:3])  # distinct (K,N) weights, one replica

    ncase = len(cases)
    # kernels per call (outlier scan, row quantization, GEMV) as the library plans them
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for d in cases:
        c = d["c"]
        d["kpc"] = api.llmint8_kernels_per_call(c.M, c.K, c.N, c.threshold)
        # the decode GEMV: one 16-column tile per CTA, or a persistent grid of two
        # CTAs per SM when M <= 8 and the tiles would need several waves
        d["kernel"] = "k_gemv_decode_tiles" if c.M <= 8 and c.N // 16 > 2 * sms else "k_gemv_decode"
    launches_per_step = sum(d["kpc"] for d in cases)

    # ---- one CUDA graph per step (the 9 llmint8_matmul calls), so the GPU is not
    # starved by host launch latency.  Inside a call the kernels overlap through
    # programmatic dependent launch; nothing is inserted between them here.
    def capture(gi, instrumented):
        g = torch.cuda.CUDAGraph()
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(ncase)] if instrumented else None
        with torch.cuda.graph(g):
            for ci, d in enumerate(cases):
                c = d["c"]
                Wq, sw, Wd = d["reps"][(gi * ncase + ci) % R]
                if instrumented:  # xpass, [event], GEMV, [event]
                    api.llmint8_xpass(d["Xd"], c.threshold, c.N, d["ws"])
                    evs[ci][0].record()
                    api.llmint8_gemm(d["Xd"], c.threshold, Wq, sw, Wd, d["Y"], d["ws"])
                    evs[ci][1].record()
                else:
                    api.llmint8_matmul(d["Xd"], c.threshold, Wq, sw, Wd, Y=d["Y"], workspace=d["ws"])
        return g, evs

    G = min(args.steps, args.max_graphs)
    graphs = [capture(gi, False) for gi in range(G)]
    torch.cuda.synchronize()
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    sampler = ClockSampler(local)
    time.sleep(0.3)
    for i in range(args.warmup):
        graphs[i % G][0].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev_a.record(stream)
    for i in range(args.steps):
        graphs[i % G][0].replay()
    ev_b.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    elapsed_ms = ev_a.elapsed_time(ev_b)
    del graphs
    # dominant kernel: the same steps with event nodes around every GEMV (this
    # separates the GEMV from its X pass, so it runs without their overlap)
    G = min(args.steps, args.max_graphs, 64)
    igraphs = [capture(gi, True) for gi in range(G)]
    for i in range(args.warmup):
        igraphs[i % G][0].replay()
    torch.cuda.synchronize()
    for i in range(G):
        igraphs[i][0].replay()
    torch.cuda.synchronize()
    gemv_ms = [[e0.elapsed_time(e1) for (e0, e1) in igraphs[gi][1]] for gi in range(G)]
    del igraphs
    # ... and back to back: per shape, one captured graph of B consecutive
    # llmint8_gemm calls (A3-A5) on a workspace its X pass filled beforehand,
    # weights rotating through the replicas; consecutive GEMVs overlap through
    # programmatic dependent launch as they do inside a step.  Events around the
    # replays; per launch = elapsed / launches.
    B, GR = 4 * R, 8
    b2b_us = []
    for d in cases:
        c = d["c"]
        api.llmint8_xpass(d["Xd"], c.threshold, c.N, d["ws"])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for r in range(B):
                Wq, sw, Wd = d["reps"][r % R]
                api.llmint8_gemm(d["Xd"], c.threshold, Wq, sw, Wd, d["Y"], d["ws"])
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        ev_a.record(stream)
        for _ in range(GR):
            g.replay()
        ev_b.record(stream)
        torch.cuda.synchronize()
        b2b_us.append(1e3 * ev_a.elapsed_time(ev_b) / (B * GR))
        del g
    st = api.llmint8_device_status(cases[0]["ws"])
    if st != 0:
        raise SystemExit(f"device error word {st}")
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    total_bytes = step_bytes * args.steps * world
    value = job_rate(step_bytes, args.steps, world, elapsed_ms) / 1e9
    iso_us = [1e3 * sum(gemv_ms[gi][ci] for gi in range(G)) / G for ci in range(ncase)]
    per_shape = [{"M": d["c"].M, "K": d["c"].K, "N": d["c"].N, "outliers": d["n_o"], "kernel": d["kernel"],
                  "bytes": d["bytes"], "kernel_us": b2b_us[ci], "kernel_gbs": d["bytes"] / (b2b_us[ci] * 1e-6) / 1e9,
                  "frac": d["bytes"] / (b2b_us[ci] * 1e-6) / 1e9 / hbm_peak,
                  "isolated_us": iso_us[ci], "isolated_gbs": d["bytes"] / (iso_us[ci] * 1e-6) / 1e9}
                 for ci, d in enumerate(cases)]
    dom = "k_gemv_decode"  # both forms (k_gemv_decode, k_gemv_decode_tiles) come from gemv.cuh
    launch_bytes = sum(d["bytes"] for d in cases) / ncase
    launch_us = sum(b2b_us) / ncase
    achieved = launch_bytes / (launch_us * 1e-6) / 1e9
    iso_launch_us = sum(iso_us) / ncase
    kernels = {dom: {"launches_timed": ncase * B * GR, "launch_us_avg": launch_us,
                     "alg_bytes_per_launch": launch_bytes, "achieved_gbs": achieved,
                     "time_share_of_step": ncase * launch_us * 1e-3 / (elapsed_ms / args.steps),
                     "isolated_launch_us_avg": iso_launch_us,
                     "isolated_achieved_gbs": launch_bytes / (iso_launch_us * 1e-6) / 1e9}}
    time.sleep(0.1)

    # ---- end to end through the public call: pinned host X -> device,
    # llmint8_matmul, Y -> pinned host; eager (each call from Python) and as a graph
    hX = [torch.from_numpy(d["X"]).pin_memory() for d in cases]
    hY = [torch.empty((d["c"].M, d["c"].N), dtype=torch.float16).pin_memory() for d in cases]
    h2d = sum(d["X"].nbytes for d in cases)
    d2h = sum(d["c"].M * d["c"].N * 2 for d in cases)

    def e2e_step(i):
        # the public host-buffer call: X_host -> device, A1..A5, Y -> Y_host, one C call per matmul
        for ci, d in enumerate(cases):
            c = d["c"]
            Wq, sw, Wd = d["reps"][(i * ncase + ci) % R]
            api.llmint8_matmul_host(hX[ci], d["Xd"], c.threshold, Wq, sw, Wd, d["Y"], hY[ci], d["ws"])

    def timed(fn, n):
        for i in range(args.warmup):
            fn(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ev_a.record()
        for i in range(n):
            fn(i)
        ev_b.record()
        torch.cuda.synchronize()
        return max_over_ranks(ev_a.elapsed_time(ev_b), world, dev)

    e2e_ms = timed(e2e_step, args.steps)
    e2e_value = total_bytes / (e2e_ms * 1e-3) / 1e9
    G2 = min(args.steps, 8)
    e2e_graphs = []
    for gi in range(G2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_step(gi)
        e2e_graphs.append(g)
    e2e_graph_ms = timed(lambda i: e2e_graphs[i % G2].replay(), args.steps)
    e2e_graph_value = total_bytes / (e2e_graph_ms * 1e-3) / 1e9
    del e2e_graphs
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)

    # ---- prefill calls (context in the same line): TOPS of the call and of the GEMM stage
    prefill = None
    if not args.no_prefill:
        prefill = run_prefill(args, dev, stream, bf16_peak, peak_src)
    chain = None
    if not args.no_chain:
        chain = run_chain(args, dev, stream)
    sweep = None
    if not args.no_sweep:
        sweep = run_sweep(args, dev, stream, hbm_peak, bf16_peak, peak_src)

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu:
            b, t, reps, threads = cpu_oracle_time([(d["c"].M, d["c"].K, d["c"].N, d["X"], d["W"]) for d in cases])
            cpu = {"value": b / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
                   "sample": f"the 9 decode calls of one step, repeated {reps}x ({t:.1f} s of oracle time; "
                             f"A1..A5 per call, weights quantized beforehand)"}
        trec = traffic_record(dom)
        traffic = None if trec is None else trec["dram_bytes_per_launch"]
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "s8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "calls_per_step": ncase, "weight_replicas": R,
                       "launch": "each step is one CUDA graph of the 9 calls (replayed; captured beforehand)",
                       "l2": (f"inputs larger than L2: {R} rotating weight replicas; each matrix is re-read only "
                              f"after >= {(R - 1) * weight_set / 2**20:.0f} MB of other weights (L2 126 MB)"),
                       "outliers_per_call": [d["n_o"] for d in cases], "bytes_per_step": step_bytes},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": traffic, "kernel": dom,
                         "alg_bytes_per_launch": kernels[dom]["alg_bytes_per_launch"],
                         "launch_us_avg": kernels[dom]["launch_us_avg"],
                         "launches_timed": kernels[dom]["launches_timed"],
                         "timing": ("CUDA events around replays of one captured graph per decode shape holding "
                                    f"{B} consecutive llmint8_gemm calls (A3-A5; X pass run once before; weights "
                                    "rotating through the replicas; PDL between the launches, as inside a step); "
                                    "per launch = elapsed / launches, averaged over the 9 shapes.  isolated_*: "
                                    "events around each GEMV launch inside captured steps, which adds the launch "
                                    "latency (~5 us on this part for an empty kernel) that PDL hides in a step"),
                         "peak_source": f"{peak_src} hbm_gbs (copy, burst)", "kernels": kernels,
                         "per_shape": per_shape},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": "eager: each call issued from Python through the public llmint8_matmul_host "
                            "(pinned host X copied in, Y copied out, inside the call)",
                    "graph_value": e2e_graph_value},
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks,
        }
        if prefill is not None:
            line["prefill"] = prefill
        if chain is not None:
            line["chain"] = chain
        if sweep is not None:
            line["sweep"] = sweep
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return line


def run_prefill(args, dev, stream, bf16_peak, peak_src, iters=None):
    import torch
    from bit_quantization_matmul_row_b300 import api
    iters = iters or max(5, min(50, args.steps))
    out = []
    tot_flop, tot_call_ms, tot_gemm_ms = 0.0, 0.0, 0.0
    for c in synthetic.prefill_7b():
        X, _ = c.x()
        W, _ = c.w()
        Xd = torch.from_numpy(X).to(dev)
        Wd = torch.from_numpy(W).to(dev)
        Wq, sw = api.llmint8_quantize_weight(Wd)
        reps = [(Wq, sw, Wd), (Wq.clone(), sw.clone(), Wd.clone())]
        ws = api.make_workspace(c.M, c.K, c.N, dev)
        Y = torch.empty((c.M, c.N), dtype=torch.float16, device=dev)
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(iters)]

        def call(i, timed):  # the public call, as a user runs it
            Wq_, sw_, Wd_ = reps[i % 2]
            if timed:
                e0[i].record(stream)
            api.llmint8_matmul(Xd, c.threshold, Wq_, sw_, Wd_, Y=Y, workspace=ws, stream=stream)
            if timed:
                e1[i].record(stream)

        def split(i, timed):  # its two halves, with events around the GEMM stage
            Wq_, sw_, Wd_ = reps[i % 2]
            api.llmint8_xpass(Xd, c.threshold, c.N, ws, stream=stream)
            if timed:
                e0[i].record(stream)
            api.llmint8_gemm(Xd, c.threshold, Wq_, sw_, Wd_, Y, ws, stream=stream)
            if timed:
                e1[i].record(stream)

        def timed_ms(fn):
            for i in range(3):
                fn(i, False)
            torch.cuda.synchronize()
            for i in range(iters):
                fn(i, True)
            torch.cuda.synchronize()
            return sum(e0[i].elapsed_time(e1[i]) for i in range(iters)) / iters

        call_ms = timed_ms(call)
        gemm_ms = timed_ms(split)
        flop = 2.0 * c.M * c.N * c.K
        n_o = api.read_intermediates(ws, c.M, c.K, c.N)["outlier_count"]
        out.append({"shape": [c.M, c.K, c.N], "outliers": n_o, "call_us": call_ms * 1e3, "gemm_us": gemm_ms * 1e3,
                    "tops_call": flop / (call_ms * 1e-3) / 1e12, "tops_gemm": flop / (gemm_ms * 1e-3) / 1e12})
        tot_flop += flop
        tot_call_ms += call_ms
        tot_gemm_ms += gemm_ms
        del reps, Wq, sw, Wd, Xd, ws, Y
    torch.cuda.empty_cache()
    tops = tot_flop / (tot_call_ms * 1e-3) / 1e12
    tops_gemm = tot_flop / (tot_gemm_ms * 1e-3) / 1e12
    return {"workload": "7B-like prefill: M=2048, K=4096, N in {4096, 11008}; 0.1% outlier columns; t=6.0",
            "value": tops, "unit": "TOPS", "iters": iters,
            "roofline": {"bound": "tensor", "achieved": tops_gemm, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": tops_gemm / bf16_peak, "kernel": "k_gemm_tc",
                         "stage": "llmint8_gemm: k_widen_codes (int8 codes -> fp16 scratch) then k_gemm_tc",
                         "peak_source": f"{peak_src} bf16_tflops (cuBLAS, burst); tcgen05 kind::f16 runs at the "
                                        "bf16 rate; sm_103a has no int8 tcgen05 kind"},
            "shapes": out}


def run_sweep(args, dev, stream, hbm_peak, bf16_peak, peak_src):
    """The larger configurations: the 13B-like FFN (M=4096, (K,N) in {(5120,13824),(13824,5120)}, 1 %
    outlier columns of absmax U(20,100), 0.5 % of W's columns x10) and the 70B-like sweep (K=8192,
    N in {8192, 28672}, M in {1,16,256,2048,8192}, outlier fractions 0 / 0.1 / 1 / 5 % of absmax
    U(20,60), W ~N(0,0.015)), plus, per (M, N), plain int8 (threshold +inf) and the fp16 matmul
    (cuBLAS through torch.matmul, context).  Each number: CUDA events around n consecutive public
    calls (after warm-up), weights rotating through replicas so that every call reads them from
    HBM.  X is drawn once per (M, fraction) and W once per (K, N) (the first case's seed).
    Metric per row: TOPS = 2MNK / t for M > 16 (against the bf16 peak: sm_103a has no int8 tcgen05
    kind), GB/s of algorithmic bytes for M <= 16 (against the HBM copy peak)."""
    import torch
    from bit_quantization_matmul_row_b300 import api
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, n, warm=3):
        for i in range(warm):
            fn(i)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return 1e3 * e0.elapsed_time(e1) / n  # us per call

    groups = {}
    for c in synthetic.ffn_13b() + synthetic.sweep_70b():
        groups.setdefault((c.K, c.N, c.sigma, c.boosted_frac), []).append(c)
    xcache = {}
    rows = []
    for (K, N, _, _), cs in groups.items():
        W, _ = cs[0].w()
        Wd = torch.from_numpy(W).to(dev)
        del W
        Wq, sw = api.llmint8_quantize_weight(Wd)
        R2 = max(2, -(-3 * L2_BYTES // (K * N)))  # replicas: >= 3 x L2 of int8 weights between re-reads
        R2 = min(R2, 4)
        reps = [(Wq, sw, Wd)] + [(Wq.clone(), sw.clone(), Wd.clone()) for _ in range(R2 - 1)]
        for c in cs:
            key = (c.M, K, c.frac, c.mag)
            if key not in xcache:
                xcache.clear()
                xcache[key] = torch.from_numpy(c.x()[0]).to(dev)
            Xd = xcache[key]
            M = c.M
            ws = api.make_workspace(M, K, N, dev)
            Y = torch.empty((M, N), dtype=torch.float16, device=dev)
            n = 20 if M <= 256 else (10 if M <= 2048 else 5)
            dec = M <= 16

            def call(i, t=c.threshold):
                Wq_, sw_, Wd_ = reps[i % R2]
                api.llmint8_matmul(Xd, t, Wq_, sw_, Wd_, Y=Y, workspace=ws, stream=stream)

            us = timed(call, n)
            n_o = api.read_intermediates(ws, M, K, N)["outlier_count"]
            flop = 2.0 * M * N * K
            row = {"case": c.name, "M": M, "K": K, "N": N, "outlier_frac": c.frac, "outliers": n_o, "us": us,
                   "tops": flop / (us * 1e-6) / 1e12}
            if dec:
                gbs = alg_bytes(M, K, N, n_o) / (us * 1e-6) / 1e9
                row.update(gbs=gbs, bound="hbm", frac=gbs / hbm_peak, kernel="k_gemv_decode")
            else:
                row.update(bound="tensor", frac=row["tops"] / bf16_peak, kernel="k_gemm_tc")
            if c.frac == 0.001 or (c.frac == 0.01 and K != 8192):
                # per (M, N): plain int8 and the fp16 matmul on the same X
                row["int8_t_inf_us"] = timed(lambda i: call(i, float("inf")), n)
                row["fp16_cublas_us"] = timed(lambda i: torch.matmul(Xd, reps[i % R2][2], out=Y), n)
            rows.append(row)
            del ws, Y
        del reps, Wq, sw, Wd
        xcache.clear()
        torch.cuda.empty_cache()
    return {"workloads": ["13B-like FFN: M=4096, (K,N) in {(5120,13824),(13824,5120)}; 1% outlier columns "
                          "U(20,100); W ~N(0,0.02) with 0.5% columns x10; t=6.0",
                          "70B-like sweep: K=8192, N in {8192,28672}, M in {1,16,256,2048,8192}; outlier "
                          "fraction in {0, 0.1%, 1%, 5%} U(20,60); W ~N(0,0.015); t=6.0; plus t=+inf and "
                          "fp16 cuBLAS per (M, N)"],
            "timing": "CUDA events around n consecutive public llmint8_matmul calls (n = 20 / 10 / 5 for "
                      "M <= 256 / 2048 / 8192), weights rotating through replicas (inputs larger than L2)",
            "peaks": {"hbm_gbs": hbm_peak, "bf16_tflops": bf16_peak, "source": peak_src},
            "rows": rows}


def run_chain(args, dev, stream, steps=None):
    """Decode chain: the three 7B-like layers (4096, 4096) -> (4096, 11008) -> (11008, 4096), each
    output the next input, for M = 1 and 4.  One step = the 3 calls as one captured graph, weights in
    rotating replicas; the chained calls (llmint8_matmul_chain: one kernel per layer after the
    first) against the same flow through llmint8_matmul (X pass + GEMV per layer).  Two weight
    recipes: the decode workload's W (N(0, 0.02): the layers' outputs carry a few % outlier
    columns at t = 6), and unit-variance W (N(0, 1/sqrt(K))) whose 0.1 % boosted output columns
    (x10) give the next layer's X a few systematic outlier features, like the X generator's."""
    import torch
    from bit_quantization_matmul_row_b300 import api
    steps = steps or max(20, min(200, args.steps))
    R = args.replicas
    cases = {(c.M, c.K, c.N): c for c in synthetic.decode_7b()}
    layers = [(4096, 4096), (4096, 11008), (11008, 4096)]

    def weights(recipe):
        wts = []
        for li, (K, N) in enumerate(layers):
            if recipe == "decode7b_weights":
                W, _ = cases[(1, K, N)].w()
            else:
                W, _ = synthetic.make_w(K, N, sigma=1.0 / math.sqrt(K), boosted_frac=0.001, boost=10.0,
                                        seed=7000 + li)
            Wd = torch.from_numpy(W).to(dev)
            Wq, sw = api.llmint8_quantize_weight(Wd)
            wts.append([(Wq, sw, Wd)] + [(Wq.clone(), sw.clone(), Wd.clone()) for _ in range(R - 1)])
        return wts

    results = {}
    for recipe in ("decode7b_weights", "unit_variance_feature_outliers"):
        wts = weights(recipe)
        out = {}
        for M in (1, 4):
            c0 = cases[(M, 4096, 4096)]
            X0 = torch.from_numpy(c0.x()[0]).to(dev)
            t = c0.threshold
            Ys = [torch.empty((M, N), dtype=torch.float16, device=dev) for _, N in layers]
            states = [api.make_chain_state(M, N, dev) for _, N in layers]
            wss = [api.make_workspace(M, K, N, dev) for K, N in layers]

            def chained(r):
                x, s_in = X0, None
                for li in range(len(layers)):
                    Wq, sw, Wd = wts[li][r % R]
                    api.llmint8_matmul_chain(x, t, s_in, Wq, sw, Wd, next_threshold=t, state_out=states[li],
                                             Y=Ys[li], workspace=wss[li])
                    x, s_in = Ys[li], states[li]

            def separate(r):
                x = X0
                for li in range(len(layers)):
                    Wq, sw, Wd = wts[li][r % R]
                    api.llmint8_matmul(x, t, Wq, sw, Wd, Y=Ys[li], workspace=wss[li])
                    x = Ys[li]

            res = {}
            for name, fn in (("separate", separate), ("chained", chained)):
                fn(0)
                torch.cuda.synchronize()
                graphs = []
                for r in range(R):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g):
                        fn(r)
                    graphs.append(g)
                for i in range(3 * R):
                    graphs[i % R].replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record(stream)
                for i in range(steps):
                    graphs[i % R].replay()
                e1.record(stream)
                torch.cuda.synchronize()
                res[name] = e0.elapsed_time(e1) / steps * 1e3  # us per step
                del graphs
            # algorithmic bytes of the step, with the outlier counts the separate flow found
            separate(0)
            torch.cuda.synchronize()
            nbytes, counts = 0, []
            for li, (K, N) in enumerate(layers):
                n_o = api.read_intermediates(wss[li], M, K, N)["outlier_count"]
                counts.append(int(n_o))
                nbytes += alg_bytes(M, K, N, n_o)
            out[f"M{M}"] = {"chained_us": res["chained"], "separate_us": res["separate"],
                            "chained_gbs": nbytes / (res["chained"] * 1e-6) / 1e9,
                            "separate_gbs": nbytes / (res["separate"] * 1e-6) / 1e9,
                            "speedup": res["separate"] / res["chained"], "bytes_per_step": nbytes,
                            "outliers_per_layer": counts}
        results[recipe] = out
        del wts
        torch.cuda.empty_cache()
    return {"workload": "7B-like decode chain: (4096,4096) -> (4096,11008) -> (11008,4096), each Y the next X; "
                        "M in {1, 4}; t=6.0 for every layer",
            "steps": steps, "unit": "GB/s", "timing": "events around replays of one captured graph per step",
            "results": results}


def run_ablation(args):
    """Error vs speed of the LLM.int8() decomposition (with the fp16 copy of W, and
    with int8 weights only) against plain vector-wise int8
    (threshold +inf: no outlier decomposition) and the fp16 matmul (cuBLAS, context),
    on the synthetic outlier workloads.  Error: relative Frobenius distance to the
    exact product (fp64 on the GPU).  Times: CUDA events around single calls."""
    import torch
    from bit_quantization_matmul_row_b300 import api
    dev = torch.device("cuda")
    torch.cuda.set_device(0)
    cases = [("decode 7B M=1 4096x4096 0.1%", 1, 4096, 4096, 0.001),
             ("decode 7B M=16 4096x11008 0.1%", 16, 4096, 11008, 0.001),
             ("prefill 7B M=2048 4096x4096 0.1%", 2048, 4096, 4096, 0.001)]
    for f in (0.0, 0.001, 0.01, 0.05):
        cases.append((f"70B M=256 8192x8192 {100 * f:g}%", 256, 8192, 8192, f))
    R = 4  # rotating weight replicas: every timed call streams its weights from HBM
    rows = []
    for name, M, K, N, frac in cases:
        X, _ = synthetic.make_x(M, K, frac=frac, min_count=4 if frac > 0 else 0, seed=M + K + N)
        W, _ = synthetic.make_w(K, N, sigma=0.015 if K == 8192 else 0.02, seed=M + K + N)
        Xd, Wd = torch.from_numpy(X).to(dev), torch.from_numpy(W).to(dev)
        Wq, sw = api.llmint8_quantize_weight(Wd)
        reps = [(Wq, sw, Wd)] + [(Wq.clone(), sw.clone(), Wd.clone()) for _ in range(R - 1)]
        ws = api.make_workspace(M, K, N, dev)
        exact = Xd.double() @ Wd.double()
        variants = {
            "llmint8_t6": lambda r: api.llmint8_matmul(Xd, 6.0, r[0], r[1], r[2], workspace=ws),
            # no fp16 copy of W kept: the outlier rows come from the dequantized codes
            "llmint8_t6_int8_weights": lambda r: api.llmint8_matmul_w8(Xd, 6.0, r[0], r[1], workspace=ws),
            "int8_no_outliers": lambda r: api.llmint8_matmul_int8(Xd, r[0], r[1], workspace=ws),
            "fp16_cublas": lambda r: torch.matmul(Xd, r[2]),
        }
        row = {"case": name, "M": M, "K": K, "N": N, "outlier_frac": frac}
        for key, fn in variants.items():
            Y = fn(reps[0])
            torch.cuda.synchronize()
            err = float(torch.linalg.norm(Y.double() - exact) / torch.linalg.norm(exact))
            if key == "llmint8_t6":
                row["n_outliers"] = api.read_intermediates(ws, M, K, N)["outlier_count"]
            for i in range(5):
                fn(reps[i % R])
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(20):
                fn(reps[i % R])
            e1.record()
            torch.cuda.synchronize()
            row[key] = {"rel_error": err, "us": 1e3 * e0.elapsed_time(e1) / 20}
        rows.append(row)
        del Xd, Wd, Wq, sw, reps, ws, exact
        torch.cuda.empty_cache()
    print(json.dumps({"ablation": rows, "data": "synthetic", "note": (
        "per-tensor scales change only the scale arrays, not the kernels' work, so their speed is the "
        "vector-wise path's; their error is measured with the CPU oracle in the tests")}), flush=True)


def run_profile(args):
    """Eager calls of one named case (warmup + steps), for profiler captures."""
    import torch
    from bit_quantization_matmul_row_b300 import api
    allc = {c.name: c for c in (synthetic.tiny() + synthetic.decode_7b() + synthetic.prefill_7b() +
                                 synthetic.ffn_13b() + synthetic.sweep_70b())}
    if args.profile not in allc:
        raise SystemExit(f"unknown case {args.profile}; known: {sorted(allc)}")
    c = allc[args.profile]
    X, _ = c.x()
    W, _ = c.w()
    dev = torch.device("cuda")
    Xd, Wd = torch.from_numpy(X).to(dev), torch.from_numpy(W).to(dev)
    Wq, sw = api.llmint8_quantize_weight(Wd)
    ws = api.make_workspace(c.M, c.K, c.N, dev)
    Y = torch.empty((c.M, c.N), dtype=torch.float16, device=dev)
    for _ in range(args.warmup):
        api.llmint8_matmul(Xd, c.threshold, Wq, sw, Wd, Y=Y, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        api.llmint8_matmul(Xd, c.threshold, Wq, sw, Wd, Y=Y, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    st = api.llmint8_device_status(ws)
    print(json.dumps({"profile": c.name, "calls": args.steps, "us_per_call": 1e3 * e0.elapsed_time(e1) / args.steps,
                      "status": st}), flush=True)
    if st != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--replicas", type=int, default=4)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-chain", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the 13B FFN / 70B sweep shapes")
    ap.add_argument("--max-graphs", type=int, default=256)
    ap.add_argument("--ablation", action="store_true",
                    help="error vs speed: LLM.int8() against plain int8 and the fp16 matmul (one JSON line)")
    ap.add_argument("--profile", metavar="CASE", default=None,
                    help="run only the named synthetic case (eager calls; for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.profile:
        run_profile(args)
        return
    if args.ablation:
        run_ablation(args)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
