#!/usr/bin/env python3
"""Benchmark of the block-scaled FP4 hot path on one GB300 (or N replicas).

One step = one pass of the whole path over one batch of synthetic input, for
the square NVFP4 GEMM M = N = K = 8192:
  global scale of the BF16 activations (amax / (6*448))      qfp4_global_scale
  BF16 -> NVFP4 quantisation, scale factors written straight   qfp4_quantize
    into the tensor-core layout (the interleave step fused)
  tensor-core GEMM with the global-scale epilogue -> BF16      qfp4_gemm_nt
against NVFP4 weights (N(0, 0.02)) quantised once beforehand.  The metric is
effective TFLOP/s = 2*M*N*K / step time.  Between steps L2 is flushed by a
read-only pass over a buffer of 4x its size (no dirty lines are left to be
written back inside the next step).  The K timed steps follow a soak of a few
seconds of the same steps; SM clocks are sampled over both, and the GEMM's
median and minimum time over all of them feed the roofline.

Also reported on the same JSON line: the roofline of the dominant kernel
(the GEMM), the CPU oracle timed on a bounded sample ("cpu_baseline"), the
end-to-end number through host buffers ("e2e"), SM clocks sampled during the
timed region, and a sweep of the other workloads (decode GEMMs and the
quantiser in GB/s against HBM, the compute-bound sweep and the grouped MoE
GEMM in TFLOP/s against the FP4 tensor peak).

Multi-GPU: the path has no exchange step, so N GPUs run N independent
replicas (weak scaling, no collective on the data path).

--impl reference times the CPU oracle instead (bounded samples per step).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_scaled_fp4_tcgen05_gb300 import synth  # noqa: E402

METRIC = "NVFP4/MXFP4 GEMM eff. TFLOP/s (2MNK) & % FP4 peak; decode/quantize HBM GB/s"
CASE = synth.SQUARE_NV
PAGES_BASELINE_TFLOPS = 1045.0     # quadbit dense FP4, square 8192, RTX PRO 6000 (SM120)
FP4_OVER_BF16 = 13.5 / 2.25        # nominal dense FP4 : BF16 tensor rate on GB300
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "block_scaled_fp4_tcgen05_gb300", "csrc")
FLUSH_BYTES = 512 << 20
SOAK_SECONDS = 2.5                 # clock-sampled steps ahead of the K timed ones


# --------------------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device) -> float:
    """Max over ranks (identity for one process)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel source changed since the counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            data = json.load(f)
        ent = data[kernel_key]
        if ent.get("source_sha") != file_sha(os.path.join(CSRC, ent["source"])):
            return None
        return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- GPU arm

class Pipeline:
    """Device buffers and the launches of one step for a GEMM case."""

    def __init__(self, case, device, with_weights=True):
        import torch
        from block_scaled_fp4_tcgen05_gb300 import qfp4
        self.q, self.torch, self.case, self.dev = qfp4, torch, case, device
        M, N, K, fmt = case.M, case.N, case.K, case.fmt
        g = qfp4.block_size(fmt)
        self.g = g
        xa = synth.activations_bf16(case.seed, M, K)
        self.X_host = torch.from_numpy(xa.view(np.int16).copy()).view(torch.bfloat16)
        self.X = self.X_host.to(device)
        self.X_pinned = self.X_host.pin_memory()
        self.gs_a = torch.ones(1, dtype=torch.float32, device=device)
        self.Qa = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
        self.SFa = torch.empty(qfp4.sf_mma_bytes(M, K // g), dtype=torch.uint8, device=device)
        self.D = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.D_pinned = torch.empty((M, N), dtype=torch.bfloat16).pin_memory()
        self.ws_bytes = qfp4.gemm_workspace_bytes(fmt, M, N, K)
        self.ws = torch.zeros(max(self.ws_bytes, 16), dtype=torch.uint8, device=device)
        if with_weights:
            xw = synth.weights_bf16(case.seed + 1000, N, K)
            W = torch.from_numpy(xw.view(np.int16).copy()).view(torch.bfloat16).to(device)
            self.gs_b = torch.ones(1, dtype=torch.float32, device=device)
            self.Qb = torch.empty((N, K // 2), dtype=torch.uint8, device=device)
            self.SFb = torch.empty(qfp4.sf_mma_bytes(N, K // g), dtype=torch.uint8, device=device)
            if fmt == qfp4.NVFP4:
                qfp4.global_scale(W, self.gs_b)
            qfp4.quantize(fmt, W, self.gs_b, self.Qb, self.SFb, qfp4.SF_MMA)
            torch.cuda.synchronize()
            del W

    def prologue(self, X=None):
        """a1 + a2 (+ a3 fused): global scale and quantisation of the activations."""
        q, c = self.q, self.case
        X = self.X if X is None else X
        if c.fmt == q.NVFP4:
            q.global_scale(X, self.gs_a)
        q.quantize(c.fmt, X, self.gs_a, self.Qa, self.SFa, q.SF_MMA)

    def gemm(self, Qb=None, SFb=None, D=None):
        q, c = self.q, self.case
        q.gemm_nt(c.fmt, c.M, c.N, c.K, self.Qa, self.SFa, self.Qb if Qb is None else Qb,
                  self.SFb if SFb is None else SFb, self.gs_a, self.gs_b, self.D if D is None else D,
                  self.ws, self.ws_bytes)


class Flush:
    """Evicts L2 between steps by READING a buffer of 4x its size: the
    previous step's dirty lines are written back during this pass, outside
    the timed events, and the next step starts from clean lines."""

    def __init__(self, device):
        import torch
        self.buf = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self):
        return self.buf.sum()


def time_steps(pipe, n, flush, stream, split=True):
    """n steps, each bracketed by CUDA events on the launching stream, with
    the L2 flush before each step outside the events.  split: one more event
    between the prologue and the GEMM, for the breakdown; it makes the GEMM
    wait for the quantiser to finish instead of starting its set-up under the
    quantiser's tail (programmatic dependent launch), which lengthens the
    step by ~6 us, so the step time itself is taken without it.  Returns
    per-step (step, gemm, prologue) ms (gemm and prologue empty unless
    split)."""
    torch = pipe.torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush()
        e0, e1, e2 = ev[i]
        e0.record(stream)
        pipe.prologue()
        if split:
            e1.record(stream)
        pipe.gemm()
        e2.record(stream)
    torch.cuda.synchronize()
    steps = [a.elapsed_time(c) for a, _, c in ev]
    if not split:
        return steps, [], []
    return steps, [b.elapsed_time(c) for _, b, c in ev], [a.elapsed_time(b) for a, b, _ in ev]


def time_main(pipe, steps, warmup, flush, world, device, clocks_gpu, soak_s=SOAK_SECONDS):
    """Warm-up, then a soak of soak_s seconds of flushed steps (not part of
    `value`), then exactly `steps` timed steps between barriers and
    synchronisations (events before and after each step only), then a second
    block of `steps` steps, also between barriers and synchronisations, with
    the event between the prologue and the GEMM that times the GEMM alone.
    SM clocks are sampled over all of them.  Returns (total ms of the timed
    steps, max over ranks; stats)."""
    torch = pipe.torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        pipe.prologue()
        pipe.gemm()
    torch.cuda.synchronize()
    sampler = ClockSampler(clocks_gpu)
    soak_step, soak_gemm, soak_pro = [], [], []
    with sampler:
        time.sleep(0.3)
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < soak_s or not soak_step:
            a, b, c = time_steps(pipe, 100, flush, stream)
            soak_step += a
            soak_gemm += b
            soak_pro += c
        soak_wall = time.perf_counter() - t0
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        step_ms, _, _ = time_steps(pipe, steps, flush, stream, split=False)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        split_ms, gemm_ms, pro_ms = time_steps(pipe, steps, flush, stream)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
    total_ms = reduce_max(sum(step_ms), world, device)
    all_gemm = soak_gemm + gemm_ms
    stats = {"gemm_ms_median": statistics.median(all_gemm), "gemm_ms_min": min(all_gemm),
             "gemm_ms_timed_median": statistics.median(gemm_ms),
             "prologue_ms_median": statistics.median(soak_pro + pro_ms),
             "split_step_ms_median": statistics.median(split_ms),
             "soak": {"steps": len(soak_step), "seconds": round(soak_wall, 2),
                      "step_us_median": round(statistics.median(soak_step) * 1e3, 2),
                      "step_us_min": round(min(soak_step) * 1e3, 2)},
             "clocks": sampler.summary()}
    return total_ms, stats


def time_e2e(pipe, steps, warmup):
    """Same step through host buffers: pinned H2D of X, the path, D2H of D,
    one step after the other on one stream.  Returns (ms per step, H2D
    bytes, D2H bytes)."""
    torch = pipe.torch
    stream = torch.cuda.current_stream()

    def one():
        pipe.X.copy_(pipe.X_pinned, non_blocking=True)
        pipe.prologue()
        pipe.gemm()
        pipe.D_pinned.copy_(pipe.D, non_blocking=True)

    for _ in range(max(warmup, 1)):
        one()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(steps):
        one()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    return ms, pipe.X_pinned.numel() * 2, pipe.D_pinned.numel() * 2


def time_e2e_pipelined(pipe, steps, warmup, slices=1):
    """The same steps as a serving loop runs them: two steps in flight, the
    H2D of X for step i+1 and the D2H of D from step i-1 overlapping the
    kernels of step i, with two device copies of X and D (and two pinned D
    buffers).  A copy may be split into `slices` row ranges on streams of
    their own; measured on GB300, four slices were slower than one (more
    host work per step, no more copy bandwidth), so one is the default.
    Every step still moves all of its X in and all of its D out inside the
    timed region.  Returns ms per step."""
    torch = pipe.torch
    dev = pipe.X.device
    Xs = [pipe.X, torch.empty_like(pipe.X)]
    Ds = [pipe.D, torch.empty_like(pipe.D)]
    Dh = [pipe.D_pinned, torch.empty_like(pipe.D_pinned).pin_memory()]
    s_in = [torch.cuda.Stream(device=dev) for _ in range(slices)]
    s_out = [torch.cuda.Stream(device=dev) for _ in range(slices)]
    s_run = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    h2d_done = [[ev() for _ in range(slices)] for _ in range(2)]
    d2h_done = [[ev() for _ in range(slices)] for _ in range(2)]
    run_done = [ev(), ev()]
    cur = torch.cuda.current_stream()
    for b in range(2):
        run_done[b].record(cur)
        for e_ in d2h_done[b]:
            e_.record(cur)
    xr = (pipe.X.shape[0] + slices - 1) // slices
    dr = (pipe.D.shape[0] + slices - 1) // slices

    def step(i):
        b = i % 2
        for k in range(slices):
            with torch.cuda.stream(s_in[k]):
                s_in[k].wait_event(run_done[b])          # step i-2 is done reading X[b]
                Xs[b][k * xr:(k + 1) * xr].copy_(pipe.X_pinned[k * xr:(k + 1) * xr], non_blocking=True)
                h2d_done[b][k].record(s_in[k])
        with torch.cuda.stream(s_run):
            for k in range(slices):
                s_run.wait_event(h2d_done[b][k])
                s_run.wait_event(d2h_done[b][k])         # step i-2's D[b] has left
            pipe.prologue(Xs[b])
            pipe.gemm(D=Ds[b])
            run_done[b].record(s_run)
        for k in range(slices):
            with torch.cuda.stream(s_out[k]):
                s_out[k].wait_event(run_done[b])
                Dh[b][k * dr:(k + 1) * dr].copy_(Ds[b][k * dr:(k + 1) * dr], non_blocking=True)
                d2h_done[b][k].record(s_out[k])

    for i in range(max(warmup, 2)):
        step(i)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_run)
    for k in range(slices):
        s_in[k].wait_stream(s_run)                       # nothing of the loop starts before `start`
    for i in range(steps):
        step(i)
    for k in range(slices):
        cur.wait_stream(s_out[k])
    cur.wait_stream(s_run)
    end.record(cur)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def graph_time(calls, reps=10):
    """Mean device time of one call, for kernels of a few microseconds where
    host launch overhead would otherwise show: the calls are captured once in
    a CUDA graph (back to back on one stream) and the graph is replayed
    between CUDA events.  Returns the median over `reps` replays divided by
    the number of calls."""
    import torch
    for c in calls:
        c()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for c in calls:
                c()
    torch.cuda.synchronize()
    # replay() launches on the current stream: the events go on that stream too
    cur = torch.cuda.current_stream()
    graph.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for _ in range(reps):
        s.record(cur)
        graph.replay()
        e.record(cur)
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e) / len(calls))
    del graph
    return statistics.median(ts)


def rotated_gemm_time(case, device, l2_bytes, reps=10):
    """Mean device time of one GEMM launch over weight copies rotated so that
    the weights' footprint exceeds twice the L2 (no L2 hits on the weights
    from the previous launch)."""
    import torch
    pipe = Pipeline(case, device)
    pipe.prologue()
    wbytes = pipe.Qb.numel() + pipe.SFb.numel()
    copies = max(1, min(16, int(np.ceil(2 * l2_bytes / max(wbytes, 1))) + 1))
    Qs = [pipe.Qb] + [pipe.Qb.clone() for _ in range(copies - 1)]
    SFs = [pipe.SFb] + [pipe.SFb.clone() for _ in range(copies - 1)]
    calls = [(lambda i=i: pipe.gemm(Qs[i], SFs[i])) for i in range(copies)]
    ms = graph_time(calls, reps)
    del Qs, SFs, calls, pipe
    torch.cuda.empty_cache()
    return ms


def sweep(device, l2_bytes, peaks):
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    out = []
    for case in (synth.DECODE_UP, synth.DECODE_ATTN):
        ms = rotated_gemm_time(case, device, l2_bytes)
        g = 16 if case.fmt == 1 else 32
        byts = case.M * case.K / 2 + case.N * case.K / 2 + (case.M + case.N) * case.K / g + 2 * case.M * case.N
        gbs = byts / (ms * 1e-3) / 1e9
        out.append({"workload": case.name, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
                    "frac_hbm": round(gbs / peaks["hbm_gbs"], 3),
                    "TFLOP/s": round(2 * case.M * case.N * case.K / (ms * 1e-3) / 1e12, 1)})
    # standalone quantiser X[16384, 4096] (input 134 MB > L2 by itself)
    for fmt in (qfp4.NVFP4, qfp4.MXFP4):
        M, K = synth.QUANT_ROWS, synth.QUANT_COLS
        g = qfp4.block_size(fmt)
        xa = synth.activations_bf16(synth.QUANT_SEED, M, K)
        X = torch.from_numpy(xa.view(np.int16).copy()).view(torch.bfloat16).to(device)
        gs = torch.ones(1, dtype=torch.float32, device=device)
        qfp4.global_scale(X, gs)
        Q = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
        SF = torch.empty(qfp4.sf_mma_bytes(M, K // g), dtype=torch.uint8, device=device)
        # X alone (134 MB) exceeds the L2, so back-to-back launches re-read it from HBM
        ms = graph_time([lambda: qfp4.quantize(fmt, X, gs, Q, SF, qfp4.SF_MMA)] * 8)
        byts = 2 * M * K + M * K / 2 + M * K / g
        gbs = byts / (ms * 1e-3) / 1e9
        out.append({"workload": f"{'nv' if fmt else 'mx'}fp4_quantize_{M}x{K}", "us": round(ms * 1e3, 2),
                    "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)})
        del X, Q, SF
    # residual add + RMSNorm + NVFP4 quantisation (per-row global scales) on X[16384, 4096]
    M, K = synth.QUANT_ROWS, synth.QUANT_COLS
    call = rmsnorm_call(device)
    # X, R and Y (400 MB) exceed the L2, so back-to-back launches stream from HBM
    ms = graph_time([call] * 8)
    byts = 3 * 2 * M * K + M * K / 2 + M * K / 16 + 4 * M
    gbs = byts / (ms * 1e-3) / 1e9
    out.append({"workload": f"nvfp4_residual_rmsnorm_quantize_{M}x{K}", "us": round(ms * 1e3, 2),
                "GB/s": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 3)})
    del call
    # the step on the prefill-attention shape 4096^3 (global scale, quantise, GEMM), L2 flushed
    pipe = Pipeline(synth.PREFILL_NV, device)
    flush = Flush(device)
    stream = torch.cuda.current_stream()
    time_steps(pipe, 5, flush, stream)
    st, _, _ = time_steps(pipe, 200, flush, stream, split=False)
    _, gm, pr = time_steps(pipe, 200, flush, stream)
    c = synth.PREFILL_NV
    flop = 2.0 * c.M * c.N * c.K
    out.append({"workload": f"nvfp4_step_{c.M}x{c.N}x{c.K}", "us_step": round(statistics.median(st) * 1e3, 2),
                "TFLOP/s_step": round(flop / (statistics.median(st) * 1e-3) / 1e12, 1),
                "us_gemm": round(statistics.median(gm) * 1e3, 2), "us_gemm_min": round(min(gm) * 1e3, 2),
                "us_prologue": round(statistics.median(pr) * 1e3, 2),
                "frac_fp4_peak_gemm": round(flop / (statistics.median(gm) * 1e-3) / 1e12 / fp4_peak, 3)})
    del pipe, flush
    # compute-bound sweep
    us_of = {}
    for case in synth.COMPUTE_SWEEP:
        ms = rotated_gemm_time(case, device, l2_bytes, reps=5)
        tf = 2 * case.M * case.N * case.K / (ms * 1e-3) / 1e12
        out.append({"workload": case.name, "us": round(ms * 1e3, 1), "TFLOP/s": round(tf, 1),
                    "frac_fp4_peak": round(tf / fp4_peak, 3)})
        us_of[(case.fmt, case.M, case.N, case.K)] = ms * 1e3
    # NVFP4 / MXFP4 time on the same shapes (the DeepGEMM pull request's
    # "Benchmark" section reports 1.09-1.16x; it does not name the GPU)
    for (fmt, M, N, K), us in sorted(us_of.items()):
        if fmt == qfp4.NVFP4 and (qfp4.MXFP4, M, N, K) in us_of:
            out.append({"workload": f"nvfp4_over_mxfp4_time_{M}x{N}x{K}",
                        "ratio": round(us / us_of[(qfp4.MXFP4, M, N, K)], 3)})
    # scale-factor interleave, row-major -> MMA layout, on the scales of an
    # NVFP4 [65536, 16384] operand (64 MiB in, 64 MiB out; two buffer sets
    # rotated so that consecutive launches do not find their input in L2)
    rows, cols = 65536, 16384 // 16
    sets = []
    for _ in range(2):
        src = torch.randint(0, 0x7F, (rows, cols), dtype=torch.uint8, device=device)
        dst = torch.empty(qfp4.sf_mma_bytes(rows, cols), dtype=torch.uint8, device=device)
        sets.append((src, dst))
    byts = rows * cols + qfp4.sf_mma_bytes(rows, cols)
    # both directions: row-major -> MMA layout, then back on the same buffers
    for name, layout, fwd in (("to_mma", qfp4.SF_MMA, True), ("to_rowmajor", qfp4.SF_ROWMAJOR, False)):
        calls = [(lambda a=a, b=b, layout=layout, fwd=fwd: qfp4.sf_interleave(a, rows, cols, b, layout) if fwd
                  else qfp4.sf_interleave(b, rows, cols, a, layout)) for a, b in sets] * 4
        ms = graph_time(calls, 10)
        out.append({"workload": f"sf_interleave_{name}_{rows}x{cols}", "us": round(ms * 1e3, 2),
                    "GB/s": round(byts / (ms * 1e-3) / 1e9, 1),
                    "frac_hbm": round(byts / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3)})
    del sets, calls
    # 2:4 pair-sparse GEMM against the dense one
    out += sparse_time(device, l2_bytes, fp4_peak)
    # grouped MoE up-projection
    out.append(grouped_time(device, fp4_peak))
    # two-level NVFP4 (per-row global scales, row/column rescale in the epilogue)
    out.append(two_level_time(device, l2_bytes, fp4_peak))
    # up-projection with SwiGLU and requantisation in the epilogue
    for grouped in (False, True):
        try:
            out.append(swiglu_time(device, l2_bytes, fp4_peak, grouped))
        except Exception as exc:       # keep the rest of the line if this entry fails
            out.append({"workload": f"nvfp4_swiglu_up{'_grouped' if grouped else ''}", "error": repr(exc)[:200]})
    torch.cuda.empty_cache()
    return out


# sweep workload -> the key of its ncu DRAM counters in profiles/dram_traffic.json
SWEEP_TRAFFIC = {
    "nvfp4_quantize_16384x4096": "quantize_kernel nvfp4 16384x4096",
    "nvfp4_gemm_nt_128x14336x4096": "gemm_decode_kernel nvfp4 128x14336x4096",
    "nvfp4_gemm_nt_128x4096x4096": "gemm_decode_kernel nvfp4 128x4096x4096",
    "nvfp4_gemm_nt_4096x4096x4096": "gemm_pair_kernel nvfp4 4096x4096x4096",
    "nvfp4_gemm_nt_8192x8192x8192": "gemm_pair_kernel nvfp4 8192x8192x8192",
    "nvfp4_grouped_up_4096tok_top2_8exp": "gemm_pair_kernel grouped nvfp4 moe_up_8x14336x4096",
    "nvfp4_swiglu_up_4096x7168x4096": "gemm_pair_kernel swiglu nvfp4 4096x7168x4096",
    "nvfp4_b32_sparse24_gemm_nt_8192x8192x8192": "gemm_sparse_kernel nvfp4_b32 8192x8192x8192",
    "nvfp4_residual_rmsnorm_quantize_16384x4096": "rmsnorm_quant_kernel nvfp4 16384x4096",
}


def attach_traffic(entries):
    """Adds each sweep entry's DRAM bytes per launch from its committed ncu
    summary (absent when the kernel source changed since the capture)."""
    for e in entries:
        key = SWEEP_TRAFFIC.get(e.get("workload"))
        t = ncu_traffic(key) if key else None
        if t is not None:
            e["ncu_dram_bytes_per_launch"] = t
            e["ncu_key"] = key
    return entries


SPARSE_SHAPES = ((4096, 4096, 4096), (4096, 14336, 4096), (4096, 4096, 14336), (8192, 8192, 8192))


def sparse_operands(device, M, N, K):
    """Operands of the 2:4 pair-sparse GEMM: X quantised to NVFP4 with 32-element
    scale blocks; W likewise, pruned to two of every four pair bytes (a seeded
    pattern) and compressed; D.  Returns (Qx, SFx, Wc, meta, SFw, gx, gw, D)."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    X = torch.from_numpy(synth.activations_bf16(synth.SEED_BASE + 11, M, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    W = torch.from_numpy(synth.weights_bf16(synth.SEED_BASE + 12, N, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    gx = torch.empty(1, dtype=torch.float32, device=device)
    gw = torch.empty(1, dtype=torch.float32, device=device)
    qfp4.global_scale(X, gx)
    qfp4.global_scale(W, gw)
    Qx = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
    SFx = torch.empty(qfp4.sf_mma_bytes(M, K // 32), dtype=torch.uint8, device=device)
    qfp4.quantize(qfp4.NVFP4_B32, X, gx, Qx, SFx, qfp4.SF_MMA)
    Qw = torch.empty((N, K // 2), dtype=torch.uint8, device=device)
    SFw = torch.empty(qfp4.sf_mma_bytes(N, K // 32), dtype=torch.uint8, device=device)
    qfp4.quantize(qfp4.NVFP4_B32, W, gw, Qw, SFw, qfp4.SF_MMA)
    del X, W
    gen = torch.Generator(device=device).manual_seed(synth.SEED_BASE + 13)
    keep = torch.rand((N, K // 8, 4), generator=gen, device=device).argsort(dim=2)[..., :2]
    mask = torch.zeros((N, K // 8, 4), dtype=torch.bool, device=device).scatter_(2, keep, True)
    Qw = torch.where(mask.view(N, K // 2), Qw, torch.zeros_like(Qw))
    Wc = torch.empty((N, K // 4), dtype=torch.uint8, device=device)
    meta = torch.empty(qfp4.sparse24_meta_bytes(N, K, qfp4.SF_MMA), dtype=torch.uint8, device=device)
    qfp4.sparse24_compress(Qw, Wc, meta, qfp4.SF_MMA)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    return Qx, SFx, Wc, meta, SFw, gx, gw, D


def rmsnorm_call(device):
    """The residual-add + RMSNorm NVFP4 quantiser on X[16384, 4096] with a
    residual and per-row global scales, MMA-layout scales; returns the call."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    M, K = synth.QUANT_ROWS, synth.QUANT_COLS
    X = torch.from_numpy(synth.activations_bf16(synth.QUANT_SEED, M, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    R = torch.from_numpy(synth.activations_bf16(synth.QUANT_SEED + 1, M, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    gamma = torch.from_numpy(synth.norm_weight_bf16(synth.QUANT_SEED + 2, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    Y = torch.empty_like(X)
    gs_rows = torch.empty(M, dtype=torch.float32, device=device)
    Q = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
    SF = torch.empty(qfp4.sf_mma_bytes(M, K // 16), dtype=torch.uint8, device=device)
    return lambda: qfp4.residual_rmsnorm_quantize(qfp4.NVFP4, X, R, gamma, 1e-6, Y, gs_rows, Q, SF, qfp4.SF_MMA)


def sparse_time(device, l2_bytes, fp4_peak):
    """The 2:4 pair-sparse GEMM (NVFP4 with 32-element scale blocks) at the
    shapes the pages measure it on (quadbit README, "Headline result": attn
    4096^3, ffn-up, ffn-down, square 8192), weights rotated past the L2, in
    effective TFLOP/s = 2*M*N*K / t (the pages' count), beside the dense NVFP4
    GEMM on the same shape."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    out = []
    for (M, N, K) in SPARSE_SHAPES:
        Qx, SFx, Wc, meta, SFw, gx, gw, D = sparse_operands(device, M, N, K)
        wbytes = Wc.numel() + meta.numel() + SFw.numel()
        copies = max(1, min(16, int(np.ceil(2 * l2_bytes / wbytes)) + 1))
        Wcs = [Wc] + [Wc.clone() for _ in range(copies - 1)]
        Ms = [meta] + [meta.clone() for _ in range(copies - 1)]
        SFs = [SFw] + [SFw.clone() for _ in range(copies - 1)]
        calls = [(lambda i=i: qfp4.gemm_nt_sparse24(qfp4.NVFP4_B32, M, N, K, Qx, SFx, Wcs[i], Ms[i], SFs[i], gx,
                                                    gw, D)) for i in range(copies)]
        ms = graph_time(calls, 5)
        assert qfp4.poll_device_status() == 0
        del Wcs, Ms, SFs, calls, Qx, SFx, Wc, meta, SFw, D
        torch.cuda.empty_cache()
        dense = next((c for c in synth.COMPUTE_SWEEP + (synth.PREFILL_NV,)
                      if c.fmt == 1 and (c.M, c.N, c.K) == (M, N, K)), None)
        dense_ms = rotated_gemm_time(dense, device, l2_bytes, reps=5) if dense else None
        tf = 2 * M * N * K / (ms * 1e-3) / 1e12
        e = {"workload": f"nvfp4_b32_sparse24_gemm_nt_{M}x{N}x{K}", "us": round(ms * 1e3, 1),
             "TFLOP/s_effective": round(tf, 1), "frac_fp4_dense_peak": round(tf / fp4_peak, 3)}
        if dense_ms:
            e["us_dense_nvfp4"] = round(dense_ms * 1e3, 1)
            e["speedup_vs_dense"] = round(dense_ms / ms, 3)
        out.append(e)
    return out


def two_level_time(device, l2_bytes, fp4_peak):
    """NVFP4 4096^3 with per-row global scales: the step (per-row scales and
    quantisation of the activations, GEMM with the row/column rescale) and the
    rescaled GEMM against the plain one, weights rotated past the L2."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    case = synth.PREFILL_NV
    M, N, K = case.M, case.N, case.K
    X = torch.from_numpy(synth.activations_bf16(case.seed, M, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    W = torch.from_numpy(synth.weights_bf16(case.seed + 1000, N, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    gs_x = torch.empty(M, dtype=torch.float32, device=device)
    gs_w = torch.empty(N, dtype=torch.float32, device=device)
    Qa = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
    SFa = torch.empty(qfp4.sf_mma_bytes(M, K // 16), dtype=torch.uint8, device=device)
    Qb = torch.empty((N, K // 2), dtype=torch.uint8, device=device)
    SFb = torch.empty(qfp4.sf_mma_bytes(N, K // 16), dtype=torch.uint8, device=device)
    qfp4.global_scale_rows(W, gs_w)
    qfp4.quantize_rows(qfp4.NVFP4, W, gs_w, Qb, SFb, qfp4.SF_MMA)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    copies = max(1, min(16, int(np.ceil(2 * l2_bytes / (Qb.numel() + SFb.numel()))) + 1))
    Qs = [Qb] + [Qb.clone() for _ in range(copies - 1)]
    SFs = [SFb] + [SFb.clone() for _ in range(copies - 1)]

    def step(i):
        qfp4.global_scale_rows(X, gs_x)
        qfp4.quantize_rows(qfp4.NVFP4, X, gs_x, Qa, SFa, qfp4.SF_MMA)
        qfp4.gemm_nt_scaled(qfp4.NVFP4, M, N, K, Qa, SFa, Qs[i], SFs[i], None, None, gs_x, gs_w, D)

    step_ms = graph_time([(lambda i=i: step(i)) for i in range(copies)], 5)
    scaled_ms = graph_time([(lambda i=i: qfp4.gemm_nt_scaled(qfp4.NVFP4, M, N, K, Qa, SFa, Qs[i], SFs[i], None,
                                                              None, gs_x, gs_w, D)) for i in range(copies)], 5)
    plain_ms = graph_time([(lambda i=i: qfp4.gemm_nt(qfp4.NVFP4, M, N, K, Qa, SFa, Qs[i], SFs[i], None, None, D))
                           for i in range(copies)], 5)
    flop = 2 * M * N * K
    res = {"workload": f"nvfp4_two_level_{M}x{N}x{K}", "us_step": round(step_ms * 1e3, 2),
           "TFLOP/s_step": round(flop / (step_ms * 1e-3) / 1e12, 1),
           "us_gemm_rescaled": round(scaled_ms * 1e3, 2), "us_gemm_plain": round(plain_ms * 1e3, 2),
           "rescale_cost": round(scaled_ms / plain_ms - 1.0, 3),
           "frac_fp4_peak_gemm": round(flop / (scaled_ms * 1e-3) / 1e12 / fp4_peak, 3)}
    del Qs, SFs, X, W
    return res


def swiglu_setup(device, l2_bytes, grouped):
    """Operands of the SwiGLU up-projection (dense 4096 tokens x I = 7168 x
    K = 4096, W: 14336 gate/up rows; or the top-2-of-8 MoE batch with I = 7168
    per expert).  Returns (fused(i), plain(i), copies, rows, I, K, Qh, SFh, D):
    call i uses weight copy i (dense weights are rotated past the L2)."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    fmt, g, K = qfp4.NVFP4, 16, 4096
    I = synth.MOE_UP.N // 2
    if grouped:
        case = synth.MOE_UP
        counts = synth.moe_counts(case.seed, case.tokens, case.experts, case.topk)
        E = case.experts
    else:
        counts = np.array([4096])
        E = 1
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offs[-1])
    X = torch.from_numpy(synth.activations_bf16(synth.SEED_BASE + 7, rows, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    W = torch.from_numpy(synth.weights_bf16(synth.SEED_BASE + 8, E * 2 * I, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    d_offs = torch.from_numpy(offs).to(device)
    w_offs = torch.arange(0, (E + 1) * 2 * I, 2 * I, dtype=torch.int32, device=device)
    gs_a = torch.empty(E, dtype=torch.float32, device=device)
    gs_w = torch.empty(E, dtype=torch.float32, device=device)
    gs_o = torch.full((E,), 0.01, dtype=torch.float32, device=device)
    Qa = torch.empty((rows, K // 2), dtype=torch.uint8, device=device)
    SFa = torch.empty(qfp4.sf_mma_grouped_bytes(rows, E, K // g), dtype=torch.uint8, device=device)
    Qw = torch.empty((E * 2 * I, K // 2), dtype=torch.uint8, device=device)
    SFw = torch.empty(qfp4.sf_mma_grouped_bytes(E * 2 * I, E, K // g), dtype=torch.uint8, device=device)
    qfp4.global_scale_grouped(X, d_offs, gs_a)
    qfp4.quantize_grouped(fmt, X, d_offs, gs_a, Qa, SFa)
    qfp4.global_scale_grouped(W, w_offs, gs_w)
    qfp4.quantize_grouped(fmt, W, w_offs, gs_w, Qw, SFw)
    del X, W
    Qh = torch.empty((rows, I // 2), dtype=torch.uint8, device=device)
    SFh = torch.empty(qfp4.sf_mma_grouped_bytes(rows, E, I // g), dtype=torch.uint8, device=device)
    D = torch.empty((rows, 2 * I), dtype=torch.bfloat16, device=device)
    if grouped:
        def fused(i):
            qfp4.gemm_swiglu_quantize_grouped(fmt, d_offs, rows, I, K, Qa, SFa, Qw, SFw, gs_a, gs_w, gs_o, Qh, SFh)

        def plain(i):
            qfp4.gemm_nt_grouped(fmt, d_offs, rows, int(counts.max()), 2 * I, K, Qa, SFa, Qw, SFw, gs_a, gs_w, D)
        copies = 1
    else:
        copies = max(1, min(16, int(np.ceil(2 * l2_bytes / (Qw.numel() + SFw.numel()))) + 1))
        Qs = [Qw] + [Qw.clone() for _ in range(copies - 1)]
        SFs = [SFw] + [SFw.clone() for _ in range(copies - 1)]

        def fused(i):
            qfp4.gemm_swiglu_quantize(fmt, rows, I, K, Qa, SFa, Qs[i], SFs[i], gs_a, gs_w, gs_o, Qh, SFh)

        def plain(i):
            qfp4.gemm_nt(fmt, rows, 2 * I, K, Qa, SFa, Qs[i], SFs[i], gs_a, gs_w, D)
    return fused, plain, copies, rows, I, K, Qh, SFh, D


def swiglu_time(device, l2_bytes, fp4_peak, grouped):
    """Up-projection with SwiGLU and NVFP4 requantisation fused into the
    epilogue, against the plain GEMM writing BF16 on the same operands.
    Weights rotated past the L2 (dense) or the L2 flushed (grouped)."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    fused, plain, copies, rows, I, K, Qh, SFh, D = swiglu_setup(device, l2_bytes, grouped)
    if grouped:
        flush = Flush(device)

        def timed(fn):
            for _ in range(3):
                fn(0)
            torch.cuda.synchronize()
            ts = []
            for _ in range(5):
                flush()
                s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s0.record()
                fn(0)
                e0.record()
                torch.cuda.synchronize()
                ts.append(s0.elapsed_time(e0))
            return statistics.median(ts)
        fused_ms, plain_ms = timed(fused), timed(plain)
    else:
        fused_ms = graph_time([(lambda i=i: fused(i)) for i in range(copies)], 5)
        plain_ms = graph_time([(lambda i=i: plain(i)) for i in range(copies)], 5)
    assert qfp4.poll_device_status() == 0
    flop = 2.0 * rows * 2 * I * K
    name = (synth.MOE_UP.name.replace("grouped_up", "grouped_swiglu_up") if grouped
            else f"nvfp4_swiglu_up_{rows}x{I}x{K}")
    return {"workload": name, "us_fused": round(fused_ms * 1e3, 2), "us_gemm_bf16_out": round(plain_ms * 1e3, 2),
            "fused_cost": round(fused_ms / plain_ms - 1.0, 3),
            "TFLOP/s_fused": round(flop / (fused_ms * 1e-3) / 1e12, 1),
            "frac_fp4_peak_fused": round(flop / (fused_ms * 1e-3) / 1e12 / fp4_peak, 3),
            "bytes_out_fused": int(Qh.numel() + SFh.numel()), "bytes_out_bf16": int(D.numel() * 2)}


def grouped_setup(device):
    """Operands of the grouped MoE up-projection (quantised weights; the
    activations' global scales and quantisation are the prologue).  Returns
    (prologue(), gemm(), rows, counts)."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    case = synth.MOE_UP
    counts = synth.moe_counts(case.seed, case.tokens, case.experts, case.topk)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows, E, N, K = int(offs[-1]), case.experts, case.N, case.K
    g = qfp4.block_size(case.fmt)
    X = torch.from_numpy(synth.activations_bf16(case.seed, rows, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    W = torch.from_numpy(synth.weights_bf16(case.seed + 1000, E * N, K).view(np.int16).copy()).view(
        torch.bfloat16).to(device)
    d_offs = torch.from_numpy(offs).to(device)
    w_offs = torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device=device)
    gs_a = torch.empty(E, dtype=torch.float32, device=device)
    gs_b = torch.empty(E, dtype=torch.float32, device=device)
    Qa = torch.empty((rows, K // 2), dtype=torch.uint8, device=device)
    SFa = torch.empty(qfp4.sf_mma_grouped_bytes(rows, E, K // g), dtype=torch.uint8, device=device)
    Qb = torch.empty((E * N, K // 2), dtype=torch.uint8, device=device)
    SFb = torch.empty(qfp4.sf_mma_grouped_bytes(E * N, E, K // g), dtype=torch.uint8, device=device)
    D = torch.empty((rows, N), dtype=torch.bfloat16, device=device)
    qfp4.global_scale_grouped(W, w_offs, gs_b)
    qfp4.quantize_grouped(case.fmt, W, w_offs, gs_b, Qb, SFb)
    del W

    def prologue():
        qfp4.global_scale_grouped(X, d_offs, gs_a)
        qfp4.quantize_grouped(case.fmt, X, d_offs, gs_a, Qa, SFa)

    def gemm():
        qfp4.gemm_nt_grouped(case.fmt, d_offs, rows, int(counts.max()), N, K, Qa, SFa, Qb, SFb,
                             gs_a, gs_b, D)
    return prologue, gemm, rows, counts


def grouped_time(device, fp4_peak):
    import torch
    case = synth.MOE_UP
    N, K = case.N, case.K
    prologue, gemm, rows, counts = grouped_setup(device)
    for _ in range(3):
        prologue()
        gemm()
    torch.cuda.synchronize()
    flush = Flush(device)
    ts, gts = [], []
    # the step without an event between prologue and GEMM (which would make
    # the GEMM wait for the quantiser), then the GEMM alone with one
    for split in (False, True):
        for _ in range(5):
            flush()
            s, m, e = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            s.record()
            prologue()
            if split:
                m.record()
            gemm()
            e.record()
            torch.cuda.synchronize()
            if split:
                gts.append(m.elapsed_time(e))
            else:
                ts.append(s.elapsed_time(e))
    flops = 2.0 * rows * N * K
    ms, gms = statistics.median(ts), statistics.median(gts)
    return {"workload": case.name, "expert_rows": counts.tolist(), "us_step": round(ms * 1e3, 1),
            "TFLOP/s_step": round(flops / (ms * 1e-3) / 1e12, 1), "us_gemm": round(gms * 1e3, 1),
            "TFLOP/s_gemm": round(flops / (gms * 1e-3) / 1e12, 1),
            "frac_fp4_peak_gemm": round(flops / (gms * 1e-3) / 1e12 / fp4_peak, 3)}


def single_kernel(args, device):
    """--kernel NAME: only that kernel, `--warmup` then `--steps` launches
    (the short runs that ncu captures).  Prints one JSON line with the mean
    launch time over the timed launches."""
    import torch
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    name = args.kernel
    if name.startswith("quantize"):
        fmt = qfp4.NVFP4 if name.endswith("nvfp4") else qfp4.MXFP4
        M, K = synth.QUANT_ROWS, synth.QUANT_COLS
        g = qfp4.block_size(fmt)
        X = torch.from_numpy(synth.activations_bf16(synth.QUANT_SEED, M, K).view(np.int16).copy()).view(
            torch.bfloat16).to(device)
        gs = torch.ones(1, dtype=torch.float32, device=device)
        qfp4.global_scale(X, gs)
        Q = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
        SF = torch.empty(qfp4.sf_mma_bytes(M, K // g), dtype=torch.uint8, device=device)
        run = lambda: qfp4.quantize(fmt, X, gs, Q, SF, qfp4.SF_MMA)
        workload = f"{name}_{M}x{K}"
    elif name == "rmsnorm":
        run = rmsnorm_call(device)
        workload = f"nvfp4_residual_rmsnorm_quantize_{synth.QUANT_ROWS}x{synth.QUANT_COLS}"
    elif name == "sparse":
        M = N = K = 8192
        Qx, SFx, Wc, meta, SFw, gx, gw, D = sparse_operands(device, M, N, K)
        run = lambda: qfp4.gemm_nt_sparse24(qfp4.NVFP4_B32, M, N, K, Qx, SFx, Wc, meta, SFw, gx, gw, D)
        workload = f"nvfp4_b32_sparse24_gemm_nt_{M}x{N}x{K}"
    elif name == "grouped":
        prologue, run, _, _ = grouped_setup(device)
        prologue()
        workload = synth.MOE_UP.name
    elif name == "swiglu":
        fused, _, _, rows, I, K, _, _, _ = swiglu_setup(device, 0, False)
        run = lambda: fused(0)
        workload = f"nvfp4_swiglu_up_{rows}x{I}x{K}"
    else:
        case = {"decode_up": synth.DECODE_UP, "decode_attn": synth.DECODE_ATTN,
                "prefill": synth.PREFILL_NV, "square": synth.SQUARE_NV}[name]
        pipe = Pipeline(case, device)
        pipe.prologue()
        run = pipe.gemm
        workload = case.name
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(args.steps):
        run()
    e.record()
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    print(json.dumps({"kernel": name, "workload": workload, "launches": args.steps,
                      "us_per_launch": round(s.elapsed_time(e) * 1e3 / args.steps, 2)}), flush=True)


# --------------------------------------------------------------------------- CPU oracle arm

def oracle_sample(case, target_s):
    """Time the oracle on a bounded sample of the step: global scale over the
    whole activation tensor, quantisation of a slab of rows, and the GEMM of
    that slab against all N columns.  Returns (TFLOP/s, seconds, rows, threads)."""
    import oracle
    xa = synth.activations_bf16(case.seed, case.M, case.K)
    xw = synth.weights_bf16(case.seed + 1000, case.N, case.K)
    gw = oracle.global_scale(xw) if case.fmt == 1 else np.float32(1.0)
    qw, sfw = oracle.quantize(case.fmt, xw, gw)

    def run(rows):
        t0 = time.perf_counter()
        gs = oracle.global_scale(xa) if case.fmt == 1 else np.float32(1.0)
        qa, sfa = oracle.quantize(case.fmt, xa[:rows], gs)
        mi = np.repeat(np.arange(rows), case.N)
        ni = np.tile(np.arange(case.N), rows)
        oracle.gemm_nt_entries(case.fmt, qa, sfa, qw, sfw, gs, gw, mi, ni)
        return time.perf_counter() - t0

    t1 = run(1)
    rows = int(max(1, min(case.M, target_s / max(t1, 1e-3))))
    return rows, run, oracle.num_threads()


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or ''."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


def oracle_configs(target_s=2.0):
    """The oracle on every config, each on a bounded sample (about target_s
    seconds): GEMM configs as TFLOP/s of global scale + quantisation of a slab
    of activation rows + the GEMM of that slab against all N columns; the
    quantiser as GB/s of its algorithmic bytes.  All host cores, and one core
    for the small MXFP4 case and the decode attention shape."""
    import oracle
    out = []
    full = oracle.num_threads()

    def gemm_entry(case, threads, label):
        oracle.set_num_threads(threads)
        try:
            rows, run, _ = oracle_sample(case, target_s)
            dt = run(rows)
        finally:
            oracle.set_num_threads(full)
        out.append({"config": label, "value": 2.0 * rows * case.N * case.K / dt / 1e12, "unit": "TFLOP/s",
                    "threads": threads, "sample": f"{rows} of {case.M} rows x {case.N} columns, {dt:.2f} s"})

    # the small MXFP4 case: fp32 operands quantised by the oracle, whole GEMM
    c = synth.SMALL_MX
    a = synth.normal_f32(synth.rng(c.seed), (c.M, c.K))
    b = synth.normal_f32(synth.rng(c.seed + 1), (c.N, c.K))
    for threads in (full, 1):
        oracle.set_num_threads(threads)
        try:
            t0 = time.perf_counter()
            reps = 0
            while time.perf_counter() - t0 < min(target_s, 1.0) or reps == 0:
                qa, sfa = oracle.quantize(c.fmt, a)
                qb, sfb = oracle.quantize(c.fmt, b)
                oracle.gemm_nt(c.fmt, qa, sfa, qb, sfb)
                reps += 1
            dt = (time.perf_counter() - t0) / reps
        finally:
            oracle.set_num_threads(full)
        out.append({"config": c.name, "value": 2.0 * c.M * c.N * c.K / dt / 1e12, "unit": "TFLOP/s",
                    "threads": threads, "sample": f"whole problem, {reps} runs, {dt * 1e3:.2f} ms each"})
    gemm_entry(synth.PREFILL_NV, full, synth.PREFILL_NV.name)
    gemm_entry(synth.DECODE_UP, full, synth.DECODE_UP.name)
    gemm_entry(synth.DECODE_ATTN, full, synth.DECODE_ATTN.name)
    gemm_entry(synth.DECODE_ATTN, 1, synth.DECODE_ATTN.name)
    # the quantiser, NVFP4 X[16384, 4096]: global scale and quantisation of a slab
    M, K = synth.QUANT_ROWS, synth.QUANT_COLS
    x = synth.activations_bf16(synth.QUANT_SEED, M, K)
    gs = oracle.global_scale(x)
    t0 = time.perf_counter()
    oracle.quantize(1, x[:64], gs)
    t1 = max(time.perf_counter() - t0, 1e-4)
    rows = int(max(64, min(M, 64 * target_s / t1)))
    t0 = time.perf_counter()
    oracle.quantize(1, x[:rows], gs)
    dt = time.perf_counter() - t0
    out.append({"config": f"nvfp4_quantize_{M}x{K}", "value": rows * K * (2 + 0.5 + 1 / 16) / dt / 1e9,
                "unit": "GB/s", "threads": full, "sample": f"{rows} of {M} rows, {dt:.2f} s"})
    # the grouped MoE up-projection: one expert's rows against its weights
    g = synth.MOE_UP
    counts = synth.moe_counts(g.seed, g.tokens, g.experts, g.topk)
    e0 = synth.GemmCase(f"{g.name}_expert0", g.fmt, int(counts[0]), g.N, g.K, g.seed)
    gemm_entry(e0, full, f"{g.name} (expert 0 of {g.experts}, {int(counts[0])} rows)")
    return out


def cpu_baseline(case, target_s=10.0):
    rows, run, threads = oracle_sample(case, target_s)
    dt = run(rows)
    tf = 2.0 * rows * case.N * case.K / dt / 1e12
    return {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{case.name}: global scale of all {case.M} rows, quantise {rows} rows, "
                      f"GEMM of those {rows} rows x {case.N} columns (fp64), {dt:.1f} s",
            "cpu_model": cpu_model(), "nproc": os.cpu_count(), "configs": oracle_configs()}


def reference_arm(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return                      # the oracle arm runs on rank 0 only
    case = CASE
    rows, run, threads = oracle_sample(case, 3.0)
    for _ in range(args.warmup):
        run(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(rows)
    dt = (time.perf_counter() - t0) / args.steps
    tf = 2.0 * rows * case.N * case.K / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": tf, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": case.name, "M": case.M, "N": case.N, "K": case.K, "format": "NVFP4",
                       "sample_rows_per_step": rows, "l2": "n/a (host)"},
            "cpu_baseline": {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": f"{rows} of {case.M} activation rows per step (global scale, "
                                       f"quantise, GEMM vs all {case.N} columns)"},
            "e2e": {"value": tf, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--soak", type=float, default=SOAK_SECONDS,
                    help="seconds of clock-sampled steps ahead of the timed ones (0 for profiler runs)")
    ap.add_argument("--kernel", default=None,
                    choices=["quantize_nvfp4", "quantize_mxfp4", "decode_up", "decode_attn", "prefill",
                             "square", "grouped", "swiglu", "sparse", "rmsnorm"],
                    help="launch only this kernel (for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference_arm(args)
        return

    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    from block_scaled_fp4_tcgen05_gb300 import qfp4
    qfp4.load()
    if qfp4.device_check() != 0:
        raise SystemExit("bench.py needs an sm_103 GPU")
    props = torch.cuda.get_device_properties(device)
    l2_bytes = getattr(props, "L2_cache_size", 128 << 20)
    peaks = load_peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    if args.kernel:
        single_kernel(args, device)
        return

    case = CASE
    pipe = Pipeline(case, device)
    flush = Flush(device)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else local
    total_ms, stats = time_main(pipe, args.steps, args.warmup, flush, world, device, gpu_index, args.soak)
    clocks = stats.pop("clocks")
    gemm_ms, pro_ms = stats["gemm_ms_median"], stats["prologue_ms_median"]
    assert qfp4.poll_device_status() == 0
    flops = 2.0 * case.M * case.N * case.K
    ms_per_step = total_ms / args.steps
    value = world * flops / (ms_per_step * 1e-3) / 1e12

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return

    e2e_serial_ms, h2d, d2h = time_e2e(pipe, max(10, args.steps // 2), args.warmup)
    e2e_ms = time_e2e_pipelined(pipe, max(20, args.steps), args.warmup)
    gemm_tf = flops / (gemm_ms * 1e-3) / 1e12
    # the GEMM is timed inside a seconds-long loop of steps: the sustained
    # bf16 figure (measured under the power cap) sets its peak
    fp4_sus = peaks["bf16_tflops_sustained"] * FP4_OVER_BF16
    traffic = ncu_traffic(f"gemm_pair_kernel nvfp4 {case.M}x{case.N}x{case.K}")
    roof = {"bound": "tensor", "achieved": round(gemm_tf, 1), "peak": round(fp4_sus, 1),
            "unit": "TFLOP/s", "frac": round(gemm_tf / fp4_sus, 4), "traffic": traffic,
            "kernel": "gemm_pair_kernel<NVFP4> (qfp4_gemm_nt, CTA pairs on 256x256 tiles)",
            "gemm_us": round(gemm_ms * 1e3, 2), "gemm_us_min": round(stats["gemm_ms_min"] * 1e3, 2),
            "gemm_us_timed_median": round(stats["gemm_ms_timed_median"] * 1e3, 2),
            "gemm_samples": stats["soak"]["steps"] + args.steps,
            "prologue_us": round(pro_ms * 1e3, 2),
            "frac_of_burst_peak": round(gemm_tf / fp4_peak, 4),
            "peak_note": f"{peaks['source']} sustained bf16 {peaks['bf16_tflops_sustained']} TFLOP/s x "
                         f"{FP4_OVER_BF16:g} (nominal dense FP4:BF16 ratio), of {peaks['source']}; the GEMM "
                         f"runs inside a {stats['soak']['seconds']} s loop of steps.  Burst: "
                         f"{peaks['bf16_tflops']} x {FP4_OVER_BF16:g} = {fp4_peak:.1f}",
            "algorithmic_bytes": int(case.M * case.K / 2 + case.N * case.K / 2 +
                                     (case.M + case.N) * case.K / 16 + 2 * case.M * case.N)}
    if traffic is None:
        roof["traffic_note"] = ("no DRAM counters for the current source of this kernel's file "
                                "(profiles/dram_traffic.json is keyed to the source it was captured on)")
    del pipe
    torch.cuda.empty_cache()
    extra = [] if args.no_sweep else attach_traffic(sweep(device, l2_bytes, peaks))
    cpu = None if args.no_cpu else cpu_baseline(case)
    line = {"metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "vs_baseline_note": f"no GB300 number on the pages; context: quadbit dense FP4 square 8192, "
                                f"{PAGES_BASELINE_TFLOPS:g} TF/s on RTX PRO 6000 (SM120), another machine",
            "dtype": "nvfp4 (e2m1 x ue4m3) -> fp32 accumulate -> bf16", "data": "synthetic",
            "config": {"workload": case.name, "M": case.M, "N": case.N, "K": case.K, "format": "NVFP4",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "flushed between timed steps (read-only pass over 512 MiB, 4x L2)",
                       "step": "global scale + quantise (SF in MMA layout) + GEMM",
                       "timing": "value: the timed steps, CUDA events before and after each step only; "
                                 "gemm_us / prologue_us: the soak and a second block of the same number of "
                                 "steps, with an event between the prologue and the GEMM (which makes the "
                                 "GEMM wait for the quantiser to finish)",
                       "step_us_with_split_event": round(stats["split_step_ms_median"] * 1e3, 2),
                       "soak": stats["soak"]},
            "gpu_launches": pipe_kernels(case) * args.steps,
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "mode": "pipelined: H2D of step i+1 and D2H of step i-1 overlap step i (copy-in, "
                            "kernel and copy-out streams, two device copies of X and D)",
                    "ms_per_step": round(e2e_ms, 4),
                    "serial_value": round(world * flops / (e2e_serial_ms * 1e-3) / 1e12, 2)},
            "clocks": clocks, "sweep": extra}
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def pipe_kernels(case):
    # library launches per step: the global scale (NVFP4 only, one launch),
    # the quantiser and the GEMM
    return (1 if case.fmt == 1 else 0) + 2


if __name__ == "__main__":
    main()
