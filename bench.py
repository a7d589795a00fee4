"""Benchmark of the fine-grained FP8 GEMM path on B300.

One step is one pass of the path over the dense prefill workload
(M=4096 tokens, K=7168, weights N in {2112, 24576, 7168, 4096}; the shapes of
the DeepGEMM article's Table 1 and the DeepSeek-V3 prefill): 1x128
quantization of the BF16 activations, 128x128 quantization of each BF16
weight, and one FP8 GEMM per weight with FP32 promotion and BF16 output.

Printed metric: FP8 GEMM TFLOP/s of the whole step (2*M*N*K summed over the
four weights, divided by the step time), with the GEMM kernel's roofline
fraction (against the FP8 tensor peak) and the quantizers' HBM fraction.

Timing: the K timed steps are captured once into a CUDA graph, with a timing
event node around every kernel, and the graph is replayed inside the timed
region (host launch overhead stays out of the device time; an eager reading
of the same steps is reported beside it). Warm-up runs W eager steps and at
least a second of work. The line's ``configs`` object adds one graph-timed
entry per other workload (decode, grouped MoE, masked MoE, weight gradient,
requantization, small dense case) with its roofline fraction.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       python bench.py --case CASE --shape ...   (one kernel, see run_case)
With N>1 (torchrun), every rank runs the same workload on its own GPU
(independent replicas: the path has no exchange step); rank 0 prints.
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

M_PREFILL, K_PREFILL = 4096, 7168
N_PREFILL = (2112, 24576, 7168, 4096)
METRIC = "FP8 block-scaled GEMM TFLOP/s & % of B300 FP8 peak; quant GB/s vs HBM"
L2_ROTATE_BYTES = 3 * 126 * 2**20  # --case mode: working set of consecutive calls
FP8_PER_BF16 = 2.0  # nominal dense FP8 / BF16 tensor rate ratio (4.5 / 2.25 PFLOP/s)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}

# DRAM traffic of one GEMM launch per N, measured with ncu
# (dram__bytes_read.sum + dram__bytes_write.sum) on
# `bench.py --case gemm --shape 4096,N,7168` for the kernel source whose hash
# is given. When the kernel source changes the hash no longer matches and the
# reported traffic is null. Writes sit below M*N*2 because output lines still
# in L2 when the kernel ends are written back after it.
NCU_TRAFFIC = {
    "kernel_sha": "b8b09da913048397",
    "per_launch": {2112: 45532672 + 573952, 24576: 211239680 + 179841792,
                   7168: 83652608 + 37178368, 4096: 60663552 + 11681024},
}


# ---------------------------------------------------------------- models
def gemm_flops(M, N, K):
    return 2.0 * M * N * K


def gemm_bytes(M, N, K, out_bytes=2):
    """Algorithmic bytes of one GEMM: FP8 A and B once, scales once, C once."""
    return M * K + N * K + M * (K // 128) * 4 + ((N + 127) // 128) * (K // 128) * 4 + M * N * out_bytes


def quant_1x128_bytes(M, K, in_bytes=2):
    return M * K * in_bytes + M * K + M * (K // 128) * 4


def quant_128x128_bytes(N, K, in_bytes=2):
    return N * K * in_bytes + N * K + ((N + 127) // 128) * (K // 128) * 4


def table1_gbs(M, N, K, tflops):
    """Table 1's byte model (FP8 A and B, BF16 C) over the time its TFLOPS implies."""
    t = gemm_flops(M, N, K) / (tflops * 1e12)
    return (M * K + N * K + 2 * M * N) / t / 1e9


def kernel_sha():
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_common.cuh", "common.cuh", "quant_math.cuh"):
        h.update(open(os.path.join(ROOT, "fp8_fine_grained_24_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            ids = [v.strip() for v in vis.split(",")]
            if gpu_index < len(ids):
                self.gpu = ids[gpu_index]
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        t0, t1 = getattr(self, "window", (0.0, float("inf")))
        inside = [p for t, p in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.samples = inside
        def col(i):
            return [float(s[i]) for s in self.samples if len(s) > i and s[i].replace(".", "").isdigit()]

        sm, mx, power, mem = col(1), col(2), col(3), col(9)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples),
                "mem_mhz": statistics.median(mem) if mem else None,
                "power_w": round(statistics.median(power), 1) if power else None}


# ---------------------------------------------------------------- our arm
class PrefillStep:
    """Device-resident buffers and the launches of one step."""

    KINDS = ("quant_1x128", "quant_128x128", "gemm")

    def __init__(self, fg, torch, device, seed=1001):
        import workloads as wl
        self.fg, self.torch = fg, torch
        M, K = M_PREFILL, K_PREFILL
        self.x = wl.activations(M, K, seed, device=device)
        self.w = [wl.weights((n, K), seed + 1 + i, device=device) for i, n in enumerate(N_PREFILL)]
        self.qa = torch.empty((M, K), dtype=torch.uint8, device=device)
        self.sa = torch.empty((K // 128, fg.scale_ld(M)), dtype=torch.float32, device=device)
        self.qb = [torch.empty((n, K), dtype=torch.uint8, device=device) for n in N_PREFILL]
        self.sb = [torch.empty(((n + 127) // 128, K // 128), dtype=torch.float32, device=device) for n in N_PREFILL]
        self.c = [torch.empty((M, n), dtype=torch.bfloat16, device=device) for n in N_PREFILL]
        # one zero-filled Stream-K workspace, shared by the step's GEMMs (they
        # run in order on one stream), sized for the largest need
        ws_bytes = max(fg.gemm_workspace_size(M, n, K) for n in N_PREFILL)
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device) if ws_bytes else None
        self.flops = sum(gemm_flops(M, n, K) for n in N_PREFILL)
        self.launches = 1 + 2 * len(N_PREFILL)

    def run(self, events=None):
        """Enqueue one step on the current stream. If `events` is a list,
        bracket every launch with a pair of timing events (appended as
        (kind, start, end)); they are external events, so that inside a
        graph capture they become event-record nodes of the graph."""
        fg, torch = self.fg, self.torch

        def timed(kind, fn):
            if events is None:
                fn()
                return
            s = torch.cuda.Event(enable_timing=True, external=True)
            e = torch.cuda.Event(enable_timing=True, external=True)
            s.record()
            fn()
            e.record()
            events.append((kind, s, e))

        timed("quant_1x128", lambda: fg.fp8_quant_1x128_out(self.x, self.qa, self.sa))
        for i in range(len(N_PREFILL)):
            timed("quant_128x128", lambda i=i: fg.fp8_quant_128x128_out(self.w[i], self.qb[i], self.sb[i]))
            timed("gemm", lambda i=i: fg.fp8_gemm_dense_out(self.qa, self.sa, self.qb[i], self.sb[i], self.c[i],
                                                            workspace=self.ws))


def capture_steps(step, torch, stream, steps):
    """One CUDA graph holding `steps` steps with a timing event pair around
    every launch. Returns (graph, events)."""
    events = []
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(steps):
                step.run(events)
    torch.cuda.synchronize()
    return graph, events


# ---------------------------------------------------------------- replicas
def slowest_replica_ms(total_ms, dist, device):
    """The job's timed span: the maximum over ranks of each replica's span
    (every rank must call this; without a process group it is the local span)."""
    import torch
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_step, world, ms_per_step):
    """Whole-job rate: the units all `world` replicas processed per second."""
    return units_per_step * world / (ms_per_step * 1e-3)


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


MIN_WARMUP_S = 1.0  # warm-up wall time floor: clocks and power settle under load


def run_ours(args, rank, world, local_rank):
    import torch
    import fp8_fine_grained_24_b300 as fg

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    step = PrefillStep(fg, torch, device)
    stream = torch.cuda.Stream(device=device)
    stream.wait_stream(torch.cuda.current_stream())
    # The timed steps, captured once (outside the timed region).
    with torch.cuda.stream(stream):
        step.run()  # first calls outside capture: one-time per-device set-up
    torch.cuda.synchronize()
    # Two graphs of the K timed steps: the plain one gives the step time
    # (kernels back to back, programmatic launch overlap intact); the other
    # has an event-record node around every kernel, for the per-kernel
    # times (event nodes between kernels cost a few percent of step time).
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(args.steps):
                step.run()
    torch.cuda.synchronize()
    try:
        graph_ev, events = capture_steps(step, torch, stream, args.steps)
        per_kernel_timing = "event-record nodes around every kernel in a second replay of the K steps"
    except RuntimeError as exc:  # event nodes refused in capture: time kernels eagerly instead
        print(f"note: per-kernel event nodes unavailable in capture ({exc}); timing kernels eagerly",
              file=sys.stderr)
        torch.cuda.synchronize()
        graph_ev, events = None, None
        per_kernel_timing = "eager launches with events around each (host gaps included)"

    clocks = ClockSampler(local_rank)
    clocks.start()
    # Warm-up: W eager steps, then more until MIN_WARMUP_S of wall time has
    # passed (a fixed count of ~1 ms steps leaves the clocks and the power
    # state of an idle GPU still settling in the timed region).
    t_warm = time.time()
    warm_steps = 0
    with torch.cuda.stream(stream):
        while warm_steps < args.warmup or time.time() - t_warm < MIN_WARMUP_S:
            step.run()
            warm_steps += 1
            if warm_steps % 50 == 0:
                stream.synchronize()
        graph.replay()  # the graphs' own first replays are warm-up too
        if graph_ev is not None:
            graph_ev.replay()
    fg.check()
    barrier()

    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    w0 = time.time()
    with torch.cuda.stream(stream):
        start.record()
        graph.replay()
        end.record()
    barrier()
    total_ms = start.elapsed_time(end)
    # second timed replay: the same steps with per-kernel event nodes
    ev_ms = None
    if graph_ev is not None:
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s2.record()
            graph_ev.replay()
            e2.record()
        barrier()
        ev_ms = s2.elapsed_time(e2) / args.steps
    clocks.mark(w0, time.time())
    clocks.stop()
    fg.check()
    if events is None:
        events = []
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                step.run(events)
        barrier()
    per_kind = {}
    for kind, s, e in events:
        per_kind.setdefault(kind, []).append(s.elapsed_time(e))
    total_ms = slowest_replica_ms(total_ms, dist, device)
    ms_per_step = total_ms / args.steps

    # Eager reading of the same steps (launches from the host, no graph):
    # what a caller that does not capture gets.
    with torch.cuda.stream(stream):
        barrier()
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record()
        for _ in range(args.steps):
            step.run()
        ee.record()
    barrier()
    eager_ms = es.elapsed_time(ee) / args.steps

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(step, fg, torch, device, max(4, min(args.steps, 10)), barrier)

    cfgs = None
    if not args.no_configs:
        cfgs = run_configs(fg, torch, device)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return None

    peaks, peak_src = load_peaks()
    fp8_peak_burst = peaks["bf16_tflops"] * FP8_PER_BF16
    # The GEMM runs inside a long, power-capped step (a second of warm-up,
    # then the timed steps): its denominator is the sustained peak.
    fp8_peak = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * FP8_PER_BF16
    gemm_ms = sum(per_kind["gemm"])
    gemm_tflops = step.flops * args.steps / (gemm_ms * 1e-3) / 1e12
    q1_ms = sum(per_kind["quant_1x128"])
    q2_ms = sum(per_kind["quant_128x128"])
    q1_gbs = quant_1x128_bytes(M_PREFILL, K_PREFILL) * args.steps / (q1_ms * 1e-3) / 1e9
    q2_gbs = sum(quant_128x128_bytes(n, K_PREFILL) for n in N_PREFILL) * args.steps / (q2_ms * 1e-3) / 1e9
    sha = kernel_sha()
    traffic = None
    if NCU_TRAFFIC["kernel_sha"] == sha:
        # mean over the step's four launches, like `achieved`
        traffic = round(statistics.mean(NCU_TRAFFIC["per_launch"][n] for n in N_PREFILL))
    value = job_throughput(step.flops, world, ms_per_step) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 (fp32 accumulate, bf16 out)",
        "data": "synthetic (seeded N(0,1) activations with 1% channels x30, N(0,0.02) weights)",
        "config": {
            "workload": "dense prefill: M=4096, K=7168, N in {2112,24576,7168,4096}; bf16 in, "
                        "1x128 + 128x128 E4M3 quant, FP8 GEMM, bf16 out",
            "M": M_PREFILL, "K": K_PREFILL, "N": list(N_PREFILL),
            "l2": "no flush: each step streams ~1.3 GB (> 126 MB L2)",
            "parallelism": f"replicas x{world}",
            "timing": "K steps captured in one CUDA graph (no event nodes), replayed once in the timed region",
            "per_kernel_timing": per_kernel_timing,
        },
        "eager_ms_per_step": round(eager_ms, 4),
        "ms_per_step_with_event_nodes": None if ev_ms is None else round(ev_ms, 4),
        "roofline": {
            "bound": "tensor",
            "achieved": round(gemm_tflops, 1),
            "peak": round(fp8_peak, 1),
            "unit": "TFLOP/s",
            "frac": round(gemm_tflops / fp8_peak, 4),
            "traffic": traffic,
            "algorithmic_bytes": round(statistics.mean(gemm_bytes(M_PREFILL, n, K_PREFILL) for n in N_PREFILL)),
            "kernel": "fp8_gemm_kernel<256> (4 launches per step)",
            "peak_note": f"{peak_src} sustained bf16 {peaks.get('bf16_tflops_sustained')} x {FP8_PER_BF16} "
                         f"(nominal FP8/BF16): the kernel runs inside a long power-capped step; against the "
                         f"burst-based peak {round(fp8_peak_burst, 1)} the fraction is "
                         f"{round(gemm_tflops / fp8_peak_burst, 4)}",
        },
        "kernels": {
            "gemm_ms_per_step": round(gemm_ms / args.steps, 4),
            "quant_1x128_ms_per_step": round(q1_ms / args.steps, 4),
            "quant_1x128_gbs": round(q1_gbs, 1),
            "quant_128x128_ms_per_step": round(q2_ms / args.steps, 4),
            "quant_128x128_gbs": round(q2_gbs, 1),
            "hbm_peak_gbs": peaks["hbm_gbs"],
            "gemm_per_n_ms": {str(n): round(statistics.mean(per_kind["gemm"][i::len(N_PREFILL)]), 4)
                              for i, n in enumerate(N_PREFILL)},
            "shares": {k: round(sum(per_kind[k]) / sum(sum(v) for v in per_kind.values()), 4) for k in per_kind},
        },
        "e2e": e2e,
        "gpu_launches": step.launches * args.steps,
        "clocks": clocks.summary(),
        "kernel_sha": sha,
    }
    line["warmup_done"] = {"steps": warm_steps, "min_seconds": MIN_WARMUP_S}
    if cfgs is not None:
        line["configs"] = cfgs
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    if dist is not None:
        dist.destroy_process_group()
    return line


def run_e2e(step, fg, torch, device, steps, barrier):
    """Same step through the public API, with pinned host inputs copied in
    and every output copied out each step. Double-buffered on three streams:
    the inputs of step i+1 go in while step i computes, and its outputs come
    back while step i+1 computes, so that both directions of the host link
    are busy at once (every step still moves all of its own bytes)."""
    hx = step.x.cpu().pin_memory()
    hw = [w.cpu().pin_memory() for w in step.w]
    hc = [[torch.empty(c.shape, dtype=c.dtype, pin_memory=True) for c in step.c] for _ in range(2)]
    h2d = hx.numel() * hx.element_size() + sum(w.numel() * w.element_size() for w in hw)
    d2h = sum(c.numel() * c.element_size() for c in step.c)
    dx = [torch.empty_like(step.x) for _ in range(2)]
    dw = [[torch.empty_like(w) for w in step.w] for _ in range(2)]
    dc = [[torch.empty_like(c) for c in step.c] for _ in range(2)]
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[b])  # the buffers' previous step has finished with them
            dx[b].copy_(hx, non_blocking=True)
            for d, h in zip(dw[b], hw):
                d.copy_(h, non_blocking=True)
            ev_in[b].record()

    def compute(i):
        b = i % 2
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(ev_in[b])
            s_comp.wait_event(ev_out[b])  # the outputs of step i-2 have been copied out
            fg.fp8_quant_1x128_out(dx[b], step.qa, step.sa)
            for j in range(len(N_PREFILL)):
                fg.fp8_quant_128x128_out(dw[b][j], step.qb[j], step.sb[j])
                fg.fp8_gemm_dense_out(step.qa, step.sa, step.qb[j], step.sb[j], dc[b][j], workspace=step.ws)
            ev_comp[b].record()

    def copy_out(i):
        b = i % 2
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for h, d in zip(hc[b], dc[b]):
                h.copy_(d, non_blocking=True)
            ev_out[b].record()

    def run(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)

    run(2)
    barrier()
    t0 = time.perf_counter()
    run(steps)
    barrier()
    dt = (time.perf_counter() - t0) / steps
    return {"value": round(step.flops / dt / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": round(dt * 1e3, 3), "steps": steps,
            "pipelining": "double-buffered: step i+1's inputs in and step i-1's outputs out during step i"}


# Every other workload of the path, graph-timed one kernel at a time
# (case, shape, requant source). Shapes: decode M in {64, 128} x
# (N, K) in {(7168, 16384), (4096, 7168)}; grouped-contiguous MoE, 8
# experts and 8192 Zipf-routed tokens, (N, K) in {(4096, 7168), (7168,
# 2048)}; grouped-masked MoE, 16 experts of <= 256 tokens, N=4096, K=7168;
# its weight gradient; the 128x1 requantization from E4M3 and from BF16;
# the small dense case; the prefill GEMM with its output quantized in the
# epilogue, beside the unfused GEMM + quantizer pair; the data gradient of
# the N=7168 prefill layer; the dense weight gradient over 4096 tokens; and
# the prefill step's own quantizations one at a time (1x128 of the 4096 x
# 7168 activations, 128x128 of each of the four weights), outside the step's
# per-kernel event windows.
CONFIG_CASES = (
    ("gemm", (128, 256, 512), None),
    ("gemm", (64, 7168, 16384), None),
    ("gemm", (128, 7168, 16384), None),
    ("gemm", (64, 4096, 7168), None),
    ("gemm", (128, 4096, 7168), None),
    ("contig", (8, 8192, 4096, 7168), None),
    ("contig", (8, 8192, 7168, 2048), None),
    ("masked", (16, 256, 4096, 7168), None),
    ("wgrad", (16, 256, 4096, 7168), None),
    ("requant", (4096, 7168), "e4m3"),
    ("requant", (4096, 7168), "bf16"),
    ("gemm_quant", (4096, 7168, 7168), None),
    ("gemm_then_quant", (4096, 7168, 7168), None),
    ("dgrad", (4096, 7168, 7168), None),
    ("wgrad_dense", (4096, 4096, 7168), None),
    ("wgrad_dense_bs", (4096, 4096, 7168), None),
    ("quant1x128", (4096, 7168), None),
    ("quant128x128", (2112, 7168), None),
    ("quant128x128", (24576, 7168), None),
    ("quant128x128", (7168, 7168), None),
    ("quant128x128", (4096, 7168), None),
)


def run_configs(fg, torch, device):
    peaks, src = load_peaks()
    fp8_peak = peaks["bf16_tflops"] * FP8_PER_BF16
    hbm = peaks["hbm_gbs"]
    out = {}
    for case, dims, rsrc in CONFIG_CASES:
        r = time_case(case, dims, rsrc or "e4m3", steps=10, warmup=3, graph_reps=10)
        name = f"{case}{'_' + rsrc if rsrc else ''} {'x'.join(map(str, dims))}"
        t = r["ms_median"] * 1e-3
        ent = {"ms": r["ms_median"], "GB/s": r["GB/s"]}
        if "TFLOP/s" in r:
            t_tc = r["flops"] / (fp8_peak * 1e12)
            t_hbm = r["bytes"] / (hbm * 1e9)
            ent["TFLOP/s"] = r["TFLOP/s"]
            ent["bound"] = "tensor" if t_tc >= t_hbm else "hbm"
            ent["roofline_frac"] = round(max(t_tc, t_hbm) / t, 4)
        else:
            ent["bound"] = "hbm"
            ent["roofline_frac"] = round(r["GB/s"] / hbm, 4)
        out[name] = ent
    out["_note"] = (f"graph-timed medians, rotating buffer sets (every call reads HBM); roofline time = "
                    f"max(flops / {round(fp8_peak, 1)} TFLOP/s, bytes / {hbm} GB/s), {src} peaks")
    return out


# ---------------------------------------------------------------- oracle arm
def oracle_sample(seconds_budget=15.0, seed=1001):
    """Time the oracle on a bounded sample of the prefill workload.

    Sample: R activation rows (1x128 quantization) against one 128-row block
    of every weight (128x128 quantization), FP64 product of the dequantized
    operands. R is grown until the run takes about `seconds_budget`.
    Returns (flops, seconds, description).
    """
    import torch
    import workloads as wl
    from oracle import gemm, quant

    x = wl.activations(M_PREFILL, K_PREFILL, seed, device="cpu").float().numpy()
    ws = [wl.weights((128, K_PREFILL), seed + 1 + i, device="cpu").float().numpy() for i in range(len(N_PREFILL))]
    rows = 64
    while True:
        t0 = time.perf_counter()
        qa, sa = quant.quant_1x128(x[:rows])
        flops = 0.0
        for w in ws:
            qb, sb = quant.quant_128x128(w)
            gemm.gemm_dense(qa, sa, qb, sb)
            flops += gemm_flops(rows, 128, K_PREFILL)
        dt = time.perf_counter() - t0
        if dt >= seconds_budget / 3 or rows >= M_PREFILL:
            desc = (f"{rows} activation rows x {len(ws)} weight blocks of 128 rows (K=7168): 1x128 + 128x128 "
                    f"quantization and FP64 product, numpy")
            return flops, dt, desc
        rows = min(M_PREFILL, rows * 2)
    del torch


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        return int(max(n)) if n else os.cpu_count()
    except Exception:
        return os.cpu_count()


def cpu_baseline(seconds=15.0):
    flops, dt, desc = oracle_sample(seconds)
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": desc, "seconds": round(dt, 2), "host_cpus": os.cpu_count(), "cpu_model": cpu_model()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    vals = []
    desc = ""
    for _ in range(args.warmup):
        oracle_sample(args.cpu_seconds / 3)
    t_total = 0.0
    for _ in range(args.steps):
        flops, dt, desc = oracle_sample(args.cpu_seconds / 3)
        vals.append(flops / dt / 1e12)
        t_total += dt
    value = statistics.mean(vals)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_total / args.steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (oracle)",
        "data": "synthetic",
        "config": {"workload": "dense prefill: M=4096, K=7168, N in {2112,24576,7168,4096} (bounded sample)",
                   "M": M_PREFILL, "K": K_PREFILL, "N": list(N_PREFILL)},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": desc, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def time_case(case, dims, src="e4m3", steps=20, warmup=5, graph_reps=10, rotate=True, workspace=True):
    """Time one kernel on one shape through a captured CUDA graph; returns a dict.

    gemm M,N,K        dense GEMM, bf16 out (operands quantized once, untimed)
    gemm_quant M,N,K  dense GEMM whose output is quantized per 1x128 tile in the epilogue
    gemm_then_quant M,N,K  the unfused pair: dense GEMM (bf16 out), then fp8_quant_1x128
    dgrad M,N,K       data gradient dX[M,K] = dY[M,N] W[N,K] (W read MN-major), bf16 out
    wgrad_dense T,N,C dense weight gradient dW[N,C] += G^T X over T tokens (128x1 pow2, FP32 accumulate)
    wgrad_dense_bs T,N,C  the same with the power-of-two scales applied in the tensor core (block-scaled MMA)
    contig E,T,N,K    grouped-contiguous MoE GEMM: T tokens routed by Zipf(1.1) counts
    masked E,M,N,K    grouped-masked MoE GEMM: uniform counts up to M tokens per expert
    wgrad E,T,N,C     masked-K weight gradient dW_e = G_e^T X_e (128x1 pow2 operands, FP32 out)
    quant1x128 M,K    activation quantization of bf16 [M, K]
    quant128x128 N,K  weight quantization of bf16 [N, K]
    requant T,C       128x1 requantization (pow2) of [T, C]: E4M3 with 1x128 scales, or --src bf16/fp32
    """
    import torch
    import fp8_fine_grained_24_b300 as fg
    import workloads as wl

    dims = [int(v) for v in dims]
    dev = torch.device("cuda", torch.cuda.current_device())

    def make(seed):
        """One independent buffer set: returns (call, algorithmic bytes, flops or None)."""
        if case == "gemm":
            M, N, K = dims
            qa, sa = fg.fp8_quant_1x128(wl.activations(M, K, seed, device=dev))
            qb, sb = fg.fp8_quant_128x128(wl.weights((N, K), seed + 1, device=dev))
            c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            ws = None if (not workspace) else fg.gemm_workspace(M, N, K, device=dev)
            return (lambda: fg.fp8_gemm_dense_out(qa, sa, qb, sb, c, workspace=ws),
                    gemm_bytes(M, N, K), gemm_flops(M, N, K))
        if case == "gemm_quant":
            # the GEMM with its output quantized per 1x128 tile in the epilogue
            M, N, K = dims
            qa, sa = fg.fp8_quant_1x128(wl.activations(M, K, seed, device=dev))
            qb, sb = fg.fp8_quant_128x128(wl.weights((N, K), seed + 1, device=dev))
            q = torch.empty((M, N), dtype=torch.uint8, device=dev)
            s = torch.empty((N // 128, fg.scale_ld(M)), dtype=torch.float32, device=dev)
            ws = None if (not workspace) else fg.gemm_workspace(M, N, K, device=dev)
            nb = M * K + N * K + M * (K // 128) * 4 + (N // 128) * (K // 128) * 4 + M * N + M * (N // 128) * 4
            return (lambda: fg.fp8_gemm_dense_quant_out(qa, sa, qb, sb, q, s, workspace=ws), nb, gemm_flops(M, N, K))
        if case == "gemm_then_quant":
            # the unfused pair: BF16 GEMM, then fp8_quant_1x128 of its output
            M, N, K = dims
            qa, sa = fg.fp8_quant_1x128(wl.activations(M, K, seed, device=dev))
            qb, sb = fg.fp8_quant_128x128(wl.weights((N, K), seed + 1, device=dev))
            c = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            q = torch.empty((M, N), dtype=torch.uint8, device=dev)
            s = torch.empty((N // 128, fg.scale_ld(M)), dtype=torch.float32, device=dev)
            ws = None if (not workspace) else fg.gemm_workspace(M, N, K, device=dev)

            def both():
                fg.fp8_gemm_dense_out(qa, sa, qb, sb, c, workspace=ws)
                fg.fp8_quant_1x128_out(c, q, s)
            nb = M * K + N * K + M * (K // 128) * 4 + (N // 128) * (K // 128) * 4 + M * N + M * (N // 128) * 4
            return both, nb, gemm_flops(M, N, K)
        if case == "dgrad":
            # dX[M, K] = dY[M, N] W[N, K]: the forward weight read as its own transpose
            M, N, K = dims
            qdy, sdy = fg.fp8_quant_1x128(wl.normal((M, N), seed, device=dev, dtype=torch.bfloat16))
            qw, sw = fg.fp8_quant_128x128(wl.weights((N, K), seed + 1, device=dev))
            dx = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
            ws = None if (not workspace) else fg.gemm_workspace(M, K, N, device=dev)
            return (lambda: fg.fp8_gemm_dgrad_out(qdy, sdy, qw, sw, dx, workspace=ws), gemm_bytes(M, K, N),
                    gemm_flops(M, K, N))
        if case in ("wgrad_dense", "wgrad_dense_bs"):
            # dW[N, C] += G^T X over T tokens: both operands 128x1 (pow2), FP32
            # accumulate; _bs applies the power-of-two scales in the tensor core
            T, N, C = dims
            kind = fg.SCALE_ROW_POW2 if case == "wgrad_dense_bs" else fg.SCALE_ROW
            qgT, sgT = fg.fp8_requant_128x1(wl.normal((T, N), seed, device=dev, dtype=torch.bfloat16), pow2=True)
            qx, sx = fg.fp8_quant_1x128(wl.activations(T, C, seed + 1, device=dev))
            qxT, sxT = fg.fp8_requant_128x1(qx.view(torch.float8_e4m3fn), sx, pow2=True)
            dw = torch.zeros((N, C), dtype=torch.float32, device=dev)
            ws = None if (not workspace) else fg.gemm_workspace(N, C, T, device=dev)
            nb = T * (N + C) + 2 * (T // 128) * (N + C) * 4 + 2 * N * C * 4   # dW read and written
            return (lambda: fg.fp8_gemm_dense_out(qgT, sgT, qxT, sxT, dw, b_scale_kind=kind, accumulate=True,
                                                  workspace=ws), nb, 2.0 * T * N * C)
        if case == "contig":
            E, T, N, K = dims
            counts = wl.zipf_counts(T, E, 1.1, seed)
            lay = wl.contig_layout(counts)
            Mt = len(lay.m_indices)
            qa, sa = fg.fp8_quant_1x128(wl.activations(Mt, K, seed, device=dev))
            qb, sb = fg.fp8_quant_128x128(wl.weights((E, N, K), seed + 1, device=dev))
            mi = torch.as_tensor(lay.m_indices, device=dev)
            c = torch.empty((Mt, N), dtype=torch.bfloat16, device=dev)
            nb = Mt * K + E * N * K + Mt * (K // 128) * 4 + E * (N // 128) * (K // 128) * 4 + T * N * 2
            return (lambda: fg.fp8_gemm_grouped_contig_out(qa, sa, qb, sb, mi, c), nb, 2.0 * T * N * K)
        if case == "masked":
            E, Mmax, N, K = dims
            counts = wl.masked_counts(E, Mmax, seed)
            qa, sa = fg.fp8_quant_1x128(wl.activations(E * Mmax, K, seed, device=dev))
            qa, sa = qa.view(E, Mmax, K), sa.view(K // 128, -1)
            sa3 = torch.empty((E, K // 128, fg.scale_ld(Mmax)), dtype=torch.float32, device=dev)
            for e in range(E):
                sa3[e, :, :Mmax] = sa[:, e * Mmax:(e + 1) * Mmax]
            qb, sb = fg.fp8_quant_128x128(wl.weights((E, N, K), seed + 1, device=dev))
            mm = torch.as_tensor(counts, device=dev)
            c = torch.empty((E, Mmax, N), dtype=torch.bfloat16, device=dev)
            T = int(counts.sum())
            nb = T * K + E * N * K + T * N * 2
            return (lambda: fg.fp8_gemm_grouped_masked_out(qa, sa3, qb, sb, mm, c, expected_m=Mmax), nb,
                    2.0 * T * N * K)
        if case == "wgrad":
            # per expert dW_e[N, C] = G_e^T X_e over its valid tokens: operands
            # requantized to 128x1 tiles with power-of-2 scales, FP32 out
            E, Tmax, N, C = dims
            counts = wl.masked_counts(E, Tmax, seed)
            vr = torch.as_tensor(counts, device=dev)
            g = wl.normal((E, Tmax, N), seed, device=dev, dtype=torch.bfloat16)
            x = wl.activations(E * Tmax, C, seed + 1, device=dev).view(E, Tmax, C)
            qgT, sgT = fg.fp8_requant_128x1(g, None, vr, pow2=True)
            qxT, sxT = fg.fp8_requant_128x1(x.contiguous(), None, vr, pow2=True)
            out = torch.zeros((E, N, C), dtype=torch.float32, device=dev)
            T = int(counts.sum())
            nb = T * (N + C) + E * N * C * 4
            return (lambda: fg.fp8_gemm_grouped_masked_out(qgT, sgT, qxT, sxT, vr, out, b_scale_kind=fg.SCALE_ROW,
                                                           mask_dim=fg.MASK_K, expected_m=Tmax),
                    nb, 2.0 * T * N * C)
        if case == "quant1x128":
            M, K = dims
            x = wl.activations(M, K, seed, device=dev)
            q = torch.empty((M, K), dtype=torch.uint8, device=dev)
            s = torch.empty((K // 128, fg.scale_ld(M)), dtype=torch.float32, device=dev)
            return lambda: fg.fp8_quant_1x128_out(x, q, s), quant_1x128_bytes(M, K), None
        if case == "quant128x128":
            N, K = dims
            w = wl.weights((N, K), seed + 1, device=dev)
            q = torch.empty((N, K), dtype=torch.uint8, device=dev)
            s = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=dev)
            return lambda: fg.fp8_quant_128x128_out(w, q, s), quant_128x128_bytes(N, K), None
        if case == "requant":
            T, C = dims
            x = wl.activations(T, C, seed, device=dev)
            qT = torch.empty((C, T), dtype=torch.uint8, device=dev)
            sT = torch.empty((T // 128, fg.scale_ld(C)), dtype=torch.float32, device=dev)
            out_bytes = T * C + (T // 128) * C * 4
            if src == "e4m3":
                qa, sa = fg.fp8_quant_1x128(x)
                return (lambda: fg.fp8_requant_128x1_out(qa.view(torch.float8_e4m3fn), sa, qT, sT, pow2=True),
                        T * C + T * (C // 128) * 4 + out_bytes, None)
            xs = x if src == "bf16" else x.float()
            return (lambda: fg.fp8_requant_128x1_out(xs, None, qT, sT, pow2=True),
                    T * C * xs.element_size() + out_bytes, None)
        raise SystemExit(f"unknown case {case}")

    # Independent buffer sets, called round robin, so that the working set
    # of consecutive calls exceeds the 126 MB L2 (every call reads from HBM).
    first = make(1001)
    nbytes, work = first[1], first[2]
    nsets = 1 if not rotate else max(1, min(8, -(-L2_ROTATE_BYTES // max(1, nbytes))))
    fns = [first[0]] + [make(1001 + 10 * i)[0] for i in range(1, nsets)]
    unit = "TFLOP/s" if work is not None else "GB/s"
    calls = [0]

    def fn():
        fns[calls[0] % nsets]()
        calls[0] += 1

    for _ in range(warmup):
        fn()
    fg.check()
    # R calls captured in one CUDA graph: replays keep host launch overhead
    # out of the per-call device time.
    reps = -(-max(1, graph_reps) // nsets) * nsets  # whole rounds over the buffer sets
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # first call outside capture (one-time setup)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(reps):
                fn()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record()
        graph.replay()
        e_.record()
        times.append((s_, e_))
    torch.cuda.synchronize()
    fg.check()
    ms = [a.elapsed_time(b) / reps for a, b in times]
    med = statistics.median(ms)
    out = {"case": case, "shape": dims, "ms_median": round(med, 5), "ms_min": round(min(ms), 5),
           "bytes": int(nbytes), "GB/s": round(nbytes / (med * 1e-3) / 1e9, 1), "graph_reps": reps,
           "buffer_sets": nsets}
    if case == "requant":
        out["src"] = src
    if work is not None:
        out["flops"] = work
        out["TFLOP/s"] = round(work / (med * 1e-3) / 1e12, 1)
    del graph, fns, first
    torch.cuda.empty_cache()
    return out


def run_case(args):
    """--case mode: time one kernel on --shape and print one JSON line."""
    dims = [int(v) for v in args.shape.split(",")]
    out = time_case(args.case, dims, args.src, args.steps, args.warmup, args.graph_reps,
                    rotate=not args.no_rotate, workspace=not args.no_workspace)
    out.pop("flops", None)
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--src", choices=["e4m3", "bf16", "fp32"], default="e4m3",
                    help="requant case: source type (E4M3 with 1x128 scales, BF16 or FP32)")
    ap.add_argument("--case", choices=["gemm", "gemm_quant", "gemm_then_quant", "dgrad", "wgrad_dense",
                                       "wgrad_dense_bs", "contig",
                                       "masked", "wgrad", "quant1x128", "quant128x128", "requant"],
                    default=None,
                    help="time a single kernel on --shape instead of the full step")
    ap.add_argument("--shape", default="4096,7168,7168")
    ap.add_argument("--graph-reps", type=int, default=10, help="calls per captured graph in --case mode")
    ap.add_argument("--no-workspace", action="store_true",
                    help="--case gemm: pass no Stream-K workspace (tiles are never split along K)")
    ap.add_argument("--no-rotate", action="store_true",
                    help="--case mode: reuse one buffer set (L2-warm when it fits in L2)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the graph-timed entries of the other workloads")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.case is not None:
        run_case(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local_rank)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
