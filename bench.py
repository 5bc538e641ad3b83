#!/usr/bin/env python3
"""Benchmark of the V:N:M hot path on GB300: magnitude prune-and-encode of a
dense fp16 weight matrix (vnm_compress) followed by the SpMM C = A_vnm . B
(vnm_spmm), through libvnm's C ABI.

One step = one pass of the whole path over one batch of synthetic input:
vnm_compress(W) then vnm_spmm(B) -> C, for the square compute-bound workload
(A 4096 x 4096, V = 64, 2:8, B 4096 x 2048, fp16 C; --workload/--case pick
another). Inputs are resident in HBM when the timed region starts; the steps
rotate over enough distinct input/output sets that each set is evicted from
L2 before it is used again. The K timed steps are captured once in a CUDA
graph and replayed between two events; each kernel's own launch duration
comes from graphs of K launches of that kernel alone over the same sets.

Output: one JSON line (rank 0). ``value`` is the dense-equivalent TFLOP/s of
the whole step (2*R*N*K per step over the step time); ``e2e`` is the same
metric through the public API with host buffers, copies included; the
``roofline`` object covers the kernel that takes most of the step.

``--impl reference`` times the CPU oracle (the only other implementation of
this path here) on a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "V:N:M SpMM TFLOP/s (dense-equiv & effective), % of sparse-TC/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["vnm", "reference"], default="vnm")
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--case", type=int, default=0)
    ap.add_argument("--rows", type=int, default=0,
                    help="override R of the chosen case (a smaller case of the same kernels, e.g. for ncu)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target seconds of oracle work")
    ap.add_argument("--clock-seconds", type=float, default=2.0, help="seconds of load around the timed region")
    ap.add_argument("--no-context", action="store_true", help="skip the dense torch.matmul context timing")
    ap.add_argument("--e2e-in-streams", type=int, default=1,
                    help="streams that carry a step's host-to-device copies (row chunks of W, then B)")
    ap.add_argument("--no-per-config", action="store_true", help="skip the per-workload kernel table")
    ap.add_argument("--per-config-launches", type=int, default=10,
                    help="kernel launches per graph in the per-workload table (median of 10 replays)")
    ap.add_argument("--profile-op", choices=["gemm_compress", "linear", "bitmap"], default=None,
                    help="run a few launches of one of the other entry points on its first table case and exit "
                         "(for ncu captures)")
    return ap.parse_args()


def profile_op(op: str) -> None:
    """A few launches of vnm_gemm_compress, vnm_linear or vnm_bitmap_spmm on
    a case of their bench tables, checked for a clean status (for ncu
    captures)."""
    import torch

    from structured_sparse_matmul_gb300 import vnm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    if op == "bitmap":
        R, K, sp = BITMAP_CASES[0]
        W = (torch.randn(R, K, device=dev, generator=gen) * 0.02).half()
        cut = W.abs().float().flatten().kthvalue(max(1, int(sp * R * K))).values
        W[W.abs().float() <= cut] = 0
        Bm = vnm.bitmap_encode(W)
        B = torch.randn(K, 1, device=dev, generator=gen).half()
        C = torch.empty(R, 1, dtype=torch.float16, device=dev)
        ws = torch.empty(max(1, vnm.bitmap_spmm_workspace_size(R, K, 1) // 4), dtype=torch.float32, device=dev)
        for _ in range(3):
            vnm.bitmap_spmm(Bm, B, C, workspace=ws)
        torch.cuda.synchronize(dev)
        print(f"{op}: 3 launches, ok")
        return
    if op == "gemm_compress":
        R, K, D, V, M = GEMM_COMPRESS_CASES[1]
        A = vnm.vnm_matrix_alloc(R, K, V, M, dev)
        X = torch.randn(R, D, device=dev, generator=gen).half()
        Y = torch.randn(K, D, device=dev, generator=gen).half()
        for _ in range(3):
            vnm.vnm_gemm_compress(A, X, Y)
    else:
        R, K, T, V, M = LINEAR_CASES[0]
        A = vnm.vnm_matrix_alloc(R, K, V, M, dev)
        vnm.vnm_compress(A, (torch.randn(R, K, device=dev, generator=gen) * 0.02).half())
        X = torch.randn(T, K, device=dev, generator=gen).half()
        Y = torch.empty(T, R, dtype=torch.float16, device=dev)
        bias = torch.randn(R, device=dev, generator=gen).half()
        for _ in range(3):
            vnm.vnm_linear(A, X, Y, bias, vnm.VNM_ACT_GELU)
    torch.cuda.synchronize(dev)
    st = vnm.vnm_get_status(A)
    if st != vnm.VNM_OK:
        raise SystemExit(f"status {vnm.status_string(st)}")
    print(f"{op}: 3 launches, status ok")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def dist_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = [p for (t, p) in self.rows if t0 <= t <= t1] or [p for (_, p) in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in rows if num(p[1]) is not None]
        smax = [num(p[2]) for p in rows if num(p[2]) is not None]
        reasons = set()
        for p in rows:
            for name, val in (("hw_slowdown", p[5]), ("hw_thermal_slowdown", p[6]), ("sw_thermal_slowdown", p[7]),
                              ("sw_power_cap", p[8])):
                if val.lower().startswith("active"):
                    reasons.add(name)
        power = [num(p[3]) for p in rows if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(power) if power else None}


# --------------------------------------------------------------------------- CPU oracle

def host_cpu() -> str:
    """The host CPU's model, as the kernel reports it (Arm: implementer and part)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    if "CPU part" in fields:
        return f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    return platform.processor() or platform.machine()


def time_oracle(case, seconds: float):
    """Time the CPU oracle (compress + fp32-accumulate SpMM, as it stands) on
    the first S V-block rows of the workload, S chosen for ~``seconds``."""
    import numpy as np

    import oracle
    from structured_sparse_matmul_gb300 import inputs, workloads

    V = case.V
    # one V-block row first, to size the sample
    def one(rows):
        W = inputs.normal_f16((rows, case.K), case.seed, case.a_stream, workloads.A_SIGMA)
        B = inputs.normal_f16((case.K, case.N), case.seed, case.b_stream, workloads.B_SIGMA)
        t0 = time.perf_counter()
        values, meta, colidx = oracle.compress(W, V, case.M)
        oracle.spmm(values, meta, colidx, rows, case.K, V, case.M, B)
        return time.perf_counter() - t0

    rows = V
    t1 = one(rows)
    blocks = max(1, min(case.R // V, int(seconds / max(t1, 1e-6))))
    rows = blocks * V
    t = one(rows) if blocks > 1 else t1
    flops = 2.0 * rows * case.N * case.K
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"compress + fp32 SpMM of rows 0..{rows - 1} ({blocks} of {case.R // V} V-block rows) of "
                      f"{case.R}x{case.K}x{case.N}, {t:.2f} s single-threaded",
            "seconds": t, "row_parallel": time_oracle_rows_parallel(case, seconds, t1)}


def time_oracle_rows_parallel(case, seconds: float, t_block: float):
    """The same oracle calls, row-parallel: one host thread per core, each on
    its own whole V-block rows (the C oracle runs outside the GIL)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from structured_sparse_matmul_gb300 import inputs, workloads

    V = case.V
    threads = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))
    per = max(1, min(max(1, (case.R // V) // threads), int(seconds / max(t_block, 1e-6))))
    threads = max(1, min(threads, (case.R // V) // per))
    rows = threads * per * V
    W = inputs.normal_f16((rows, case.K), case.seed, case.a_stream, workloads.A_SIGMA)
    B = inputs.normal_f16((case.K, case.N), case.seed, case.b_stream, workloads.B_SIGMA)

    def work(i):
        Wi = W[i * per * V:(i + 1) * per * V]
        values, meta, colidx = oracle.compress(Wi, V, case.M)
        oracle.spmm(values, meta, colidx, per * V, case.K, V, case.M, B)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        list(ex.map(work, range(threads)))
        t = time.perf_counter() - t0
    flops = 2.0 * rows * case.N * case.K
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": threads,
            "sample": f"compress + fp32 SpMM of rows 0..{rows - 1} ({threads * per} of {case.R // V} V-block rows), "
                      f"{per} V-block rows per thread on {threads} threads, {t:.2f} s"}


# --------------------------------------------------------------------------- reference arm

def run_reference(args, case):
    """The oracle as it stands, on the host: W untimed warm-up steps, then K
    timed steps, each a bounded sample of the workload (whole V-block rows
    of compress + fp32 SpMM), sized so that all K + W steps take about 2.5
    minutes (at most --cpu-seconds each)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from structured_sparse_matmul_gb300 import inputs, workloads

    V = case.V
    budget = max(0.05, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    B = inputs.normal_f16((case.K, case.N), case.seed, case.b_stream, workloads.B_SIGMA)

    def sample(blocks):
        rows = blocks * V
        W = inputs.normal_f16((rows, case.K), case.seed, case.a_stream, workloads.A_SIGMA)
        t0 = time.perf_counter()
        values, meta, colidx = oracle.compress(W, V, case.M)
        oracle.spmm(values, meta, colidx, rows, case.K, V, case.M, B)
        return time.perf_counter() - t0

    t1 = sample(1)
    blocks = max(1, min(case.R // V, int(budget / max(t1, 1e-6))))
    for _ in range(args.warmup):
        sample(blocks)
    total = 0.0
    for _ in range(max(1, args.steps)):
        total += sample(blocks)
    steps = max(1, args.steps)
    flops = 2.0 * blocks * V * case.N * case.K * steps
    value = flops / total / 1e12
    desc = (f"compress + fp32 SpMM of rows 0..{blocks * V - 1} ({blocks} of {case.R // V} V-block rows) of "
            f"{case.R}x{case.K}x{case.N} per step, single-threaded, {total / steps:.3f} s a step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": args.warmup, "ms_per_step": total / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": config_of(case, None),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": 1, "kind": "oracle", "sample": desc,
                         "host_cpu": host_cpu(), "host_threads": os.cpu_count()},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# Sources of each profiled kernel: a summary's DRAM traffic is used only
# while these files are unchanged since the capture.
REPLAYS = 10  # replays of a timed graph whose median is reported (per kernel and per workload case)

KERNEL_SOURCES = {
    "spmm_tc_kernel": ["spmm_tc.cu", "vnm_ptx.cuh", "vnm_internal.h", "api.cu"],  # api.cu: the tile plan
    "lift_expand_kernel": ["spmm_tc.cu", "vnm_internal.h", "api.cu"],
    "compress": ["compress.cu", "vnm_internal.h"],
}


def sources_sha256(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "structured_sparse_matmul_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch of `kernel` on `workload` from the
    ncu summary under profiles/, or None when there is none or the kernel's
    sources changed after it was taken."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.startswith(" "):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    try:
        if fields.get("source_sha256") != sources_sha256(kernel):
            return None
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError, OSError):
        return None


def workload_tag(case) -> str:
    return f"{case.R}x{case.K}x{case.N}_v{case.V}m{case.M}"


def config_of(case, l2_note):
    c = {"workload": (f"V:N:M magnitude compress + SpMM, A {case.R}x{case.K} fp16 N(0,0.02) {case.V}:2:{case.M} "
                      f"({100 * (1 - 2 / case.M):.1f}% sparse), B {case.K}x{case.N} fp16 N(0,1), "
                      f"{'fp32' if case.c_f32 else 'fp16'} C, fp32 accumulate"),
         "R": case.R, "K": case.K, "N": case.N, "V": case.V, "M": case.M,
         "c_dtype": "f32" if case.c_f32 else "f16"}
    if l2_note:
        c["l2"] = l2_note
    return c


# --------------------------------------------------------------------------- per-workload table

def roofline_of(case, peaks, spmm_us, a_bytes):
    """Roofline of one SpMM launch: the bound (tensor or HBM, by the larger
    roofline time), the fraction achieved, and the roofline time."""
    c_bytes = case.R * case.N * (4 if case.c_f32 else 2)
    byts = a_bytes + 2 * case.K * case.N + c_bytes
    t_tc = case.effective_flops() / (peaks["bf16_tflops"] * 1e12)
    t_hbm = byts / (peaks["hbm_gbs"] * 1e9)
    t_roof = max(t_tc, t_hbm)
    return {"bound": "tensor" if t_tc >= t_hbm else "hbm", "t_roof_us": t_roof * 1e6,
            "frac": t_roof / (spmm_us * 1e-6), "bytes": byts, "effective_flops": case.effective_flops()}


def _time_graph(dev, fn, launches: int) -> float:
    """Median of REPLAYS replays of a CUDA graph of `launches` calls fn(i, stream),
    in microseconds per call (events on the replaying stream)."""
    import torch
    cur = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        fn(0, side)  # warm (and the kernels' one-time set-up) outside the capture
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for i in range(launches):
                fn(i, side)
    torch.cuda.synchronize(dev)
    g.replay()
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(REPLAYS):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        g.replay()
        e1.record(cur)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1) * 1e3 / launches)
    return statistics.median(ts)


# The fused dense GEMM + prune-and-encode (vnm_gemm_compress) on attention-
# score-like products X . Y^T (X, Y: L tokens x head dimension D), the
# operand DFSS prunes on the fly, and one weight-like product with a long D.
GEMM_COMPRESS_CASES = [
    # R, K, D, V, M
    (4096, 4096, 64, 1, 4),
    (4096, 4096, 128, 16, 8),
    (8192, 8192, 128, 64, 8),
    (4096, 4096, 4096, 64, 8),
]


def measure_gemm_compress(dev, peaks, launches: int):
    """vnm_gemm_compress against the same result in two launches (dense
    torch.matmul writing W, then vnm_compress reading it), both timed like
    the per-workload table, with the fused kernel's roofline: dense flops
    2*R*K*D against the measured tensor peak, bytes X + Y + the compressed
    arrays against HBM."""
    import torch

    from structured_sparse_matmul_gb300 import vnm

    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20))
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    out = {}
    for (R, K, D, V, M) in GEMM_COMPRESS_CASES:
        vb, mb, cb = vnm.vnm_sizes(R, K, V, M)
        set_bytes = 2 * (R + K) * D + vb + mb + cb
        n_sets = max(2, math.ceil(2 * l2 / set_bytes) + 1)
        sets = [{"X": torch.randn(R, D, device=dev, generator=gen).half(),
                 "Y": torch.randn(K, D, device=dev, generator=gen).half(),
                 "A": vnm.vnm_matrix_alloc(R, K, V, M, dev)} for _ in range(n_sets)]
        W = torch.empty(R, K, dtype=torch.float16, device=dev)

        def fused(i, st):
            x = sets[i % n_sets]
            vnm.vnm_gemm_compress(x["A"], x["X"], x["Y"], stream=st)

        def unfused(i, st):
            x = sets[i % n_sets]
            torch.matmul(x["X"], x["Y"].t(), out=W)
            vnm.vnm_compress(x["A"], W, stream=st)

        t_f = _time_graph(dev, fused, launches)
        t_u = _time_graph(dev, unfused, launches)
        for x in sets:
            st_ = vnm.vnm_get_status(x["A"])
            if st_ != vnm.VNM_OK:
                raise RuntimeError(f"kernel status {vnm.status_string(st_)} in gemm_compress {R}x{K}x{D}")
        flops = 2.0 * R * K * D
        byts = 2 * (R + K) * D + vb + mb + cb
        t_roof = max(flops / (peaks["bf16_tflops"] * 1e12), byts / (peaks["hbm_gbs"] * 1e9)) * 1e6
        out[f"{R}x{K}x{D}-{V}:2:{M}"] = {
            "fused_us": t_f, "matmul_then_compress_us": t_u,
            "roofline": {"bound": "tensor" if flops / peaks["bf16_tflops"] / 1e12 > byts / peaks["hbm_gbs"] / 1e9
                         else "hbm", "t_roof_us": t_roof, "frac": t_roof / t_f},
            "sets": n_sets}
        del sets, W
        torch.cuda.empty_cache()
    return {"launches_per_graph": launches, "replays": REPLAYS, "statistic": "median",
            "inputs": "torch seeded device generator, X, Y ~ N(0, 1)",
            "l2_eviction": "rotating input sets of more than twice the L2 in each graph", "cases": out}


# The Linear-layer form Y = act(X . A^T + bias) on the transformer-encoder
# linear shapes of workload 3 (8192 tokens), V = 128.
LINEAR_CASES = [
    # R (out features), K (in features), T (tokens), V, M
    (4096, 1024, 8192, 128, 4),
    (4096, 1024, 8192, 128, 8),
    (1024, 4096, 8192, 128, 4),
    (1024, 4096, 8192, 128, 16),
]


def measure_linear(dev, peaks, launches: int):
    """vnm_linear with and without a bias + GELU epilogue, against what the
    SpMM alone needs for the same layer (X transposed, vnm_spmm, C transposed
    back) and dense torch.nn.functional.linear + GELU (context). Timed like
    the per-workload table; the roofline of the plain vnm_linear launch is the
    SpMM's (effective flops, bytes A + X + Y)."""
    import torch
    import torch.nn.functional as F

    from structured_sparse_matmul_gb300 import vnm

    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20))
    gen = torch.Generator(device=dev)
    gen.manual_seed(5151)
    out = {}
    for (R, K, T, V, M) in LINEAR_CASES:
        vb, mb, cb = vnm.vnm_sizes(R, K, V, M)
        set_bytes = vb + mb + cb + 2 * T * K + 2 * T * R
        n_sets = max(2, math.ceil(2 * l2 / set_bytes) + 1)
        Wd = (torch.randn(R, K, device=dev, generator=gen) * 0.02).half()
        bias = (torch.randn(R, device=dev, generator=gen) * 0.5).half()
        A = vnm.vnm_matrix_alloc(R, K, V, M, dev)
        vnm.vnm_compress(A, Wd)
        Wp = torch.empty_like(Wd)
        vnm.vnm_decompress(A, Wp)  # the pruned weight, dense (for the dense context line)
        sets = [{"X": torch.randn(T, K, device=dev, generator=gen).half(),
                 "Y": torch.empty(T, R, dtype=torch.float16, device=dev)} for _ in range(n_sets)]
        ws = torch.empty(max(1, vnm.vnm_linear_workspace_size(A, T)), dtype=torch.uint8, device=dev)
        Xt = torch.empty(K, T, dtype=torch.float16, device=dev)
        Ct = torch.empty(R, T, dtype=torch.float16, device=dev)
        sws = vnm.workspace_for(A, T, dev)

        def lin(i, st, b=None, act=vnm.VNM_ACT_NONE):
            x = sets[i % n_sets]
            vnm.vnm_linear(A, x["X"], x["Y"], b, act, workspace=ws, stream=st)

        def via_spmm(i, st):
            x = sets[i % n_sets]
            Xt.copy_(x["X"].t())
            vnm.vnm_spmm(A, Xt, Ct, workspace=sws, stream=st)
            x["Y"].copy_(Ct.t())

        def dense(i, st):
            x = sets[i % n_sets]
            F.gelu(F.linear(x["X"], Wp, bias))

        t_plain = _time_graph(dev, lin, launches)
        t_epi = _time_graph(dev, lambda i, st: lin(i, st, bias, vnm.VNM_ACT_GELU), launches)
        t_via = _time_graph(dev, via_spmm, launches)
        try:
            t_dense = _time_graph(dev, dense, launches)
        except Exception as exc:  # context only
            t_dense = f"unavailable: {exc}"
        st_ = vnm.vnm_get_status(A)
        if st_ != vnm.VNM_OK:
            raise RuntimeError(f"kernel status {vnm.status_string(st_)} in vnm_linear {R}x{K}x{T}")
        eff = 2.0 * R * T * K * 2 / M
        byts = vb + mb + cb + 2 * T * K + 2 * T * R
        t_roof = max(eff / (peaks["bf16_tflops"] * 1e12), byts / (peaks["hbm_gbs"] * 1e9)) * 1e6
        out[f"Y[{T}x{R}] = X[{T}x{K}] . A^T, {V}:2:{M}"] = {
            "vnm_linear_us": t_plain, "vnm_linear_bias_gelu_us": t_epi,
            "transpose_spmm_transpose_us": t_via, "dense_linear_gelu_us": t_dense,
            "roofline": {"t_roof_us": t_roof, "frac": t_roof / t_plain}, "sets": n_sets}
        del sets, Wd, Wp, Xt, Ct, ws
        torch.cuda.empty_cache()
    return {"launches_per_graph": launches, "replays": REPLAYS, "statistic": "median",
            "inputs": "torch seeded device generator, W ~ N(0, 0.02), X ~ N(0, 1), bias ~ N(0, 0.25)",
            "l2_eviction": "rotating X / Y sets of more than twice the L2 in each graph", "cases": out}


# Decode-time products with unstructured sparsity in the bitmap format
# (Coruscant: 30-70% sparsity, Llama-style projections): R, K, sparsity.
BITMAP_CASES = [(4096, 4096, 0.5), (11008, 4096, 0.5), (4096, 11008, 0.5), (4096, 4096, 0.3), (4096, 4096, 0.7)]
BITMAP_N = (1, 8, 16)


def measure_bitmap(dev, peaks, launches: int):
    """vnm_bitmap_spmm on magnitude-pruned N(0, 0.02) weights (the smallest
    |w| zeroed), timed like the per-workload table, against the HBM roofline
    of its bytes (bitmaps + offsets + values + B + C) and dense torch.matmul
    on the same shape (context)."""
    import torch

    from structured_sparse_matmul_gb300 import vnm

    gen = torch.Generator(device=dev)
    gen.manual_seed(6161)
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20))
    out = {}
    for (R, K, sp) in BITMAP_CASES:
        W = (torch.randn(R, K, device=dev, generator=gen) * 0.02).half()
        cut = W.abs().float().flatten().kthvalue(max(1, int(sp * R * K))).values
        W[W.abs().float() <= cut] = 0
        A = vnm.bitmap_encode(W)
        a_bytes = A.bitmaps.numel() * 8 + A.offsets.numel() * 4 + A.bases.numel() * 8 + A.values.numel() * 2
        n_sets = max(2, math.ceil(2 * l2 / a_bytes) + 1)
        mats = [A] + [vnm.bitmap_encode(W) for _ in range(n_sets - 1)]
        for N in BITMAP_N:
            Bs = [torch.randn(K, N, device=dev, generator=gen).half() for _ in range(n_sets)]
            Cs = [torch.empty(R, N, dtype=torch.float16, device=dev) for _ in range(n_sets)]
            nws = vnm.bitmap_spmm_workspace_size(R, K, N)
            ws = torch.empty(max(1, nws // 4), dtype=torch.float32, device=dev)

            def run(i, st):
                vnm.bitmap_spmm(mats[i % n_sets], Bs[i % n_sets], Cs[i % n_sets], workspace=ws, stream=st)

            def dense(i, st):
                torch.matmul(W, Bs[i % n_sets])

            t = _time_graph(dev, run, launches)
            td = _time_graph(dev, dense, launches)
            byts = a_bytes + 2 * K * N + 2 * R * N
            t_roof = byts / (peaks["hbm_gbs"] * 1e9) * 1e6
            out[f"{R}x{K}, {int(sp * 100)}% zeros, N={N}"] = {
                "bitmap_spmm_us": t, "dense_matmul_us": td,
                "roofline": {"bound": "hbm", "t_roof_us": t_roof, "frac": t_roof / t},
                "format_bytes_vs_dense": a_bytes / (2.0 * R * K)}
        del mats, W, A
        torch.cuda.empty_cache()
    return {"launches_per_graph": launches, "replays": REPLAYS, "statistic": "median",
            "inputs": "torch seeded device generator, W ~ N(0, 0.02) with the smallest |w| zeroed, B ~ N(0, 1)",
            "cases": out}


def measure_energy(dev):
    """Energy (magnitude preservation) of the three selection policies at the
    V:N:M densities 2/4 .. 2/40 on a synthetic N(0, 0.02) weight of the
    768 x 768 shape of the pages' Figure 11 study (VENOM section 5; 768 x 960
    for 2:40, which 768 columns do not divide), and the time of one vnm_energy
    call (its host read-back included) on a 4096 x 4096 weight."""
    import torch

    from structured_sparse_matmul_gb300 import inputs, vnm

    table = {}
    # 768 x 768 for M dividing 768; 768 x 960 for M = 40 (the densest the study goes to)
    for M, K, seed in ((4, 768, 1011), (8, 768, 1011), (16, 768, 1011), (32, 768, 1011), (40, 960, 1013)):
        W = torch.from_numpy(inputs.normal_f16((768, K), seed, 0, 0.02)).to(dev)
        row = {"weight": f"768x{K}"}
        A1 = vnm.vnm_matrix_alloc(768, K, 16, M, dev)
        row["unstructured"] = vnm.vnm_energy(A1, W, vnm.VNM_PATTERN_UNSTRUCTURED)[0]
        for V in (1, 16, 32, 64, 128):
            A = vnm.vnm_matrix_alloc(768, K, V, M, dev)
            vnm.vnm_compress(A, W)
            row[f"{V}:2:{M}"] = vnm.vnm_energy(A, W, vnm.VNM_PATTERN_VNM)[0]
        for l in (4, 8, 16, 32):
            A = vnm.vnm_matrix_alloc(768, K, l, M, dev)
            row[f"vw_{l}"] = vnm.vnm_energy(A, W, vnm.VNM_PATTERN_VECTORWISE)[0]
        table[f"density 2/{M}"] = row
    big = torch.from_numpy(inputs.normal_f16((4096, 4096), 1012, 0, 0.02)).to(dev)
    A = vnm.vnm_matrix_alloc(4096, 4096, 64, 8, dev)
    vnm.vnm_compress(A, big)
    ws = torch.empty(vnm.vnm_energy_workspace_size(A), dtype=torch.uint8, device=dev)
    times = {}
    for name, pat in (("vnm", vnm.VNM_PATTERN_VNM), ("unstructured", vnm.VNM_PATTERN_UNSTRUCTURED),
                      ("vectorwise", vnm.VNM_PATTERN_VECTORWISE)):
        ts = []
        for _ in range(REPLAYS):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            vnm.vnm_energy(A, big, pat, workspace=ws)
            ts.append((time.perf_counter() - t0) * 1e6)
        times[name] = statistics.median(ts)
    return {"weight": "768x768 N(0, 0.02), synthetic (the shape of the pages' Figure 11 study); 768x960 for 2:40",
            "energy": table,
            "call_us_4096x4096_v64m8": times}


def measure_per_config(dev, peaks, launches: int):
    """Every case of workloads 1-5: SpMM and compress launch times (median of
    REPLAYS replays of a graph of `launches` launches over rotating input sets that
    together exceed twice the L2), the SpMM roofline, the plan, and dense
    torch.matmul on the same shape (context). Inputs come from torch's seeded
    device generator with the workloads' distributions (A ~ N(0, 0.02),
    B ~ N(0, 1)); the kernels' speed does not depend on which generator
    drew them."""
    import torch

    from structured_sparse_matmul_gb300 import vnm, workloads

    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20))
    cur = torch.cuda.current_stream(dev)
    gen = torch.Generator(device=dev)

    def time_graph(fn):
        side = torch.cuda.Stream(dev)
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            fn(0, side)  # warm (and the kernels' one-time set-up) outside the capture
            side.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for i in range(launches):
                    fn(i, side)
        torch.cuda.synchronize(dev)
        g.replay()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(REPLAYS):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            g.replay()
            e1.record(cur)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1) * 1e3 / launches)
        return statistics.median(ts)

    table = {}
    for w in range(1, 6):
        for case in workloads.workload_cases(w):
            gen.manual_seed(case.seed)
            R, K, N, V, M = case.R, case.K, case.N, case.V, case.M
            c_dtype = torch.float32 if case.c_f32 else torch.float16
            vb, mb, cb = vnm.vnm_sizes(R, K, V, M)
            set_bytes = 2 * R * K + vb + mb + cb + 2 * K * N + R * N * (4 if case.c_f32 else 2)
            n_sets = max(2, math.ceil(2 * l2 / set_bytes) + 1)
            sets = []
            for _ in range(n_sets):
                W = (torch.randn(R, K, device=dev, generator=gen) * workloads.A_SIGMA).half()
                A = vnm.vnm_matrix_alloc(R, K, V, M, dev)
                Bm = (torch.randn(K, N, device=dev, generator=gen) * workloads.B_SIGMA).half()
                C = torch.empty(R, N, dtype=c_dtype, device=dev)
                vnm.vnm_compress(A, W)
                sets.append({"A": A, "W": W, "B": Bm, "C": C, "ws": vnm.workspace_for(A, N, dev)})
            torch.cuda.synchronize(dev)
            plan = vnm.vnm_spmm_plan_query(sets[0]["A"], sets[0]["B"], c_dtype,
                                           0 if sets[0]["ws"] is None else sets[0]["ws"].numel() * 4)

            def spmm(i, st):
                x = sets[i % n_sets]
                vnm.vnm_spmm(x["A"], x["B"], x["C"], workspace=x["ws"], stream=st)

            def comp(i, st):
                x = sets[i % n_sets]
                vnm.vnm_compress(x["A"], x["W"], stream=st)

            def dense(i, st):
                x = sets[i % n_sets]
                torch.matmul(x["W"], x["B"])

            spmm_us = time_graph(spmm)
            comp_us = time_graph(comp)
            try:
                dense_us = time_graph(dense)
            except Exception as exc:  # context only
                dense_us = f"unavailable: {exc}"
            for x in sets:
                st_ = vnm.vnm_get_status(x["A"])
                if st_ != vnm.VNM_OK:
                    raise RuntimeError(f"kernel status {vnm.status_string(st_)} in {case.name}")
            roof = roofline_of(case, peaks, spmm_us, vb + mb + cb)
            comp_bytes = 2 * R * K + vb + mb + cb
            table[case.name] = {
                "spmm_us": spmm_us, "compress_us": comp_us,
                "spmm_effective_tflops": case.effective_flops() / (spmm_us * 1e-6) / 1e12,
                "spmm_dense_equiv_tflops": case.dense_flops() / (spmm_us * 1e-6) / 1e12,
                "roofline": {"bound": roof["bound"], "frac": roof["frac"], "t_roof_us": roof["t_roof_us"]},
                "compress_hbm_frac": comp_bytes / (comp_us * 1e-6) / (peaks["hbm_gbs"] * 1e9),
                "dense_matmul_us": dense_us, "plan": plan.as_dict(), "sets": n_sets,
            }
            del sets
            torch.cuda.empty_cache()
    return {"launches_per_graph": launches, "replays": REPLAYS, "statistic": "median",
            "inputs": "torch seeded device generator, A ~ N(0, 0.02), B ~ N(0, 1)",
            "l2_eviction": "rotating input sets of more than twice the L2 in each graph", "cases": table}


# --------------------------------------------------------------------------- main arm

def main():
    args = parse_args()
    if args.profile_op:
        profile_op(args.profile_op)
        return
    from structured_sparse_matmul_gb300 import workloads
    case = workloads.workload_cases(args.workload)[args.case]
    if args.rows:
        if args.rows % 128 or args.rows % case.V:
            raise SystemExit(f"--rows must be a multiple of 128 and of V={case.V}")
        case = dataclasses.replace(case, R=args.rows)
    if args.impl == "reference":
        world, _, _ = dist_env()
        dist_init(world, "gloo")
        run_reference(args, case)
        return

    import numpy as np
    import torch

    from structured_sparse_matmul_gb300 import inputs, vnm

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    vnm.lib()  # fails loudly if libvnm is not built

    peaks, peak_src = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))

    R, K, N, V, M = case.R, case.K, case.N, case.V, case.M
    c_dtype = torch.float32 if case.c_f32 else torch.float16
    W_h = inputs.normal_f16((R, K), case.seed, case.a_stream, workloads.A_SIGMA)
    B_h = inputs.normal_f16((K, N), case.seed, case.b_stream, workloads.B_SIGMA)
    vb, mb, cb = vnm.vnm_sizes(R, K, V, M)
    c_bytes = R * N * (4 if case.c_f32 else 2)
    set_bytes = 2 * R * K + 2 * K * N + c_bytes + vb + mb + cb
    n_sets = max(2, math.ceil(2 * l2 / set_bytes) + 1)

    W0 = torch.from_numpy(W_h).to(dev)
    B0 = torch.from_numpy(B_h).to(dev)
    sets = []
    for _ in range(n_sets):
        A = vnm.vnm_matrix_alloc(R, K, V, M, dev)
        sets.append({"A": A, "W": W0.clone(), "B": B0.clone(), "C": torch.empty((R, N), dtype=c_dtype, device=dev),
                     "ws": vnm.workspace_for(A, N, dev)})
    del W0, B0
    plan = vnm.vnm_spmm_plan_query(sets[0]["A"], sets[0]["B"], c_dtype,
                                   0 if sets[0]["ws"] is None else sets[0]["ws"].numel() * 4)
    splits = plan.splits if plan.path == vnm.VNM_PATH_TC else 1
    # compress, the SpMM, its split-K reduction, and for lift = 2 the kernel that writes A out as 2:4
    kernels_per_step = (1 + (1 if plan.path != vnm.VNM_PATH_NONE else 0) + (1 if splits > 1 else 0)
                        + (1 if plan.path == vnm.VNM_PATH_TC and plan.lift == 2 else 0))

    stream = torch.cuda.current_stream(dev)

    def step(i, comp=True, spmm=True):
        s = sets[i % n_sets]
        if comp:
            vnm.vnm_compress(s["A"], s["W"], stream=stream)
        if spmm:
            vnm.vnm_spmm(s["A"], s["B"], s["C"], workspace=s["ws"], stream=stream)

    # warm-up (eager), then check the status words
    for i in range(max(args.warmup, 1)):
        step(i)
    torch.cuda.synchronize(dev)
    for s in sets:
        st = vnm.vnm_get_status(s["A"])
        if st != vnm.VNM_OK:
            raise RuntimeError(f"kernel status {vnm.status_string(st)} during warm-up")

    # CUDA graphs over the same rotating sets, each captured once: K whole
    # steps on one stream (reported as the serial step), K SpMM launches and
    # K compress launches (each kernel's average launch duration, for the
    # breakdown and the roofline), and below the timed graph of K pipelined
    # steps. No timing event sits inside a graph (an event node adds
    # microseconds per kernel); cross-stream dependencies are graph edges.
    steps = args.steps

    def capture(**kw):
        nonlocal stream
        g = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream(dev)
        cap_stream.wait_stream(torch.cuda.current_stream(dev))
        prev = stream
        with torch.cuda.stream(cap_stream):
            stream = cap_stream
            with torch.cuda.graph(g, stream=cap_stream):
                for i in range(steps):
                    step(i, **kw)
        stream = prev
        torch.cuda.synchronize(dev)
        g.replay()  # warm replay
        torch.cuda.synchronize(dev)
        return g

    graph_serial = capture()
    graph_spmm = capture(comp=False)
    graph_comp = capture(spmm=False)

    # The timed graph: the same K steps with the compressions on one stream
    # and the products on another. Step i's SpMM waits for step i's compress;
    # step i's compress waits for the last SpMM that read its set. So step
    # i+1's compress runs while step i's SpMM finishes (on the SMs its last
    # wave of tiles leaves idle); every step still compresses its W and
    # multiplies its B.
    def capture_pipelined():
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        s_c, s_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        with torch.cuda.stream(cap), torch.cuda.graph(g, stream=cap):
            s_c.wait_stream(cap)
            s_s.wait_stream(cap)
            ev_c = [torch.cuda.Event() for _ in range(steps)]
            ev_s = [torch.cuda.Event() for _ in range(steps)]
            for i in range(steps):
                st = sets[i % n_sets]
                if i >= n_sets:
                    s_c.wait_event(ev_s[i - n_sets])
                vnm.vnm_compress(st["A"], st["W"], stream=s_c)
                ev_c[i].record(s_c)
                s_s.wait_event(ev_c[i])
                vnm.vnm_spmm(st["A"], st["B"], st["C"], workspace=st["ws"], stream=s_s)
                ev_s[i].record(s_s)
            cap.wait_stream(s_c)
            cap.wait_stream(s_s)
        torch.cuda.synchronize(dev)
        g.replay()  # warm replay
        torch.cuda.synchronize(dev)
        return g

    graph = capture_pipelined()

    def timed(g):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    # clocks: sample across a load phase that brackets the timed replay
    sampler = ClockSampler(local)
    sampler.start()
    t_load0 = time.time()
    while time.time() - t_load0 < args.clock_seconds / 2:
        graph.replay()
        torch.cuda.synchronize(dev)
    dist_barrier(world, dev)
    torch.cuda.synchronize(dev)
    elapsed_ms = timed(graph)
    dist_barrier(world, dev)
    serial_ms = timed(graph_serial) / steps
    # each kernel's average launch duration: median of REPLAYS replays of its graph
    spmm_ms = statistics.median(timed(graph_spmm) for _ in range(REPLAYS)) / steps
    comp_ms = statistics.median(timed(graph_comp) for _ in range(REPLAYS)) / steps
    # launch floor: K empty kernels (a sleep of zero cycles), captured and
    # timed the same way
    empty_ms = None
    try:
        g_empty = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap), torch.cuda.graph(g_empty, stream=cap):
            for _ in range(steps):
                torch.cuda._sleep(0)
        torch.cuda.synchronize(dev)
        g_empty.replay()
        torch.cuda.synchronize(dev)
        empty_ms = timed(g_empty) / steps
    except Exception:  # noqa: BLE001 - the floor is context, not the measurement
        empty_ms = None
    t_load1 = time.time()
    while time.time() - t_load1 < args.clock_seconds / 2:
        graph.replay()
        torch.cuda.synchronize(dev)
    sampler.stop()
    clocks = sampler.summary(t_load0, time.time())
    for s in sets:
        st = vnm.vnm_get_status(s["A"])
        if st != vnm.VNM_OK:
            raise RuntimeError(f"kernel status {vnm.status_string(st)} during the timed region")

    max_ms = dist_max(elapsed_ms, world, dev)
    dense_flops = case.dense_flops()
    eff_flops = case.effective_flops()
    value = dense_flops * steps * world / (max_ms * 1e-3) / 1e12

    # roofline of the kernel that takes most of the step
    a_bytes = vb + mb + cb
    spmm_bytes = a_bytes + 2 * K * N + c_bytes
    comp_bytes = 2 * R * K + a_bytes
    if spmm_ms >= comp_ms:
        t_tc = eff_flops / (peaks["bf16_tflops"] * 1e12)
        t_hbm = spmm_bytes / (peaks["hbm_gbs"] * 1e9)
        if t_tc >= t_hbm:
            achieved = eff_flops / (spmm_ms * 1e-3) / 1e12
            roof = {"kernel": "vnm_spmm (tcgen05 sparse)" if plan.path == vnm.VNM_PATH_TC else "vnm_spmm (CUDA core)",
                    "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": achieved / peaks["bf16_tflops"],
                    "per_launch": f"{eff_flops:.4g} effective flops (2 per kept non-zero per column of B)"}
        else:
            achieved = spmm_bytes / (spmm_ms * 1e-3) / 1e9
            roof = {"kernel": "vnm_spmm", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "per_launch": f"{spmm_bytes} bytes (A values+meta+colidx, B, C once)"}
    else:
        achieved = comp_bytes / (comp_ms * 1e-3) / 1e9
        roof = {"kernel": "vnm_compress", "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "per_launch": f"{comp_bytes} bytes (dense W read, compressed arrays written)"}
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
    if empty_ms is not None:
        # for launches near the floor: the roofline time plus one empty
        # kernel's time, against the launch's own duration
        k_ms = spmm_ms if roof["kernel"].startswith("vnm_spmm") else comp_ms
        t_roof_ms = (eff_flops / (roof["peak"] * 1e12) if roof["unit"] == "TFLOP/s"
                     else (spmm_bytes if roof["kernel"].startswith("vnm_spmm") else comp_bytes) / (roof["peak"] * 1e9)) * 1e3
        roof["launch_floor"] = {"t_empty_us": empty_ms * 1e3, "t_roof_us": t_roof_ms * 1e3,
                                "frac_with_floor": (t_roof_ms + empty_ms) / k_ms}
    if roof["kernel"].startswith("vnm_spmm"):
        # vnm_spmm is one tensor-core launch, after the write-out of A as 2:4 when the plan says so
        parts = ["lift_expand_kernel", "spmm_tc_kernel"] if plan.lift == 2 else ["spmm_tc_kernel"]
        counts = [profiled_traffic(k, workload_tag(case)) for k in parts]
        roof["traffic"] = None if None in counts else sum(counts)
        roof["traffic_kernels"] = parts
    else:
        roof["traffic"] = profiled_traffic("compress", workload_tag(case))

    # end to end: host buffers, copies inside the timed region. Every step
    # copies its W and B in from pinned host memory and its C out; the steps
    # are pipelined over three streams (inputs in, compute, result out) and
    # the rotating device sets, so step i+1's inputs and step i-1's result
    # move while step i computes. Events order each step's copy -> compute ->
    # copy and keep a set from being overwritten before its last use is done.
    e2e = None
    if not args.no_e2e:
        W_pin = torch.from_numpy(W_h).pin_memory()
        B_pin = torch.from_numpy(B_h).pin_memory()
        C_pin = [torch.empty((R, N), dtype=c_dtype).pin_memory() for _ in range(2)]
        e_steps = max(3, min(steps, 50))
        n_in = max(1, args.e2e_in_streams)
        s_ins = [torch.cuda.Stream(dev) for _ in range(n_in)]
        s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        # W row chunks, one per input stream; B goes with the last one
        bounds = [R * q // n_in for q in range(n_in + 1)]

        def run_e2e(count):
            ev_cmp = [None] * count
            ev_out = [None] * count
            for i in range(count):
                st = sets[i % n_sets]
                prev = i - n_sets  # the step that used this set last
                for q, s_in in enumerate(s_ins):
                    if prev >= 0:
                        s_in.wait_event(ev_cmp[prev])  # its W and B are no longer read
                    with torch.cuda.stream(s_in):
                        if bounds[q + 1] > bounds[q]:
                            st["W"][bounds[q]:bounds[q + 1]].copy_(W_pin[bounds[q]:bounds[q + 1]], non_blocking=True)
                        if q == n_in - 1:
                            st["B"].copy_(B_pin, non_blocking=True)
                    ev_in = torch.cuda.Event()
                    ev_in.record(s_in)
                    s_cmp.wait_event(ev_in)
                if prev >= 0:
                    s_cmp.wait_event(ev_out[prev])  # its C has been copied out
                vnm.vnm_compress(st["A"], st["W"], stream=s_cmp)
                vnm.vnm_spmm(st["A"], st["B"], st["C"], workspace=st["ws"], stream=s_cmp)
                ev_cmp[i] = torch.cuda.Event()
                ev_cmp[i].record(s_cmp)
                s_out.wait_event(ev_cmp[i])
                with torch.cuda.stream(s_out):
                    C_pin[i % 2].copy_(st["C"], non_blocking=True)
                ev_out[i] = torch.cuda.Event()
                ev_out[i].record(s_out)
            return ev_out[count - 1]

        run_e2e(min(e_steps, 4))  # warm
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        dist_barrier(world, dev)
        torch.cuda.synchronize(dev)
        e0.record(s_cmp)
        for s_ in s_ins + [s_out]:
            s_.wait_event(e0)
        last = run_e2e(e_steps)
        s_out.wait_event(last)
        e1.record(s_out)
        torch.cuda.synchronize(dev)
        e_ms = dist_max(e0.elapsed_time(e1), world, dev)
        for s_ in sets:
            st_ = vnm.vnm_get_status(s_["A"])
            if st_ != vnm.VNM_OK:
                raise RuntimeError(f"kernel status {vnm.status_string(st_)} during the end-to-end leg")
        e2e = {"value": dense_flops * e_steps * world / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(W_h.nbytes + B_h.nbytes),
               "d2h_bytes_per_step": int(C_pin[0].numel() * C_pin[0].element_size()),
               "steps": e_steps, "ms_per_step": e_ms / e_steps,
               "pipelined": f"inputs in ({n_in} streams) / compute / result out, overlapped across steps"}

    # context: dense torch.matmul on the same shape (fp16 in, fp32 accumulate)
    ctx = {}
    try:
        if args.no_context:
            raise RuntimeError("skipped (--no-context)")
        Wd = sets[0]["W"]
        Bd = sets[0]["B"]
        for _ in range(3):
            torch.matmul(Wd, Bd)
        torch.cuda.synchronize(dev)
        m0 = torch.cuda.Event(enable_timing=True)
        m1 = torch.cuda.Event(enable_timing=True)
        m0.record()
        for _ in range(20):
            torch.matmul(Wd, Bd)
        m1.record()
        torch.cuda.synchronize(dev)
        ctx["torch_matmul_dense_tflops"] = dense_flops * 20 / (m0.elapsed_time(m1) * 1e-3) / 1e12
    except Exception as exc:  # context only
        ctx["torch_matmul_dense_tflops"] = f"unavailable: {exc}"

    per_config = None
    if not args.no_per_config:
        per_config = measure_per_config(dev, peaks, max(2, args.per_config_launches))
        per_config["gemm_compress"] = measure_gemm_compress(dev, peaks, max(2, args.per_config_launches))
        per_config["energy"] = measure_energy(dev)
        per_config["linear"] = measure_linear(dev, peaks, max(2, args.per_config_launches))
        per_config["bitmap"] = measure_bitmap(dev, peaks, max(2, args.per_config_launches))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        c = time_oracle(case, args.cpu_seconds)
        cpu = {k: c[k] for k in ("value", "unit", "cores", "kind", "sample", "row_parallel")}
        cpu["host_cpu"] = host_cpu()
        cpu["host_threads"] = os.cpu_count()

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": max_ms / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": config_of(case, f"{n_sets} rotating input/output sets of {set_bytes / 2**20:.1f} MiB "
                                      f"(> 2x the {l2 / 2**20:.0f} MiB L2)"),
            "effective_tflops": eff_flops * steps * world / (max_ms * 1e-3) / 1e12,
            "step_schedule": {"ms_per_step": max_ms / steps, "serial_ms_per_step": serial_ms,
                              "pipelined": "compress on one stream, SpMM on another: step i+1's compress overlaps "
                                           "step i's SpMM; serial_ms_per_step = the same steps on one stream"},
            "kernels": {"vnm_compress_ms": comp_ms, "vnm_spmm_ms": spmm_ms,
                        "spmm_dense_equiv_tflops": dense_flops / (spmm_ms * 1e-3) / 1e12,
                        "spmm_effective_tflops": eff_flops / (spmm_ms * 1e-3) / 1e12,
                        "compress_gbs": comp_bytes / (comp_ms * 1e-3) / 1e9,
                        "plan": plan.as_dict()},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks, "per_config": per_config,
            "gpu_launches": steps * kernels_per_step, "context": ctx,
            "gpu": props.name, "sm_count": props.multi_processor_count,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
