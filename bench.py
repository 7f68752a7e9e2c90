#!/usr/bin/env python
"""Throughput of the AWQ per-layer scale search on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl awq|reference]

One step is one full search (channel statistic, scales, residuals for the
20-point grid, tcgen05 error GEMM, losses, argmin, final quantize + pack) of
the workload's calls.  The default workload is the largest one that fits one
GPU, the 70B-class layer shapes: W 8192x8192 and 28672x8192 fp16, one X of
8192 tokens x 8192 fp16 with 0.5 % outlier channels, INT4 group 128, two
search calls per step.  Metric: weights searched per second (sum of N*K over
the searched weights / time).  Timing: CUDA events on the launching stream
around each step; between steps, outside the events, L2 is flushed by a
256 MiB write followed by a 256 MiB read of another buffer (so the step finds
none of its inputs in L2 and no dirty lines of the flush to write back); a
barrier and a device synchronisation on both sides of the timed region; the
maximum over ranks.  Under torchrun every rank searches its own replica of the
workload (independent layers: no collective on the data path, weak scaling).

``--impl reference`` times the CPU oracle (numpy, fp64) on the host cores on
a bounded row sample of the same workload, rank 0 only; the ``cpu_baseline``
leg of the default run times the same sample the same way.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "AWQ search: weights searched/s (20-α grid, T calib tokens); % of roofline"
UNIT = "weights/s"
N_GRID = 20
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed between timed steps, outside the step events: 256 MiB write, then a "
           "256 MiB read of another buffer")
DEFAULT_WORKLOAD = "llama70b"
# A timed region at least this long runs the tensor cores under the power
# cap: the roofline then takes the sustained peak instead of the burst one.
SUSTAINED_AFTER_MS = 1000.0
GEMM_SOURCES = [os.path.join(ROOT, "post_weight_quantization_33_b300", "csrc", f)
                for f in ("awq_gemm.cu", "awq_ptx.cuh")]


# --------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), tflops=float(p["bf16_tflops"]),
                    tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6400.0, tflops=1800.0, tflops_sustained=1400.0, source="fallback")


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for p in GEMM_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_summary(workload: str) -> str:
    return os.path.join(ROOT, "profiles", f"error_gemm_{workload}.md")


def profiled_traffic(workload: str):
    """DRAM bytes per error-GEMM launch from the committed ncu summary of this
    workload, if the kernel sources are unchanged since the capture; else None."""
    path = profile_summary(workload)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.strip().lstrip("-").strip()
            if line.startswith(("traffic_bytes_per_launch", "kernel_source_sha256")):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != gemm_source_hash():
        return None
    try:
        return int(float(vals["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, interval_ms: int = 50):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", gpu_id, "-lms", str(interval_ms)],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.file.read())) if len(r) >= 9]
        self.file.close()
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(wl) -> int:
    """Bytes the method itself must move: statistic over X, quantize (read W,
    write codes + fp16 scale + u8 zero per group) and the error GEMM's operand
    reads (codes-sized weights and X), per grid point."""
    total = 0
    for call in wl.calls:
        x = wl.spec(call.x)
        total += 2 * x.rows * x.cols
        for w in call.ws:
            s = wl.spec(w)
            nk = s.rows * s.cols
            per_grid = (2 * nk + nk * call.bits // 8 + 3 * nk // call.group) + \
                       (nk * call.bits // 8 + 3 * nk // call.group + 2 * x.rows * x.cols)
            total += N_GRID * per_grid
    return total


def config_for(name: str) -> dict:
    wl = workloads.WORKLOADS[name]
    calls = []
    for c in wl.calls:
        x = wl.spec(c.x)
        calls.append({"X": [x.rows, x.cols],
                      "W": [[wl.spec(w).rows, wl.spec(w).cols] for w in c.ws],
                      "bits": c.bits, "group": c.group})
    return {"workload": f"{name}: {wl.description}", "calls": calls, "grid_points": N_GRID,
            "l2": L2_NOTE}


# --------------------------------------------------------------------------- oracle timing
def oracle_pool(data):
    """A spawn-started pool of oracle workers with the workload's tensors in
    shared memory, filling every host core: a quarter as many workers as
    cores, each with a BLAS pool of 4 threads.  (Every worker repeats a call's
    work on the whole X -- the inverse-scaled activations of each grid point
    -- so fewer, wider workers move less memory per sampled row.)"""
    from oracle.row_pool import OraclePool, default_workers
    cores = default_workers()
    workers = max(1, cores // 4)
    return OraclePool(data, workers, blas_threads=cores // workers)


def oracle_step(pool, wl, rows_per_weight: int) -> int:
    """One oracle search of every call of the workload on the first
    ``rows_per_weight`` output rows of every weight (all tokens, all grid
    points); the rows of all calls are cut into one batch of blocks over the
    pool's workers.  Returns the weights searched."""
    done, calls = 0, []
    for call in wl.calls:
        rows = [np.arange(min(rows_per_weight, wl.spec(w).rows)) for w in call.ws]
        calls.append(dict(x=call.x, ws=call.ws, bits=call.bits, group=call.group, n_grid=N_GRID,
                          rows=rows))
        done += sum(len(r) * wl.spec(w).cols for r, w in zip(rows, call.ws))
    pool.search_calls(calls)
    return done


def oracle_sample(rows: int, pool) -> str:
    return (f"first {rows} output rows of every weight, all tokens, all {N_GRID} grid points, "
            f"per step; oracle.awq_oracle.search on row blocks in {pool.workers} spawned worker "
            f"processes (numpy fp64, {pool.blas_threads} BLAS threads each)")


def cpu_baseline(data, wl, rows: int, steps: int = 2) -> dict:
    """The oracle as it stands, timed the way --impl reference times it: the
    same row sample, the same pool, one untimed step then ``steps`` timed."""
    with oracle_pool(data) as pool:
        oracle_step(pool, wl, rows)
        t0 = time.perf_counter()
        n = 0
        for _ in range(steps):
            n += oracle_step(pool, wl, rows)
        dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": pool.cores, "kind": "oracle",
            "sample": oracle_sample(rows, pool) + f"; {steps} timed steps, {dt:.1f} s"}


def settle_clocks(gpu_id: str, max_s: float = 5.0) -> dict:
    """Wait (at most max_s) until the SM clock is back within 5 % of its
    maximum with no power-cap throttling: the power governor lags a heavy
    phase by a second or more, and the HBM-bound calls timed next are partly
    issue-bound, so they would be timed at the previous phase's capped clock
    (measured: the statistic 46 us instead of 28 right after the 70B-class
    searches, 28.0 again after a 3 s pause).  Returns the wait and the clock
    it ended at; without nvidia-smi, waits max_s / 2."""
    q = "clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap"
    t0 = time.perf_counter()
    last = None
    while True:
        try:
            out = subprocess.run(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                  "-i", gpu_id], capture_output=True, text=True, timeout=10)
            sm, smax, cap = [v.strip() for v in out.stdout.strip().split(",")[:3]]
            last = {"sm_mhz": float(sm), "sm_max_mhz": float(smax), "sw_power_cap": cap}
        except (OSError, ValueError, subprocess.SubprocessError):
            time.sleep(max_s / 2)
            return {"waited_s": round(time.perf_counter() - t0, 2), "clocks": "nvidia-smi unavailable"}
        ok = last["sm_mhz"] >= 0.95 * last["sm_max_mhz"] and last["sw_power_cap"] != "Active"
        waited = time.perf_counter() - t0
        if ok or waited >= max_s:
            return {"waited_s": round(waited, 2), "settled": ok, **last}
        time.sleep(0.2)


def hbm_kernels(dev, flush, hbm_gbs: float, reps: int = 5) -> dict:
    """Achieved HBM bandwidth of the HBM-bound entry points at the largest
    workload's sizes (X 8192x8192; W 28672x8192), called through the C ABI
    with preallocated buffers.  Each figure times calls back to back over
    several copies of the input, each larger than L2, so no call finds its
    input in L2; the calls are queued behind a device-side wait, so host
    launch gaps are hidden; per call = elapsed / calls.
    Bytes are the algorithmic ones: 2TK for the statistic; 2NK read + b/8 NK
    codes + 3NK/128 scales and zeros written for quantize + pack; codes,
    scales, zeros, x read and y written for the decode product."""
    import ctypes
    import torch
    import post_weight_quantization_33_b300 as awq
    L = awq.lib()
    stream = torch.cuda.current_stream()
    st = stream.cuda_stream
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    out = {}

    def timed(fns):
        for fn in fns:                         # warm-up pass
            fn()
        flush(0)
        # A device-side wait (about 2 ms) while the host queues every timed
        # call: the calls then run back to back on the GPU, so the figure is
        # their device time, not the host's launch rate (a call's host work,
        # about 20 us for the statistic, can exceed its device time).
        torch.cuda._sleep(4_000_000)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            for fn in fns:
                fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / (reps * len(fns))

    T, K = 8192, 8192
    Xs = [torch.randn(T, K, generator=g, device=dev).half() for _ in range(6)]
    sX = torch.empty(K, dtype=torch.float64, device=dev)
    ms = timed([lambda X=X: awq._check(L.awq_stats(X.data_ptr(), T, K, sX.data_ptr(), st))
                for X in Xs])
    nbytes = 2 * T * K
    out["stats"] = {"shape": f"X {T}x{K} fp16", "ms": ms, "bytes": nbytes,
                    "gbs": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / hbm_gbs,
                    "calls": f"{len(Xs)} inputs x {reps}"}
    # Context, not a denominator: a library reduction (torch.amax) reading the
    # same bytes the same way.
    ms = timed([lambda X=X: torch.amax(X) for X in Xs])
    out["read_only_context"] = {"X": {"bytes": nbytes, "ms": ms, "gbs": nbytes / ms / 1e6,
                                      "kernel": "torch.amax"}}
    del Xs
    N, K = 28672, 8192
    Ws = [(torch.randn(N, K, generator=g, device=dev) * 0.015).half() for _ in range(3)]
    W = Ws[0]
    s = torch.rand(K, generator=g, device=dev) + 0.5
    codes = [torch.empty(N * K // 8, dtype=torch.int32, device=dev) for _ in Ws]
    sc = [torch.empty(N * K // 128, dtype=torch.float16, device=dev) for _ in Ws]
    z = [torch.empty(N * K // 128, dtype=torch.uint8, device=dev) for _ in Ws]
    cfg = awq.QConfig(4, 128, 1, N_GRID)
    ms = timed([lambda i=i: awq._check(L.awq_quantize_pack(
        Ws[i].data_ptr(), N, K, s.data_ptr(), ctypes.byref(cfg), codes[i].data_ptr(),
        sc[i].data_ptr(), z[i].data_ptr(), st)) for i in range(len(Ws))])
    nbytes = 2 * N * K + N * K // 2 + 3 * N * K // 128
    out["quantize_pack"] = {"shape": f"W {N}x{K} fp16 -> INT4 g128", "ms": ms, "bytes": nbytes,
                            "gbs": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / hbm_gbs,
                            "calls": f"{len(Ws)} inputs x {reps}"}
    ms = timed([lambda W=W: torch.amax(W) for W in Ws])
    out["read_only_context"]["W"] = {"bytes": 2 * N * K, "ms": ms, "gbs": 2 * N * K / ms / 1e6,
                                     "kernel": "torch.amax"}
    # The packed layer consumed at decode: the W4A16 product for 1, 16 and 8
    # tokens and the W3A16 product for one token, each beside a cuBLAS fp16
    # product with the dense weight of the same shape (8 tokens last, so the
    # launch indices of the others stay as profiled).
    cfg3 = awq.QConfig(3, 128, 1, N_GRID)
    codes3 = [torch.empty(N * 3 * K // 32, dtype=torch.int32, device=dev) for _ in Ws]
    sc3 = [torch.empty(N * K // 128, dtype=torch.float16, device=dev) for _ in Ws]
    z3 = [torch.empty(N * K // 128, dtype=torch.uint8, device=dev) for _ in Ws]
    for i in range(len(Ws)):
        awq._check(L.awq_quantize_pack(Ws[i].data_ptr(), N, K, s.data_ptr(), ctypes.byref(cfg3),
                                       codes3[i].data_ptr(), sc3[i].data_ptr(), z3[i].data_ptr(),
                                       st))
    decode = {}
    for bits, M in ((4, 1), (4, 16), (3, 1), (4, 8)):
        c_, s_, z_, cf = (codes, sc, z, cfg) if bits == 4 else (codes3, sc3, z3, cfg3)
        x = torch.randn(M, K, generator=g, device=dev).half()
        y = torch.empty(M, N, dtype=torch.float32, device=dev)
        ms = timed([lambda i=i: awq._check(L.awq_w4a16_matvec(
            c_[i].data_ptr(), s_[i].data_ptr(), z_[i].data_ptr(), N, K, ctypes.byref(cf),
            x.data_ptr(), M, y.data_ptr(), st)) for i in range(len(Ws))])
        nbytes = N * K * bits // 8 + 3 * N * K // 128 + 2 * M * K + 4 * M * N
        dense_ms = timed([lambda W=W: torch.matmul(x, W.t()) for W in Ws])
        decode[f"int{bits}_m{M}"] = {
            "shape": f"W {N}x{K} INT{bits} g128, {M} token(s)", "ms": ms, "bytes": nbytes,
            "gbs": nbytes / ms / 1e6, "frac": nbytes / ms / 1e6 / hbm_gbs,
            "fp16_cublas_ms": dense_ms, "speedup_vs_fp16": dense_ms / ms}
    out["decode_product"] = decode
    del Ws, W
    return out


def dequant_mainloop_bound(calls, flush, stages_ms: dict, step_ms: float) -> dict:
    """Measured lower bound on the step time of the design that dequantizes
    packed codes inside the error GEMM's main loop and subtracts a prologue
    reference output Y = W X^T in its epilogue (instead of this library's
    fp16 residual pass).  That design cannot avoid (a) the prologue GEMM
    Y = W X^T and (b) a quantize + pack pass per grid point writing the codes
    its main loop reads; its MMA work equals this GEMM's.  Both are timed
    here on this step's weights (this library's own tcgen05 reference GEMM
    and quantize + pack kernels); the bound assumes the dequantization costs
    the main loop nothing and the epilogue's reads of Y (4 N T bytes per grid
    point) are free:  bound = step - residual pass + (a) + (b)."""
    import ctypes
    import torch
    import post_weight_quantization_33_b300 as awq
    L = awq.lib()
    stream = torch.cuda.current_stream()
    st = stream.cuda_stream
    yref_ms = quant_ms = 0.0
    for X, Ws, bits, group in calls:
        T, K = X.shape
        r = awq.search(X, Ws, bits, group, N_GRID)
        r.check()
        s_grid = r.s_grid()
        r.free()
        cfg = awq.QConfig(bits, group, 1, N_GRID)
        for W in Ws:
            N = W.shape[0]
            Y = torch.empty(N, T, dtype=torch.float32, device=X.device)
            status = torch.zeros(1, dtype=torch.int32, device=X.device)
            words = awq.packed_words(N, K, bits)
            gpr = awq.groups_per_row(K, group)
            outs = [(torch.empty(words, dtype=torch.int32, device=X.device),
                     torch.empty(N * gpr, dtype=torch.float16, device=X.device),
                     torch.empty(N * gpr, dtype=torch.uint8, device=X.device))
                    for _ in range(N_GRID)]

            def yref():
                awq._check(L.awq_reference_output(W.data_ptr(), N, X.data_ptr(), T, K,
                                                  Y.data_ptr(), status.data_ptr(), st))

            def quant_all():
                for a in range(N_GRID):
                    c, sc, z = outs[a]
                    awq._check(L.awq_quantize_pack(W.data_ptr(), N, K, s_grid[a].data_ptr(),
                                                   ctypes.byref(cfg), c.data_ptr(), sc.data_ptr(),
                                                   z.data_ptr(), st))

            for fn, which in ((yref, "y"), (quant_all, "q")):
                fn()
                flush(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                e1.synchronize()
                if which == "y":
                    yref_ms += e0.elapsed_time(e1)
                else:
                    quant_ms += e0.elapsed_time(e1)
            assert int(status.item()) == 0
            del Y, outs
    residual = stages_ms["residual"]
    return {"reference_gemm_ms": yref_ms, "quantize_all_grid_points_ms": quant_ms,
            "residual_pass_ms": residual, "step_ms": step_ms,
            "bound_ms": step_ms - residual + yref_ms + quant_ms,
            "note": "lower bound for dequant-in-mainloop + prologue reference GEMM: this step "
                    "minus its residual pass plus (a) Y = W X^T and (b) quantize + pack at every "
                    "grid point, both measured here"}


class L2Flush:
    """Between timed launches: write a buffer larger than L2, then read
    another one, so L2 holds neither the timed kernel's inputs nor dirty
    lines that the kernel would have to write back."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, i: int) -> None:
        import torch
        self.w.fill_(i)
        torch.sum(self.r, dim=0, out=self.sink)


# --------------------------------------------------------------------------- ranks
def max_over_ranks(ms: float, world: int, device) -> float:
    """The largest of the ranks' timed milliseconds: an all-reduce (MAX) over
    the process group when world > 1 (a CUDA tensor for nccl, a CPU one for
    gloo), else ms itself."""
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, steps: int, world: int, max_ms: float) -> float:
    """Units all ranks processed per second: every rank runs the same steps
    on its own replica (weak scaling), timed by the slowest rank."""
    return units_per_rank_step * steps * world / (max_ms / 1e3)


# --------------------------------------------------------------------------- arms
def run_reference(args, rank: int, world: int) -> None:
    if rank != 0:
        return
    wl = workloads.WORKLOADS[args.workload]
    data = workloads.generate(args.workload)
    rows = args.reference_rows
    with oracle_pool(data) as pool:
        for _ in range(args.warmup):
            oracle_step(pool, wl, rows)
        times, n = [], 0
        for _ in range(args.steps):
            t0 = time.perf_counter()
            n = oracle_step(pool, wl, rows)
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = n * args.steps / total
    sample = oracle_sample(rows, pool) + f" ({n} weights per step)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_for(args.workload),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_awq(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    import torch.distributed as dist

    import post_weight_quantization_33_b300 as awq

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    awq.lib()
    wl = workloads.WORKLOADS[args.workload]
    data = workloads.generate(args.workload)
    calls = []
    for c in wl.calls:
        calls.append((torch.from_numpy(data[c.x]).to(dev),
                      [torch.from_numpy(data[w]).to(dev) for w in c.ws], c.bits, c.group))
    weights_per_step = wl.weights_searched()
    flush = L2Flush(dev)

    def step():
        res = [awq.search(X, Ws, bits, group, N_GRID) for X, Ws, bits, group in calls]
        return res

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    awq.set_stage_timing(True)
    for _ in range(args.warmup):
        for r in step():
            r.check()
            r.free()
    stream = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    kept = []
    barrier()
    props = torch.cuda.get_device_properties(dev)
    bus = getattr(props, "pci_bus_id", None)
    gpu_id = (f"{getattr(props, 'pci_domain_id', 0):08X}:{bus:02X}:"
              f"{getattr(props, 'pci_device_id', 0):02X}.0") if bus is not None else str(local_rank)
    clocks = ClockSampler(gpu_id)
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush(i)
        starts[i].record(stream)
        kept.append(step())
        ends[i].record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    launches = 0
    gemm_ms = []
    stage_sum = {name: 0.0 for name in awq.STAGES}
    for res in kept:
        for r in res:
            r.check()
            launches += r.kernel_launches
            st = r.stage_ms()
            gemm_ms.append(st["error_gemm"])
            for name in stage_sum:
                stage_sum[name] += st[name]
            r.free()
    awq.set_stage_timing(False)
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = whole_job_rate(weights_per_step, args.steps, world, total_ms)

    # End to end through the public API with host (pinned) buffers.
    host_calls = [(torch.from_numpy(data[c.x]).pin_memory(),
                   [torch.from_numpy(data[w]).pin_memory() for w in c.ws], c.bits, c.group)
                  for c in wl.calls]
    h2d = sum(X.numel() * 2 + sum(W.numel() * 2 for W in Ws) for X, Ws, _, _ in host_calls)
    d2h = 0
    for X, Ws, bits, group in host_calls:
        for W in Ws:
            n, k = W.shape
            d2h += awq.packed_words(n, k, bits) * 4 + 3 * n * (k // group)
        d2h += X.shape[1] * 4 + N_GRID * 8
    # Steps run through awq_search_host_layers (the C ABI's host-buffer
    # pipeline, via search_host_stream): step i+1's inputs are copied in and
    # step i-1's results copied out while step i is searched.  Every step
    # still copies its own inputs in and its results out inside the timed
    # region; the region spans all steps, pipeline fill and drain included.
    e2e_steps = max(3, min(args.steps, 20))
    by_cfg = {}
    for X, Ws, bits, group in host_calls:
        by_cfg.setdefault((bits, group), []).append((X, Ws))

    def e2e_pass(n_steps):
        for (bits, group), calls in by_cfg.items():
            awq.search_host_stream(calls * n_steps, bits, group, N_GRID, device=dev)

    # Warm-up with as many steps as are timed: the pinned host buffers the
    # results land in come from torch's caching host allocator, so the timed
    # pass does not pay for page-locking fresh memory.
    e2e_pass(e2e_steps)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    flush(0)
    e0.record(stream)
    e2e_pass(e2e_steps)
    e1.record(stream)
    e1.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = whole_job_rate(weights_per_step, e2e_steps, world, e2e_ms)

    if rank != 0:
        return
    pk = peaks()
    # One error-GEMM launch per call; with several calls this is their average.
    flops_per_launch = wl.gemm_flops(N_GRID) / len(wl.calls)
    gemm_avg_ms = statistics.mean(gemm_ms)
    achieved = flops_per_launch / (gemm_avg_ms / 1e3) / 1e12
    ideal_s = max(wl.gemm_flops(N_GRID) / (pk["tflops"] * 1e12),
                  algorithmic_bytes(wl) / (pk["hbm_gbs"] * 1e9))
    # The GEMM runs inside the step: the burst peak for a short timed region,
    # the sustained (power-capped) peak for one that lasts a second or more.
    long_run = total_ms >= SUSTAINED_AFTER_MS
    gemm_peak = pk["tflops_sustained"] if long_run else pk["tflops"]
    peak_kind = "sustained" if long_run else "burst"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic", "config": config_for(args.workload),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": gemm_peak,
                     "unit": "TFLOP/s", "frac": achieved / gemm_peak,
                     "traffic": profiled_traffic(args.workload),
                     "kernel": "k_gemm_err_pair (tcgen05 cta_group::2 error GEMM), fp16 operands, f32 accumulate",
                     "peak_source": f"{pk['source']} bf16 {peak_kind} (dense fp16 taken equal)",
                     "launch_ms": gemm_avg_ms},
        "step_roofline": {"ideal_ms": ideal_s * 1e3, "frac": ideal_s * 1e3 / (total_ms / args.steps)},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "api": "awq_search_host_layers"},
        "gpu_launches": launches,
        "stages_ms_per_step": {k: v / args.steps for k, v in stage_sum.items()},
        "clocks": clk,
        "wall_s": t_wall,
    }
    # Workloads with more calibration tokens than channels: the same search
    # with the loss in its Gram form, reported as a separate variant (its
    # flops are not the metric's; the roofline above stays the direct form's).
    if any(wl.spec(c.x).rows > wl.spec(c.x).cols for c in wl.calls):
        gsteps = max(3, min(args.steps, 10))
        for _ in range(2):
            for X, Ws, bits, group in calls:
                awq.search(X, Ws, bits, group, N_GRID, gram=True).free()
        barrier()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        gms = 0.0
        for i in range(gsteps):
            flush(i)
            g0.record(stream)
            res = [awq.search(X, Ws, bits, group, N_GRID, gram=True) for X, Ws, bits, group in calls]
            g1.record(stream)
            g1.synchronize()
            gms += g0.elapsed_time(g1)
            for r in res:
                r.check()
                r.free()
        line["gram_variant"] = {
            "value": weights_per_step * gsteps / (gms / 1e3), "unit": UNIT,
            "ms_per_step": gms / gsteps, "speedup_vs_direct": (total_ms / args.steps) / (gms / gsteps),
            "note": "awq_search_layer_gram: loss as d^T (X^T X) d; same outputs within 1e-3"}
    # The residual pass: W read once, n_grid fp16 residuals written.
    res_ms = stage_sum["residual"] / args.steps
    res_bytes = sum(2 * wl.spec(w).rows * wl.spec(w).cols * (1 + N_GRID)
                    for c in wl.calls for w in c.ws)
    line["dequant_mainloop_bound"] = dequant_mainloop_bound(
        calls, flush, {k: v / args.steps for k, v in stage_sum.items()}, total_ms / args.steps)
    settle = settle_clocks(gpu_id)
    line["hbm_kernels"] = hbm_kernels(dev, flush, pk["hbm_gbs"])
    line["hbm_kernels"]["clock_settle"] = settle
    line["hbm_kernels"]["residual"] = {
        "shape": "this workload, every grid point", "ms": res_ms, "bytes": res_bytes,
        "gbs": res_bytes / res_ms / 1e6, "frac": res_bytes / res_ms / 1e6 / pk["hbm_gbs"]}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(data, wl, args.reference_rows)
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["awq", "reference"], default="awq")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOAD_ORDER))
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (used for profiler runs)")
    ap.add_argument("--reference-rows", type=int, default=256,
                    help="output rows per weight in each oracle step (--impl reference and "
                         "the cpu_baseline leg)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_awq(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
