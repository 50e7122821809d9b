#!/usr/bin/env python3
"""Benchmark of the batch-invariant GEMM on GB300.

Workload (one step): the LLM-projection sweep y = x·W, bf16 x[M,4096] · W[4096,14336], fp32
accumulation, bf16 out, for M in {1,7,8,15,16,17,63,64,65,128,129,192,193,256,512,1024,2048,
4096,8192} — one GEMM launch per M, through the C ABI (bi_gemm_run).  Metric: TFLOP/s and
fraction of roofline versus M; value = FLOPs of all launches / time.

Cold L2: three copies of (W, x) (552 MB, > 4x the 126 MB L2) rotate from launch to launch, so
every launch streams its operands from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain C, fp64, single thread) on a bounded sample of the
same workload, in the same metric.  One JSON line is printed by rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

K_DIM, N_DIM = 4096, 14336
M_SWEEP = [1, 7, 8, 15, 16, 17, 63, 64, 65, 128, 129, 192, 193, 256, 512, 1024, 2048, 4096, 8192]
N_SETS = 3
METRIC = "TFLOP/s & % roofline vs M (1-8192), 0 byte-diff batch invariance, 1 GB300"
WORKLOAD = "LLM projection sweep: bf16 x[M,4096]·W[4096,14336], fp32 accumulate, bf16 out, M in 1..8192 (19 values)"
KERNEL_SOURCES = ["invariant_bi_gemm_gb300/csrc/bi_gemm_kernel.cuh", "invariant_bi_gemm_gb300/csrc/ptx.cuh",
                  "invariant_bi_gemm_gb300/csrc/bi_gemm.cu"]
# The GEMM handle of the sweep is created with BI_GEMM_FLAG_STATIC_W: W is never written while
# the sweep runs, so each launch may start loading W before the previous launch has finished.
STATIC_W = True
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of each launch of the sweep, from one
# ncu capture of `python bench.py --steps 1 --warmup 3 --no-paths --no-cpu` (the command and the
# figures are in profiles/ncu_bf16_gemm_llm_sweep.md), for the kernel sources of the given hash.
TRAFFIC = {"source_sha256_16": "2f8d761ab6d68369", "bytes_per_launch": {
    1: 120521216, 7: 117620992, 8: 117682688, 15: 117749248,
    16: 117761792, 17: 117951744, 63: 118087168, 64: 118089728,
    65: 118169856, 128: 118985984, 129: 118648064, 192: 119137536,
    193: 119150592, 256: 119681536, 512: 123747072, 1024: 141447680,
    2048: 174518016, 4096: 278937344, 8192: 739951616}}


def flops(M, K=K_DIM, N=N_DIM):
    return 2.0 * M * K * N


def algo_bytes(M, K=K_DIM, N=N_DIM, out_bytes=2, in_bytes=2, scale_bytes=0.0):
    return in_bytes * (M * K + K * N) + out_bytes * M * N + scale_bytes * (M * K + K * N)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_hash():
    """Hash of the kernel sources' code: comments and whitespace are dropped, so that editing a
    comment does not invalidate a recorded profile."""
    import re
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        src = open(os.path.join(ROOT, f)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(M):
    """DRAM bytes (read + written) of the sweep's launch at M from the ncu capture recorded in
    TRAFFIC, or None when the kernel sources changed since that capture."""
    if TRAFFIC.get("source_sha256_16") != kernel_hash():
        return None
    return TRAFFIC["bytes_per_launch"].get(M)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, mx, reasons, pw = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [t.strip() for t in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        busy = [s for s, p in zip(sm, pw) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed

_BACKEND = None


def dist_init():
    """Join the process group when launched with WORLD_SIZE > 1 (one rank per GPU, NCCL; gloo
    without GPUs or when BI_DIST_BACKEND says so).  Returns (rank, world, local rank)."""
    global _BACKEND
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        _BACKEND = os.environ.get("BI_DIST_BACKEND") or ("nccl" if _cuda() else "gloo")
        dist.init_process_group(_BACKEND)
    return rank, world, local


def _cuda():
    import torch
    return torch.cuda.is_available()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if _BACKEND == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle baseline

def oracle_sample(budget_s: float, threads: int = 1):
    """Time the CPU oracle on rows of the sweep's x against the full W for about `budget_s`
    seconds of wall time.  With threads > 1 the rows are spread over that many threads, each
    calling the unchanged single-threaded oracle on one row at a time (the C call releases the
    interpreter lock; rows are independent, so the results are those of one thread).

    Returns (flops_done, seconds, description)."""
    import threading
    from concurrent.futures import ThreadPoolExecutor

    import inputgen as ig
    import oracle
    oracle.lib()
    W = ig.normal_bf16(ig.SEED_W, K_DIM, N_DIM, std=0.02)
    rows = min(8192, 16 * threads)
    x = ig.normal_bf16(ig.SEED_X, rows, K_DIM)
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t0 = time.perf_counter()

    def worker():
        while time.perf_counter() - t0 < budget_s:
            with lock:
                r = state["next"]
                if r >= rows:
                    return
                state["next"] = r + 1
            oracle.gemm_bf16(x[r:r + 1], W, "bf16")
            with lock:
                state["done"] += 1

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for f in [ex.submit(worker) for _ in range(threads)]:
            f.result()
    dt = time.perf_counter() - t0
    done = state["done"]
    desc = (f"{done} rows of x[8192,4096] times the full W[4096,14336] (all 14336 outputs per row), "
            f"plain C oracle, fp64, {threads} thread{'s' if threads > 1 else ''} (one row per call)")
    return flops(done), dt, desc


def roof_time(M, peaks, K=K_DIM, N=N_DIM):
    """Seconds of one launch at its roofline: max(FLOP / tensor peak, algorithmic bytes / HBM)."""
    return max(flops(M, K, N) / (peaks["bf16_tflops"] * 1e12), algo_bytes(M, K, N) / (peaks["hbm_gbs"] * 1e9))


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle as it stands, on all host cores (one thread per core,
    each running the single-threaded oracle on its own row), on a bounded sample of the same
    workload per step."""
    if rank != 0:
        return
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import inputgen as ig
    import oracle
    oracle.lib()
    cores = os.cpu_count() or 1
    W = ig.normal_bf16(ig.SEED_W, K_DIM, N_DIM, std=0.02)
    x = ig.normal_bf16(ig.SEED_X, cores, K_DIM)
    # calibrate one full row, then size each step's sample so the whole run stays near 2 minutes
    t0 = time.perf_counter()
    oracle.gemm_bf16(x[:1], W, "bf16")
    t_row = time.perf_counter() - t0
    per_step = 120.0 / max(1, args.steps + args.warmup)
    cols = int(max(64, min(N_DIM, N_DIM * per_step / max(t_row, 1e-6))) // 64 * 64)
    Wc = np.ascontiguousarray(W[:, :cols])

    with ThreadPoolExecutor(max_workers=cores) as ex:
        def step():
            for f in [ex.submit(oracle.gemm_bf16, x[r:r + 1], Wc, "bf16") for r in range(cores)]:
                f.result()

        for _ in range(args.warmup):
            step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step()
        dt = time.perf_counter() - t0
    fl = flops(cores, K_DIM, cols) * args.steps
    v = fl / dt / 1e12
    sample = (f"per step: {cores} rows of x (one per thread) times W[:, :{cols}] of the LLM projection (K=4096), "
              f"plain C oracle, fp64, {cores} threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_obj(world),
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_obj(world):
    return {"workload": WORKLOAD, "M": M_SWEEP, "K": K_DIM, "N": N_DIM, "in": "bf16", "out": "bf16",
            "accumulate": "fp32", "l2": f"{N_SETS} rotating (W, x) sets, 552 MB > L2: every launch reads cold",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ------------------------------------------------------------------ our path

def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import inputgen as ig
    from invariant_bi_gemm_gb300 import BiGemm

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    def to_dev(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    W_np = ig.normal_bf16(ig.SEED_W, K_DIM, N_DIM, std=0.02)
    X_np = ig.normal_bf16(ig.SEED_X, M_SWEEP[-1], K_DIM)
    W0, X0 = to_dev(W_np), to_dev(X_np)
    Ws = [W0] + [W0.clone() for _ in range(N_SETS - 1)]
    Xs = [X0] + [X0.clone() for _ in range(N_SETS - 1)]
    Y = torch.empty((M_SWEEP[-1], N_DIM), dtype=torch.bfloat16, device=dev)
    g = BiGemm(K_DIM, N_DIM, "bf16", static_w=STATIC_W)
    stream = torch.cuda.current_stream(dev)
    nM = len(M_SWEEP)

    def launch_step(s):
        for i, M in enumerate(M_SWEEP):
            c = (s * nM + i) % N_SETS
            g(Xs[c][:M], Ws[c], Y[:M])

    # eager warm-up through the public call, then one CUDA graph per rotation offset so that
    # step s replays graph s % 3 and every launch still reads the next (cold) copy of W and x
    for s in range(args.warmup):
        launch_step(s)
    torch.cuda.synchronize()
    assert g.device_error() == 0
    graphs = []
    for r in range(N_SETS):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            launch_step(r)
        graphs.append(gr)
    for s in range(args.warmup):
        graphs[s % N_SETS].replay()
    torch.cuda.synchronize()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for s in range(args.steps):
        graphs[s % N_SETS].replay()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    assert g.device_error() == 0
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    step_flops = sum(flops(M) for M in M_SWEEP)
    value = step_flops * args.steps * world / (elapsed_ms / 1e3) / 1e12

    # per-M launch duration: a graph of REPS launches of one M, timed with events; cold = rotating
    # copies (every launch reads W and x from HBM), warm = one copy (W and x stay in L2 when they fit)
    REPS = 30

    def time_m(M, nsets):
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm):
            for j in range(REPS):
                g(Xs[j % nsets][:M], Ws[j % nsets], Y[:M])
        gm.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            gm.replay()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / REPS)
        del gm
        return statistics.median(ts)

    per_m, per_m_warm = {}, {}
    for M in M_SWEEP:          # cold and warm of one M back to back, so both see the same clocks
        per_m[M] = time_m(M, N_SETS)
        per_m_warm[M] = time_m(M, 1)
    kernel_ms_total = sum(per_m.values())

    # the same sweep through eager per-call launches (Python + ctypes on every call)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_eager = max(3, min(args.steps, 50))
    torch.cuda.synchronize()
    e0.record(stream)
    for s in range(n_eager):
        launch_step(s)
    e1.record(stream)
    torch.cuda.synchronize()
    eager_ms = e0.elapsed_time(e1) / n_eager

    cublas = measure_cublas_context(Xs, Ws, g, stream)
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    sweep = []
    for M in M_SWEEP:
        t = per_m[M] / 1e3
        fl, by = flops(M), algo_bytes(M)
        t_roof = roof_time(M, peaks)
        tw = per_m_warm[M] / 1e3
        row = {"M": M, "us": round(t * 1e6, 2), "tflops": round(fl / t / 1e12, 2),
               "gbs": round(by / t / 1e9, 1), "bound": "hbm" if fl / by < ridge else "tensor",
               "frac": round(t_roof / t, 3), "us_warm_l2": round(tw * 1e6, 2),
               "tflops_warm_l2": round(fl / tw / 1e12, 2), "algorithmic_bytes": int(by)}
        tr = recorded_traffic(M)
        row["dram_bytes"] = tr
        row["dram_over_algorithmic"] = round(tr / by, 3) if tr else None
        row.update(cublas.get(M, {}))
        sweep.append(row)

    # Roofline of the timed region (the whole sweep): the step's time at the roofline is the sum,
    # over its launches, of max(FLOP / tensor peak, bytes / HBM bandwidth); `peak` is the FLOP rate
    # of a step that ran every launch at its roofline, so frac = achieved / peak = that sum / the
    # measured step time.
    t_step = elapsed_ms / args.steps / 1e3
    t_roof_step = sum(roof_time(M, peaks) for M in M_SWEEP)
    achieved = step_flops / t_step / 1e12
    peak_step = step_flops / t_roof_step / 1e12
    traffic = [recorded_traffic(M) for M in M_SWEEP]
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak_step, 1), "unit": "TFLOP/s",
                "frac": round(achieved / peak_step, 4),
                "traffic": int(sum(traffic)) if all(traffic) else None,
                "algorithmic_bytes": int(sum(algo_bytes(M) for M in M_SWEEP)),
                "per": "one step (19 launches of the sweep); traffic is DRAM read + write bytes of those launches "
                       "from one ncu capture (null when the kernel changed since)",
                "peak_definition": "sum over the step's launches of max(2MKN / tensor peak, bytes / HBM bandwidth); "
                                   "frac = that time / ms_per_step",
                "peak_tensor_tflops": peaks["bf16_tflops"], "peak_hbm_gbs": peaks["hbm_gbs"],
                "peak_source": peaks["source"] + " (MEASURED_PEAKS.json: bf16 burst, copy bandwidth)",
                "frac_of_tensor_peak": round(achieved / peaks["bf16_tflops"], 4),
                "kernel": "bi_gemm_kernel<bf16, out bf16, {}x{} tile on {} CTA(s), {} stages>".format(
                    g.config["block_m"], g.config["block_n"], g.config["ctas_per_tile"], g.config["stages"]),
                "launch_timing": f"per M: CUDA events around graphs of {REPS} launches, rotating cold copies "
                                 "(us); the same with one copy, warm L2 where it fits (us_warm_l2)",
                "hbm_regime_frac_M_le_64": min((r["frac"] for r in sweep if r["M"] <= 64), default=None),
                "tensor_regime_frac_M_ge_2048": min((r["frac"] for r in sweep if r["M"] >= 2048), default=None)}

    e2e = measure_e2e(g, W_np, X_np, args, dev, world)
    paths = measure_other_paths(dev, peaks) if not args.no_paths else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cores = os.cpu_count() or 1
        fl, sec, desc = oracle_sample(args.cpu_budget / 2, threads=cores)
        fl1, sec1, desc1 = oracle_sample(args.cpu_budget / 2, threads=1)
        cpu = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": desc,
               "single_thread": {"value": fl1 / sec1 / 1e12, "cores": 1, "sample": desc1},
               "extrapolated_seconds_per_step": round(step_flops / (fl / sec), 1),
               "extrapolated": "one step of the sweep (all 19 launches, 17 026 rows) at the sampled all-core rate"}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_obj(world), "roofline": roofline, "sweep": sweep, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clk, "gpu_launches": nM * args.steps, "peaks": peaks, "paths": paths,
        "kernel_ms_per_step": round(kernel_ms_total, 4), "static_w": STATIC_W,
        "timing": "timed region: K replays of the 19-launch sweep captured in CUDA graphs (one per rotation "
                  "offset); eager_ms_per_step: the same sweep through eager per-call launches",
        "eager_ms_per_step": round(eager_ms, 4),
    }
    g.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_cublas_context(Xs, Ws, g, stream, reps=30):
    """Context only, not a target: torch.matmul (cuBLAS, batch-variant) on the same launches,
    timed the same way (graphs of `reps` launches over the rotating cold copies), and per M the
    byte differences between rows 0..M-1 computed alone and the same rows of the full 8192-row
    product, for torch.matmul and for this library."""
    import torch
    X0, W0 = Xs[0], Ws[0]
    full_cublas = torch.matmul(X0, W0)
    full_ours = g(X0, W0)
    out = {}
    for M in M_SWEEP:
        y = torch.empty((M, N_DIM), dtype=torch.bfloat16, device=X0.device)
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm):
            for j in range(reps):
                torch.matmul(Xs[j % len(Xs)][:M], Ws[j % len(Ws)], out=y)
        gm.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gm.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / reps)
        del gm
        alone_c = torch.matmul(X0[:M], W0)
        alone_o = g(X0[:M], W0)
        diff_c = int((alone_c.view(torch.int16) != full_cublas[:M].view(torch.int16)).sum().item()) * 2
        diff_o = int((alone_o.view(torch.int16) != full_ours[:M].view(torch.int16)).sum().item()) * 2
        out[M] = {"cublas_us": round(statistics.median(ts) * 1e3, 2),
                  "cublas_byte_diff_vs_rows_of_M8192": diff_c, "ours_byte_diff_vs_rows_of_M8192": diff_o}
    return out


def measure_e2e(g, W_np, X_np, args, dev, world):
    """The same sweep through the public call with host buffers: every step copies W and each
    x[:M] from pinned host memory, runs, and reads each y[:M] back to pinned host memory.  The
    copies are pipelined with the GEMMs as a user would: host-to-device copies on one stream,
    GEMMs on the compute stream, device-to-host copies on a third, ordered by events.  Each
    launch has its own x and y regions, and W, x and y alternate between two device buffers from
    step to step: a step's copies into a buffer wait for the GEMMs of the step that last read it,
    and its GEMMs wait for the read-back of the step that last wrote its y, so that no copy or
    GEMM touches data another one still uses."""
    import numpy as np
    import torch
    steps = max(2, min(args.steps, 10))
    offs, o = [], 0
    for M in M_SWEEP:
        offs.append(o)
        o += M
    rows = o
    Wh = torch.from_numpy(W_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    Xh = torch.empty((rows, K_DIM), dtype=torch.bfloat16).pin_memory()
    for M, off in zip(M_SWEEP, offs):
        Xh[off:off + M] = torch.from_numpy(X_np[:M].view(np.int16)).view(torch.bfloat16)
    Yh = torch.empty((rows, N_DIM), dtype=torch.bfloat16).pin_memory()
    Wd = [torch.empty_like(Wh, device=dev) for _ in range(2)]
    Xd = [torch.empty((rows, K_DIM), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    Yd = [torch.empty((rows, N_DIM), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # per buffer set: the GEMMs of the step that last read its W and x, the read-back of the step
    # that last wrote its y
    state = {"in_free": [None, None], "out_free": [None, None], "last": None}

    def step(s):
        b = s % 2
        with torch.cuda.stream(h2d):
            if state["in_free"][b] is not None:
                h2d.wait_event(state["in_free"][b])       # the GEMMs of step s-2 read this W and x
            Wd[b].copy_(Wh, non_blocking=True)
            xs = []
            for M, off in zip(M_SWEEP, offs):
                Xd[b][off:off + M].copy_(Xh[off:off + M], non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(h2d)
                xs.append(ev)
        if state["out_free"][b] is not None:
            comp.wait_event(state["out_free"][b])         # step s-2's y has been read back
        for i, (M, off) in enumerate(zip(M_SWEEP, offs)):
            comp.wait_event(xs[i])
            g(Xd[b][off:off + M], Wd[b], Yd[b][off:off + M], stream=comp)
            done = torch.cuda.Event()
            done.record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(done)
                Yh[off:off + M].copy_(Yd[b][off:off + M], non_blocking=True)
        free = torch.cuda.Event()
        free.record(comp)
        state["in_free"][b] = free
        last = torch.cuda.Event()
        last.record(d2h)
        state["out_free"][b] = last
        state["last"] = last

    step(0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e0.record(comp)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    for s in range(steps):
        step(s + 1)
    comp.wait_event(state["last"])                  # every result is back in host memory
    e1.record(comp)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    # the pipelined results are the GEMM's: compare a few launches with a direct device run
    for i in (0, len(M_SWEEP) // 2, len(M_SWEEP) - 1):
        M, off = M_SWEEP[i], offs[i]
        ref = g(Xd[0][off:off + M], Wd[0])
        assert torch.equal(Yh[off:off + M].view(torch.int16), ref.cpu().view(torch.int16)), f"e2e M={M}"
    h2d_bytes = 2 * K_DIM * N_DIM + sum(2 * M * K_DIM for M in M_SWEEP)
    d2h_bytes = sum(2 * M * N_DIM for M in M_SWEEP)
    fl = sum(flops(M) for M in M_SWEEP) * steps * world
    # the host link alone: the same copies per step, both directions at once, without the GEMMs
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(comp)
    h2d.wait_event(c0)
    d2h.wait_event(c0)
    for s in range(steps):
        with torch.cuda.stream(h2d):
            Wd[s % 2].copy_(Wh, non_blocking=True)
            Xd[s % 2].copy_(Xh, non_blocking=True)
        with torch.cuda.stream(d2h):
            Yh.copy_(Yd[s % 2], non_blocking=True)
    comp.wait_stream(h2d)
    comp.wait_stream(d2h)
    c1.record(comp)
    torch.cuda.synchronize()
    link_ms = c0.elapsed_time(c1) / steps
    return {"value": round(fl / (ms / 1e3) / 1e12, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d_bytes,
            "d2h_bytes_per_step": d2h_bytes, "steps": steps, "ms_per_step": round(ms / steps, 3),
            "copies_only_ms_per_step": round(link_ms, 3),
            "copies_only_gbs": round((h2d_bytes + d2h_bytes) / (link_ms / 1e3) / 1e9, 1),
            "how": "pinned host buffers; host-to-device copies, GEMMs and device-to-host copies on three "
                   "streams ordered by events (copies overlap GEMMs of other launches; W, x and y in two "
                   "device buffer sets used by alternate steps, each reuse ordered after the last use); "
                   "copies_only: the same bytes copied both ways at once without the GEMMs, the host "
                   "link's own time"}


def measure_other_paths(dev, peaks):
    """Short timings of the other hot-path rows: fixed split-K (small-N long-K, fp32 out),
    MXFP8 block-scaled (LLM shape) and the linspace shape (fp32 out)."""
    import numpy as np
    import torch
    import inputgen as ig
    from invariant_bi_gemm_gb300 import BiGemm

    def timeit(fn, reps=20):
        """Seconds per launch: a CUDA graph of `reps` launches, replayed and timed with events."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for _ in range(reps):
                fn()
        gr.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gr.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / reps)
        return statistics.median(ts) / 1e3

    def bf(a):
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)

    out = {}
    # fixed split-K, S = 32: x[M,16384]·W[16384,24], fp32 out
    K, N = 16384, 24
    W = bf(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    X = bf(ig.scaled_rows_bf16(ig.SEED_X, 256, K))
    g = BiGemm(K, N, "bf16_f32")
    rows = []
    for M in (1, 64, 128, 256):
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        t = timeit(lambda: g(X[:M], W, y))
        by = algo_bytes(M, K, N, out_bytes=4)
        rows.append({"M": M, "us": round(t * 1e6, 2), "gbs": round(by / t / 1e9, 1),
                     "frac_hbm": round(by / (peaks["hbm_gbs"] * 1e9) / t, 3)})
    out["splitk_small_n_long_k"] = {"shape": "x[M,16384]·W[16384,24] bf16 -> fp32, S=32", "split_k": g.config["split_k"],
                                    "rows": rows, "note": "graph-timed, warm L2 (operands < 10 MB); latency-bound"}
    g.close()
    # MXFP8 at the LLM shape: three rotating (x, sx, W, sw) sets (3 x 94 MB, more than twice the
    # L2), so that every launch reads its operands from HBM; the warm column reuses one set
    K, N = 4096, 14336
    x8 = torch.from_numpy(ig.normal_e4m3(ig.SEED_X, 8192, K)).to(dev)
    sx = torch.from_numpy(ig.e8m0_scales("VAR", ig.SEED_X, 8192, K // 32)).to(dev)
    w8 = torch.from_numpy(ig.normal_e4m3(ig.SEED_W, K, N)).to(dev)
    sw = torch.from_numpy(ig.e8m0_scales("VAR", ig.SEED_W, K // 32, N)).to(dev)
    sets = [(x8, sx, w8, sw)] + [tuple(t.clone() for t in (x8, sx, w8, sw)) for _ in range(2)]
    g = BiGemm(K, N, "mxfp8", static_w=STATIC_W)
    p8 = 2.0 * peaks["bf16_tflops"]
    rows = []
    for M in (1, 64, 256, 2048, 8192):
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        state = {"i": 0}

        def cold():
            xa, sxa, wa, swa = sets[state["i"] % 3]
            state["i"] += 1
            g(xa[:M], wa, y, sx=sxa[:M], sw=swa)

        t = timeit(cold, reps=12)
        tw = timeit(lambda: g(x8[:M], w8, y, sx=sx[:M], sw=sw), reps=12)
        fl = flops(M, K, N)
        by = M * K + K * N + (M * K + K * N) / 32 + 2 * M * N
        t_roof = max(fl / (p8 * 1e12), by / (peaks["hbm_gbs"] * 1e9))
        rows.append({"M": M, "us": round(t * 1e6, 2), "tflops": round(fl / t / 1e12, 1), "frac": round(t_roof / t, 3),
                     "gbs": round(by / t / 1e9, 1), "bound": "hbm" if by / (peaks["hbm_gbs"] * 1e9) > fl / (p8 * 1e12)
                     else "tensor", "us_warm_l2": round(tw * 1e6, 2), "frac_warm_l2": round(t_roof / tw, 3)})
    out["mxfp8_llm"] = {"shape": "E4M3 x[M,4096]·W[4096,14336], E8M0 per 32 K (VAR,VAR), bf16 out",
                        "fp8_peak_tflops": p8, "fp8_peak_source": "2x measured bf16 (nominal fp8/bf16 ratio)",
                        "rows": rows, "note": "graph-timed; us: three rotating operand sets (cold L2); "
                                              "us_warm_l2: one set"}
    g.close()
    del sets, x8, sx, w8, sw
    # linspace shape, fp32 out, M = 2048
    a = bf(ig.linspace_bf16(-1000, 1000, 2048, 4096))
    b = bf(ig.linspace_bf16(-1000, 1000, 4096, 4096))
    g = BiGemm(4096, 4096, "bf16_f32")
    y = torch.empty((2048, 4096), dtype=torch.float32, device=dev)
    t = timeit(lambda: g(a, b, y))
    out["linspace_2048x4096x4096_f32"] = {"us": round(t * 1e6, 2), "tflops": round(flops(2048, 4096, 4096) / t / 1e12, 1),
                                          "frac_tensor": round(flops(2048, 4096, 4096) / t / 1e12 / peaks["bf16_tflops"], 3)}
    g.close()
    out["rmsnorm"] = measure_rmsnorm(dev, peaks, bf)
    out["attention_decode"] = measure_attention(dev, peaks)
    # mHC pre-norm projection (RMSNorm of the flattened streams times W), fp32 out
    from invariant_bi_gemm_gb300 import BiPreNorm
    K, N = 16384, 24
    W = bf(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    X = bf(ig.scaled_rows_bf16(ig.SEED_X, 256, K))
    h = BiPreNorm(K, N, 1e-6)
    rows = []
    for M in (1, 16, 64, 128, 256):
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        t = timeit(lambda: h(X[:M], W, y))
        by = 2 * M * K + 2 * K * N + 4 * M * N
        rows.append({"M": M, "us": round(t * 1e6, 2), "gbs": round(by / t / 1e9, 1),
                     "frac_hbm": round(by / (peaks["hbm_gbs"] * 1e9) / t, 3)})
    out["prenorm_mhc"] = {"shape": "RMSNorm(x[M,16384]) . W[16384,24], bf16 in, fp32 out, chunk 512 (32 splits)",
                          "config": h.config, "rows": rows,
                          "note": "graph-timed, warm L2 (operands < 10 MB); two kernels per call; latency-bound"}
    h.close()
    return out


ATTN = {"num_q_heads": 32, "num_kv_heads": 8, "head_dim": 128, "page_size": 16, "split_size": 512}


def attention_bytes(B, L, a=ATTN):
    """Algorithmic HBM bytes of one decode step: every request's keys and values once, its query
    and output."""
    return 2 * B * L * a["num_kv_heads"] * a["head_dim"] * 2 + 2 * B * a["num_q_heads"] * a["head_dim"] * 2


def measure_attention(dev, peaks):
    """Batch-invariant decode attention (one query token per request at its last position) over
    a paged bf16 cache with shuffled pages, 32 query heads on 8 KV heads of 128, 16-position pages,
    split size 512; graph-timed.  Values are seeded normals drawn on the device (timing only)."""
    import torch
    from invariant_bi_gemm_gb300 import BiAttention

    a = ATTN
    attn = BiAttention(a["num_q_heads"], a["num_kv_heads"], a["head_dim"], a["page_size"], split_size=a["split_size"])
    rows = []
    for B, L in ((1, 32768), (8, 4096), (32, 4096), (64, 8192), (256, 2048)):
        pages_per = (L + a["page_size"] - 1) // a["page_size"]
        P = B * pages_per
        g = torch.Generator(device=dev).manual_seed(1234)
        shape = (P, a["page_size"], a["num_kv_heads"], a["head_dim"])
        kc = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
        vc = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
        table = torch.randperm(P, generator=g, device=dev).to(torch.int32).view(B, pages_per).contiguous()
        q = torch.randn((B, a["num_q_heads"], a["head_dim"]), generator=g, device=dev).to(torch.bfloat16)
        q_seq = torch.arange(B, dtype=torch.int32, device=dev)
        q_pos = torch.full((B,), L - 1, dtype=torch.int32, device=dev)
        o = torch.empty_like(q)
        fn = lambda: attn(q, q_seq, q_pos, kc, vc, table, L - 1, o)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        reps = 10
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for _ in range(reps):
                fn()
        gr.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            gr.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / reps / 1e3)
        t = statistics.median(ts)
        by = attention_bytes(B, L)
        rows.append({"batch": B, "context": L, "us": round(t * 1e6, 2), "gbs": round(by / t / 1e9, 1),
                     "frac_hbm": round(by / t / 1e9 / peaks["hbm_gbs"], 3)})
        del kc, vc, table, q, o, gr
    err = attn.device_error()
    cfg = attn.config
    attn.close()
    return {"shape": "decode: q[B,32,128] over a paged bf16 KV cache [pages,16,8,128], one token per request at "
                     "position context-1, split size 512 positions",
            "grid_bound": cfg["max_ctas"], "rows": rows, "device_error": err,
            "kernel": ("TMA page boxes: a producer warp and four consumer warps per block, "
                       f"{cfg['ring_stages']}-stage ring at three blocks per SM; a call that fits one round of "
                       "four blocks per SM but not of three (the 512-unit shapes here) runs the same kernel built "
                       "for four, with a 2-stage ring" if cfg["tma_pages"] else
                       f"cp.async row copies, {cfg['ring_stages']}-stage ring") + f", {cfg['threads']} threads",
            "bytes": "K and V of every request once (2 x B x context x 8 x 128 x 2) + q and o",
            "note": "graph-timed; pages shuffled over the cache; two kernels per call (attention, merge), plus a "
                    "plan kernel for calls of more than 32 tokens"}


RMS_D = 4096
RMS_EPS = 1e-6


def rmsnorm_bytes(M, d=RMS_D):
    """Algorithmic HBM bytes of one RMSNorm launch: x read once, y written once, the weight."""
    return 2 * M * d + 2 * M * d + 2 * d


def measure_rmsnorm(dev, peaks, bf):
    """Batch-invariant RMSNorm of bf16 rows, d = 4096 (the LLM projection's K), graph-timed with
    rotating (x, y) sets whose total exceeds twice the L2, so every launch reads cold rows."""
    import numpy as np
    import torch
    import inputgen as ig
    from invariant_bi_gemm_gb300 import BiRmsNorm

    n = BiRmsNorm(RMS_D, RMS_EPS)
    gw = bf(ig.rmsnorm_weight_bf16(ig.SEED_W, RMS_D))
    base = bf(ig.scaled_rows_bf16(ig.SEED_X, 8192, RMS_D))
    rows = []
    for M in (1, 64, 256, 2048, 8192, 32768):
        per_set = 4 * M * RMS_D
        nsets = max(3, min(64, int(2 * 256e6 // per_set) + 1))
        xs = [base.repeat((M + 8191) // 8192, 1)[:M].contiguous() for _ in range(nsets)]
        ys = [torch.empty_like(x) for x in xs]
        reps = nsets * max(1, 30 // nsets)
        for i in range(3):
            n(xs[i % nsets], gw, ys[i % nsets])
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(reps):
                n(xs[i % nsets], gw, ys[i % nsets])
        gr.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gr.replay()
            b.record()
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b) / reps / 1e3)
        t = statistics.median(ts)
        by = rmsnorm_bytes(M)
        rows.append({"M": M, "us": round(t * 1e6, 2), "gbs": round(by / t / 1e9, 1),
                     "frac_hbm": round(by / t / 1e9 / peaks["hbm_gbs"], 3)})
        del xs, ys, gr
    cfg = n.config
    n.close()
    return {"shape": f"bf16 x[M,{RMS_D}] -> y[M,{RMS_D}], weight [{RMS_D}], eps {RMS_EPS}",
            "threads_per_row": cfg["threads"], "grid_bound": cfg["max_ctas"], "rows": rows,
            "bytes": "2Md (x) + 2Md (y) + 2d (weight)",
            "note": "graph-timed; rotating (x, y) sets > 2x L2 for every M; small M is launch-latency-bound"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of CPU oracle work")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-paths", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_init()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
