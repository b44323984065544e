#!/usr/bin/env python3
"""Benchmark of the fused GEMM + collective kernels on GB300.

One step = one call of the fused op over one batch of synthetic input: by
default matmul_reduce_scatter, W=4 emulated ranks, A_r and B_r 4096 x 4096
fp16, bias fp16 (N = 4096), uniform inputs (seed 1) -- all W ranks' GEMMs,
the fp32 partials, the rank-order reduction and the scatter run inside the
one persistent kernel.  Prints one JSON line (rank 0), last.

Before that line, the default single-GPU run also measures every other
workload of the family, one compact JSON line each (and a summary of them
inside the last line): all_gather_matmul and matmul_all_gather W=8 4096 x
14336 x 4096 bf16, the concurrent bf16 GEMM 8192^3 beside an all-reduce of
8 x 64Mi fp32 (with the sequential arms and a gemm_ctas sweep from 25 % to
90 % of the SMs), all_gather_matmul W=8 131072 x 16384 x 16384 bf16,
matmul_all_reduce W=8 8192^3 bf16 and the small all_gather_matmul W=2 256^3.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--config '{"gemm_ctas": 100}'] [--headline-only]

--impl reference times the CPU oracle (the plain definition of the same op)
on this machine's host cores, each step a bounded row slice of the workload.
Under torchrun every rank runs an independent replica (the emulated ranks all
live on one GPU; there is no data-path collective between GPUs).
"""
from __future__ import annotations

import argparse
import ctypes
import glob
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

import torch  # noqa: E402

import synthetic  # noqa: E402

METRIC = "fused AG+GEMM / GEMM+RS TFLOPS on 1 GB300; % of max(tensor, HBM) roofline"
DEFAULT_WORKLOAD = "mm_rs_w4_4096"
L2_BYTES = 129 * 1024 * 1024
KERNEL_NAME = "fused_gemm_coll_kernel"
OP_NAMES = {"ag_mm": "all_gather_matmul", "mm_rs": "matmul_reduce_scatter",
            "mm_ag": "matmul_all_gather", "mm_ar": "matmul_all_reduce"}
# Published all_gather_matmul TFLOPS for the same shapes at world size 8
# (ROCm/iris PR #506, "Performance (ws=8, MI300X)" table): another GPU, so
# vs_baseline is context, not a target.  The pages publish no numbers for the
# other ops or the concurrent mode.
PAGES_TFLOPS_MI300X = {
    ("ag_mm", 8, 131072, 16384, 16384): 420.5, ("ag_mm", 8, 147456, 28672, 4096): 466.5,
    ("ag_mm", 8, 327680, 28672, 4096): 474.7, ("ag_mm", 8, 229376, 28672, 4096): 471.5,
    ("ag_mm", 8, 8192, 8192, 262144): 161.6, ("ag_mm", 8, 262144, 8192, 8192): 253.0,
    ("ag_mm", 8, 16384, 16384, 131072): 314.5, ("ag_mm", 8, 262144, 28672, 8192): 442.1,
    ("ag_mm", 8, 196608, 18432, 16384): 445.4, ("ag_mm", 8, 4096, 14336, 4096): 248.9,
    ("ag_mm", 8, 4096, 11008, 4096): 189.8, ("ag_mm", 8, 4096, 4096, 4096): 90.9,
}


def pages_tflops(op, W, M, N, K):
    return PAGES_TFLOPS_MI300X.get((op, W, M, N, K))


# ------------------------------------------------------------------ helpers

def release_memory():
    """Return the cached device memory of a finished workload to the CUDA
    driver, then wait until it has been cleared: the GPU driver zeroes freed
    device memory in the background: right after 150 GB were freed, the headline
    kernel ran 486-501 us per step instead of 350-360 for about 42 ms, the
    time that clearing takes at ~3.6 TB/s.  Waiting at 2 TB/s of freed bytes
    keeps that clearing out of the next workload's timed steps."""
    before = torch.cuda.memory_reserved()
    torch.cuda.empty_cache()
    freed = before - torch.cuda.memory_reserved()
    torch.cuda.synchronize()
    if freed > 0:
        time.sleep(min(3.0, 0.05 + freed / 2e12))


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "gemm_collective_tiles_gb300", "csrc", "*"))):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """Per-launch DRAM bytes from the committed ncu summary of this workload,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.tmp, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.tmp.flush()
        rows = []
        with open(self.tmp.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.tmp.name)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "reasons": sorted(reasons)}


def blas_threads() -> int:
    """Threads numpy's BLAS uses (OpenBLAS queried directly when loaded)."""
    try:
        import numpy  # noqa: F401
        with open("/proc/self/maps") as f:
            libs = {line.split()[-1] for line in f if "openblas" in line.lower() and line.split()[-1].startswith("/")}
        for lib in libs:
            try:
                fn = ctypes.CDLL(lib).openblas_get_num_threads
                fn.restype = ctypes.c_int
                n = int(fn())
                if n > 0:
                    return n
            except (OSError, AttributeError):
                continue
    except Exception:
        pass
    return os.cpu_count() or 1


def max_over_ranks(x: float, pg) -> float:
    """The largest value of x over all ranks (identity without a process
    group); the tensor lives on the device the backend works on."""
    if pg is None:
        return float(x)
    dev = "cuda" if pg.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, world: int, steps: int, total_ms: float) -> float:
    """Whole-job TFLOP/s: every rank processes flops_per_step per step, the
    job takes the slowest rank's time."""
    return flops_per_step * steps * world / (total_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ CPU side

def oracle_rows(wl: dict, x, rows: int):
    """Run the oracle on the first `rows` output rows of every rank (all of N
    and K): returns the flops that sample represents."""
    import oracle
    op, W = wl["op"], wl["W"]
    if op == "mm_rs":
        oracle.matmul_reduce_scatter([a[:rows] for a in x.A], x.B, x.bias)
        return 2.0 * W * rows * wl["N"] * wl["K"]
    if op == "mm_ar":
        oracle.matmul_all_reduce([a[:rows] for a in x.A], x.B, x.bias)
        return 2.0 * W * rows * wl["N"] * wl["K"]
    if op == "ag_mm":
        oracle.all_gather_matmul([a[:rows] for a in x.A], x.B[0], x.bias)
        return 2.0 * rows * wl["N"] * wl["K"]
    oracle.matmul_all_gather([a[:rows] for a in x.A], x.B[0], x.bias)
    return 2.0 * W * rows * wl["N"] * wl["K"]


def size_oracle_sample(wl: dict, x, target_s: float):
    """Rows of every rank whose oracle run takes about target_s on this host,
    from two probes that separate the per-call cost (operand conversion) from
    the per-row cost.  Returns (rows, max_rows, seconds per pass over all rows)."""
    max_rows = wl["M"] if wl["op"] != "mm_ag" else wl["M"] // wl["W"]
    probe = [min(32, max_rows), min(128, max_rows)]
    times = []
    for r in probe:
        t0 = time.perf_counter()
        oracle_rows(wl, x, r)
        times.append(time.perf_counter() - t0)
    per_row = max((times[1] - times[0]) / max(probe[1] - probe[0], 1), 1e-7)
    fixed = max(times[0] - probe[0] * per_row, 0.0)
    rows = int(min(max_rows, max(probe[0], (target_s - fixed) / per_row)))
    return rows, max_rows, fixed + max_rows * per_row


def host_threads() -> dict:
    return {"cores": blas_threads(), "nproc": os.cpu_count() or 1}


def cpu_baseline(wl: dict, x, target_s: float = 12.0):
    """The oracle, as it stands, on a bounded sample of the workload: a row
    slice sized to about target_s, or -- when the host finishes every row
    sooner -- whole passes over all rows, repeated up to about target_s."""
    budget = target_s * 0.8
    rows, max_rows, full_s = size_oracle_sample(wl, x, budget)
    passes = 1
    if rows == max_rows:
        passes = int(max(1, min(20, budget / max(full_s, 1e-3))))
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(passes):
        flops += oracle_rows(wl, x, rows)
    dt = time.perf_counter() - t0
    what = (f"{passes} passes over all {rows} output rows of every rank" if passes > 1
            else f"first {rows} output rows of every rank")
    th = host_threads()
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": th["cores"], "nproc": th["nproc"],
            "kind": "oracle",
            "sample": f"{what} (full N={wl['N']}, K={wl['K']}), {flops:.3g} flop in {dt:.2f} s "
                      f"(fp64 dot products, numpy BLAS on {th['cores']} threads of {th['nproc']} cores)"}


def run_reference(args, wl, name, cfg):
    """The reference arm: the CPU oracle, as it stands, on the host cores.
    Each step runs the oracle on the first `rows` output rows of every rank
    (all of N and K), the same sample kind as the cpu_baseline leg, sized so
    that the whole --steps/--warmup run takes about two minutes."""
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    x = synthetic.make_fused_inputs(**wl)
    steps, warm = args.steps, args.warmup
    rows, _max_rows, _ = size_oracle_sample(wl, x, 120.0 / (steps + warm))
    for _ in range(warm):
        oracle_rows(wl, x, rows)
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(steps):
        flops += oracle_rows(wl, x, rows)
    dt = time.perf_counter() - t0
    val = flops / dt / 1e12
    th = host_threads()
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "ms_per_step": dt / steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(wl, name, cfg, args.gpus),
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": th["cores"], "nproc": th["nproc"],
                             "kind": "oracle",
                             "sample": f"first {rows} output rows of every rank per step (full N={wl['N']}, "
                                       f"K={wl['K']}; fp64 dot products, numpy BLAS)"},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU side

def workload_config(wl, name, cfg):
    d = {"workload": f"{OP_NAMES[wl['op']]} W={wl['W']} M={wl['M']} N={wl['N']} K={wl['K']} "
                     f"{wl['dtype']}{' +bias' if wl.get('bias') else ''} ({name})",
         "op": OP_NAMES[wl["op"]], "world_size_emulated": wl["W"], "M": wl["M"], "N": wl["N"],
         "K": wl["K"], "seed": wl["seed"], "dist": wl["dist"]}
    d.update({k: v for k, v in cfg.items()})
    return d


def bench_config(wl, name, cfg, world):
    """The `config` object of a bench line; both arms print the same one."""
    d = workload_config(wl, name, cfg)
    d["l2"] = "flushed before every step (258 MB memset outside the step's events)"
    d["parallelism"] = f"replicas x{world}" if world > 1 else "1 GPU"
    return d


def library_reference(prob, wl, stream, flush):
    """The same op done the plain sequential way with library calls on the same
    device data: cuBLAS GEMMs (16-bit outputs, as torch.matmul gives) plus
    torch cat / sum / slice for the collective part.  Run-only (its results
    are not checked); timed like the bench line, back to back with an L2 flush
    before every call."""
    op, W = wl["op"], wl["W"]
    A = [prob.heap.view(prob.A, r) for r in range(W)]
    B = [prob.heap.view(prob.B, r if prob.per_rank_b() else 0) for r in range(W)]
    bias = prob.heap.view(prob.bias, 0) if prob.bias is not None else None

    def add_bias(x):
        return x if bias is None else x + bias

    if op == "ag_mm":
        def fn():
            return add_bias(torch.cat(A, dim=1) @ B[0])
        what = "torch.cat of the W shards, then one cuBLAS matmul"
    elif op == "mm_ag":
        def fn():
            return torch.cat([add_bias(a @ B[0]) for a in A], dim=0)
        what = "W cuBLAS matmuls, then torch.cat along M"
    else:
        def fn():
            s = torch.stack([add_bias(A[r] @ B[r]).float() for r in range(W)]).sum(0)
            return torch.chunk(s.to(A[0].dtype), W, dim=1) if op == "mm_rs" else s.to(A[0].dtype)
        what = "W cuBLAS matmuls (16-bit partials), fp32 torch.sum over ranks, " + (
            "split along N" if op == "mm_rs" else "rounded once")
    flops = prob.flops()
    reps = max(3, min(20, int(2e16 / flops)))
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
    return {"what": what, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "reps": reps}


def concurrent_measure(cfg, steps, warm, sweep=False, two_stream=False):
    """Independent GEMM (bf16 8192^3, normal(0,1), seed 3) sharing the SMs with
    an all-reduce of W=8 fp32 buffers of 64Mi elements (uniform[-1,1], seed 4),
    in one launch.  Also times the sequential arms (the GEMM alone on every
    SM, then the all-reduce alone on every SM); optionally the gemm_ctas
    sweep and the two-stream modes.  The roofline is max(GEMM flop / tensor
    peak, all bytes / HBM bandwidth), the bytes counting the collective's
    W reads and W writes and the GEMM's A, B and C once.  The all-reduce
    writes a separate output (the same bytes as in place, and the inputs stay
    unchanged across steps)."""
    from gemm_collective_tiles_gb300 import query_status
    from gemm_collective_tiles_gb300.runner import ConcurrentProblem
    cw = synthetic.CONCURRENT_WORKLOAD
    torch.cuda.set_device(0)
    A, B = synthetic.make_gemm_inputs(cw["M"], cw["N"], cw["K"], cw["gemm_dtype"], cw["gemm_seed"],
                                      dist="normal", scale=1.0)
    X = synthetic.make_coll_inputs(cw["W"], cw["count"], cw["coll_dtype"], cw["coll_seed"])
    peaks, peak_kind = measured_peaks()

    def make(conf, gemm=True, coll=True):
        pr = ConcurrentProblem(cw["M"] if gemm else 0, cw["N"] if gemm else 0, cw["K"] if gemm else 0,
                               cw["gemm_dtype"], "all_reduce", cw["W"], cw["count"] if coll else 0,
                               coll_dtype=cw["coll_dtype"], config=conf or None)
        pr.upload(A if gemm else None, B if gemm else None, X if coll else None)
        return pr

    def timeit(probs, n, w):
        stream = torch.cuda.current_stream()
        for _ in range(w):
            for pr in probs:
                pr.run(stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            for pr in probs:
                pr.run(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        for pr in probs:
            rc = query_status(pr.ws, stream)
            if rc[0] != 0:
                raise RuntimeError(f"device status {rc}")
        return e0.elapsed_time(e1) / n

    flops = 2.0 * cw["M"] * cw["N"] * cw["K"]
    coll_bytes = 2.0 * cw["W"] * cw["count"] * 4
    gemm_bytes = 2.0 * (cw["M"] * cw["K"] + cw["K"] * cw["N"] + cw["M"] * cw["N"])
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12) * 1e3
    t_hbm = (coll_bytes + gemm_bytes) / (peaks["hbm_gbs"] * 1e9) * 1e3
    t_roof = max(t_tensor, t_hbm)
    fused = make(cfg)
    sampler = ClockSampler(0)
    sampler.start()
    ms = timeit([fused], steps, warm)
    clocks = sampler.stop()
    del fused
    res = {"flops": flops, "ms": ms, "clocks": clocks, "peak_kind": peak_kind,
           "roofline": {"bound": "hbm" if t_hbm >= t_tensor else "tensor", "roofline_ms": t_roof,
                        "frac": t_roof / ms, "bytes": coll_bytes + gemm_bytes,
                        "peak_source": f"{peak_kind} bf16 burst and HBM copy"}}
    g_only = make(cfg, coll=False)
    ms_g = timeit([g_only], steps, warm)
    del g_only
    c_only = make(cfg, gemm=False)
    ms_c = timeit([c_only], steps, warm)
    del c_only
    res["sequential"] = {"gemm_ms": ms_g, "all_reduce_ms": ms_c, "sum_ms": ms_g + ms_c,
                         "speedup_concurrent_vs_sequential": (ms_g + ms_c) / ms,
                         "gemm_tflops_alone": flops / (ms_g * 1e-3) / 1e12,
                         "all_reduce_gbs_alone": coll_bytes / (ms_c * 1e-3) / 1e9}
    if sweep:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        pts = {}
        for frac in (0.25, 0.35, 0.45, 0.55, 0.65, 0.7, 0.75, 0.85, 0.9):
            conf = dict(cfg)
            conf["gemm_ctas"] = max(1, int(round(frac * sms)))
            pr = make(conf)
            pts[str(conf["gemm_ctas"])] = timeit([pr], max(3, steps // 2), 2)
            del pr
        conf = dict(cfg)
        conf["gemm_ctas"] = -1
        pr = make(conf)
        pts["balanced"] = timeit([pr], max(3, steps // 2), 2)
        del pr
        res["gemm_ctas_sweep_ms"] = pts
    if two_stream:
        from gemm_collective_tiles_gb300 import make_config, sm_partition_release, sm_partition_streams
        two = make(cfg)
        sms_all = torch.cuda.get_device_properties(0).multi_processor_count

        def time_two(conf, s_g, s_c):
            two.config = make_config(**conf)
            for _ in range(2):
                two.run_two_stream(s_g, s_c)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(steps):
                two.run_two_stream(s_g, s_c)
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) * 1e3 / steps
        s_g, s_c = torch.cuda.Stream(), torch.cuda.Stream()
        res["two_stream_ms_by_gemm_ctas"] = {
            str(g): time_two({**cfg, "gemm_ctas": g}, s_g, s_c)
            for g in (sms_all // 2, int(sms_all * 0.55), int(sms_all * 0.45))}
        # the same on two green contexts with disjoint SM sets (the split
        # enforced by the CUDA driver): the GEMM stream gets at least g SMs
        green = {}
        for g in (72, 80, 88, 96):
            s_gemm, s_comm, gs, cs = sm_partition_streams(g)
            try:
                green[str(gs)] = time_two({**cfg, "gemm_ctas": gs, "grid": gs + cs}, s_gemm, s_comm)
            finally:
                torch.cuda.synchronize()
                sm_partition_release()
        res["two_stream_green_ctx_ms_by_gemm_sms"] = green
        del two
    release_memory()
    return res


def run_concurrent(args, cfg):
    steps = max(3, min(args.steps, 200))
    warm = max(3, args.warmup)
    r = concurrent_measure(cfg, steps, warm, sweep=args.sweep, two_stream=True)
    line = {"metric": "concurrent GEMM + all-reduce step: GEMM TFLOPS over the step; % of max(tensor, HBM) roofline",
            "value": r["flops"] / (r["ms"] * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1, "steps": steps,
            "warmup": warm, "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "concurrent: bf16 GEMM 8192^3 || all_reduce W=8 x 64Mi fp32 (concurrent_ar_w8)",
                       **cfg},
            "roofline": r["roofline"], "sequential": r["sequential"], "gpu_launches": steps, "clocks": r["clocks"]}
    for k in ("gemm_ctas_sweep_ms", "two_stream_ms_by_gemm_ctas", "two_stream_green_ctx_ms_by_gemm_sms"):
        if k in r:
            line[k] = r[k]
    print(json.dumps(line), flush=True)
    return 0


def run_shape_sweep(args, cfg):
    """all_gather_matmul at W=8 over the PR #506 shape list (bf16, N(0, 0.02)
    drawn on the device, seed 7 + shape index), each against the sequential
    path it replaces: the gather as one torch.cat of the W K-shards, then a
    cuBLAS matmul.  Prints one JSON row per shape, then a summary line.
    Both arms write into the same region-0 buffers; the fused output of a
    sampled row block is compared with cuBLAS's before the latter overwrites it.
    Each arm is timed as the median of back-to-back calls (L2 flushed before
    every call), like the bench line."""
    from gemm_collective_tiles_gb300 import query_status
    from gemm_collective_tiles_gb300.runner import FusedProblem
    torch.cuda.set_device(0)
    W = 8
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    only = set(args.shapes.split(",")) if args.shapes else None
    rows = []

    def timed(fn, reps, warm=2):
        # back to back like the bench line: an L2 flush, then the timed call,
        # with no host synchronisation (and no idle GPU) between calls
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)

    for idx, (label, M, N, K) in enumerate(synthetic.AG_MM_SHAPES):
        if only and label not in only:
            continue
        per_region = (M * (K // W) + K * N + M * N + M * K) * 2
        free, _total = torch.cuda.mem_get_info()
        if W * per_region > 0.92 * free:
            rows.append({"shape": label, "M": M, "N": N, "K": K, "skipped": f"needs {W * per_region / 1e9:.1f} GB"})
            print(json.dumps(rows[-1]), flush=True)
            continue
        prob = FusedProblem("ag_mm", W, M, N, K, "bf16", config=cfg)
        for r in range(W):
            synthetic.fill_device_(prob.heap.view(prob.A, r), 7 + idx * 16 + r)
        synthetic.fill_device_(prob.heap.view(prob.B, 0), 7 + idx * 16 + W)
        flops = 2.0 * M * N * K
        reps = max(3, min(20, int(2e16 / flops)))
        t0 = time.perf_counter()
        ms_fused = timed(lambda: prob.run(stream), reps)
        rc = query_status(prob.ws, stream)
        if rc[0] != 0:
            raise RuntimeError(f"{label}: device status {rc}")
        out0 = prob.heap.view(prob.out, 0)
        gath0 = prob.heap.view(prob.gathered, 0)
        r0 = (M // 2) // 128 * 128
        fused_rows = out0[r0:r0 + 128].float().cpu()
        shards = [prob.heap.view(prob.A, r) for r in range(W)]
        B0 = prob.heap.view(prob.B, 0)

        def seq():
            torch.cat(shards, dim=1, out=gath0)
            torch.matmul(gath0, B0, out=out0)
        ms_seq = timed(seq, reps)
        ref_rows = out0[r0:r0 + 128].float().cpu()
        rel = float((fused_rows - ref_rows).abs().max() / ref_rows.abs().max().clamp_min(1e-30))
        tf = flops / (ms_fused * 1e-3) / 1e12
        rows.append({"shape": label, "M": M, "N": N, "K": K, "ms": ms_fused, "tflops": tf,
                     "frac_of_peak": tf / peak, "cat_cublas_ms": ms_seq,
                     "cat_cublas_tflops": flops / (ms_seq * 1e-3) / 1e12, "speedup": ms_seq / ms_fused,
                     "max_rel_diff_vs_cublas": rel, "reps": reps, "wall_s": time.perf_counter() - t0,
                     "pages_mi300x_tflops": pages_tflops("ag_mm", W, M, N, K)})
        print(json.dumps(rows[-1]), flush=True)
        del prob, shards, B0, out0, gath0
        release_memory()
    done = [r for r in rows if "tflops" in r]
    print(json.dumps({"metric": "all_gather_matmul W=8 shape sweep (bf16): TFLOP/s and speedup vs torch.cat + cuBLAS",
                      "unit": "TFLOP/s", "n_gpus": 1, "dtype": "bf16", "data": "synthetic",
                      "peak": peak, "peak_source": f"{peak_kind} bf16 burst",
                      "config": {"workload": "ag_mm_shape_sweep", **cfg},
                      "shapes": len(done), "winners": sum(1 for r in done if r["speedup"] > 1.0),
                      "geomean_speedup": statistics.geometric_mean([r["speedup"] for r in done]) if done else None}),
          flush=True)
    return 0


# the workloads measured beside the headline in the default run: (name,
# inputs drawn on the host by the recipe or -- for the multi-GB ones -- on
# the device, steps multiplier)
OTHER_CONFIGS = [
    ("ag_mm_w8_4096x14336x4096", "host", 1),
    ("mm_ag_w8_4096x14336x4096", "host", 1),
    ("ag_mm_w8_131072x16384x16384", "device", 1),
    ("mm_ar_w8_8192", "device", 1),
    ("ag_mm_w2_256", "host", 10),
]


def make_problem(name, cfg, inputs="host"):
    """The fused problem of workload `name` with its inputs in the heap:
    drawn on the host by the workload's recipe (seed, distribution, draw
    order), or for timing-only runs of multi-GB workloads drawn on the device
    from the same seed and distribution (synthetic.fill_device_)."""
    from gemm_collective_tiles_gb300.runner import FusedProblem
    wl = dict(synthetic.WORKLOADS[name])
    prob = FusedProblem(wl["op"], wl["W"], wl["M"], wl["N"], wl["K"], wl["dtype"], bias=wl.get("bias", False),
                        config=cfg)
    x = None
    if inputs == "host":
        x = synthetic.make_fused_inputs(**wl)
        prob.upload(x.A, x.B, x.bias)
    else:
        seed = wl["seed"] * 1000
        for r in range(wl["W"]):
            synthetic.fill_device_(prob.heap.view(prob.A, r), seed + r, wl["dist"], wl["scale"])
            if prob.per_rank_b() or r == 0:
                synthetic.fill_device_(prob.heap.view(prob.B, r), seed + 100 + r, wl["dist"], wl["scale"])
        if prob.bias is not None:
            for r in range(wl["W"] if prob.per_rank_b() else 1):
                synthetic.fill_device_(prob.heap.view(prob.bias, r), seed + 200, "uniform", wl.get("bias_scale", 0.1))
    return wl, prob, x


def time_steps(prob, steps, warm, stream, flush, pg=None, sample_gpu=0):
    """Warm-up, then `steps` timed calls, each bracketed by its own events
    with an L2 flush before it (outside the events).  Returns (per-step ms,
    clocks sampled during the timed region, host wall seconds)."""
    from gemm_collective_tiles_gb300 import query_status
    for _ in range(warm):
        prob.run(stream)
    rc = query_status(prob.ws, stream)
    if rc[0] != 0:
        raise RuntimeError(f"device status after warm-up: {rc}")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    sampler = ClockSampler(sample_gpu)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for i in range(steps):
        flush.zero_()                      # evict L2 between steps (outside the step events)
        starts[i].record(stream)
        prob.run(stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if pg:
        pg.barrier()
    clocks = sampler.stop()
    rc = query_status(prob.ws, stream)
    if rc[0] != 0:
        raise RuntimeError(f"device status after timed steps: {rc}")
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], clocks, wall


def short_clocks(c):
    if not c:
        return None
    return {"sm_mhz": c.get("sm_mhz"), "sm_max_mhz": c.get("sm_max_mhz"), "samples": c.get("samples"),
            "reasons": c.get("reasons")}


def back_to_back_us(prob, stream, n=200):
    """Mean microseconds per call over n calls back to back: issued one by
    one, and replayed from a CUDA graph captured around one call."""
    from gemm_collective_tiles_gb300 import query_status

    def timed(fn):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(torch.cuda.current_stream())
        for _ in range(n):
            fn()
        e1.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        return round(e0.elapsed_time(e1) * 1e3 / n, 2)

    eager = timed(lambda: prob.run(stream))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        prob.run()
    torch.cuda.synchronize()
    replay = timed(g.replay)
    rc = query_status(prob.ws, stream)
    if rc[0] != 0:
        raise RuntimeError(f"device status after the back-to-back calls: {rc}")
    return {"eager": eager, "graph_replay": replay}


def run_other_configs(args, cfg, stream, flush):
    """Every other workload of the family on this GPU, one compact JSON line
    each; returns {name: summary} for the headline line."""
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])
    summary = {}
    for name, inputs, mult in OTHER_CONFIGS:
        wl, prob, _x = make_problem(name, cfg, inputs)
        steps = max(3, args.steps * mult)
        step_ms, clocks, _wall = time_steps(prob, steps, args.warmup, stream, flush)
        flops = prob.flops()
        mean_ms = statistics.mean(step_ms)
        tf = flops / (mean_ms * 1e-3) / 1e12
        base = pages_tflops(wl["op"], wl["W"], wl["M"], wl["N"], wl["K"])
        line = {"config_line": name, "workload": workload_config(wl, name, {})["workload"], "value": tf,
                "unit": "TFLOP/s", "ms_per_step": mean_ms, "median_ms": statistics.median(step_ms),
                "steps": steps, "inputs": inputs,
                "roofline": {"bound": "tensor", "frac": tf / peak, "peak": peak,
                             "peak_source": f"{peak_kind} bf16 burst"},
                "pages_mi300x_tflops": base, "gpu_launches": steps, "clocks": short_clocks(clocks)}
        if wl["M"] * wl["N"] * wl["K"] <= 1 << 27:
            # launch-bound: calls back to back with no flush, issued one by one
            # and replayed from a CUDA graph that holds one call (no host work
            # per call), the kernel's own floor beside the flushed steps
            line["back_to_back_us"] = back_to_back_us(prob, stream)
        print(json.dumps(line), flush=True)
        summary[name] = {"value": round(tf, 1), "ms": round(mean_ms, 4), "frac": round(tf / peak, 4),
                         "steps": steps}
        del prob
        release_memory()
    steps = max(3, args.steps)
    r = concurrent_measure(cfg, steps, args.warmup, sweep=True)
    sweep = r.get("gemm_ctas_sweep_ms", {})
    best = min(sweep.items(), key=lambda kv: kv[1]) if sweep else (None, None)
    pred = predictor_vs_sweep(sweep)
    line = {"config_line": "concurrent_ar_w8",
            "workload": "concurrent: bf16 GEMM 8192^3 || all_reduce W=8 x 64Mi fp32 (default split)",
            "value": r["flops"] / (r["ms"] * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": r["ms"],
            "steps": steps, "roofline": {"bound": r["roofline"]["bound"], "frac": r["roofline"]["frac"],
                                         "roofline_ms": r["roofline"]["roofline_ms"]},
            "sequential_ms": r["sequential"]["sum_ms"],
            "speedup_concurrent_vs_sequential": r["sequential"]["speedup_concurrent_vs_sequential"],
            "gemm_ms_alone": r["sequential"]["gemm_ms"], "all_reduce_ms_alone": r["sequential"]["all_reduce_ms"],
            "gemm_ctas_sweep_ms": {k: round(v, 4) for k, v in sweep.items()}, "best_gemm_ctas": best[0],
            "predictor": pred, "gpu_launches": steps, "clocks": short_clocks(r["clocks"])}
    print(json.dumps(line), flush=True)
    summary["concurrent_ar_w8"] = {"ms": round(r["ms"], 4), "frac": round(r["roofline"]["frac"], 4),
                                   "speedup_vs_sequential": round(r["sequential"]["speedup_concurrent_vs_sequential"], 3),
                                   "best_gemm_ctas": best[0]}
    return summary


def predictor_vs_sweep(sweep):
    """The split predictor's makespans for the measured gemm_ctas points (the
    default tile kind), its best split against the measured best, and the
    rank correlation of the two orders."""
    from gemm_collective_tiles_gb300 import predictor
    cw = synthetic.CONCURRENT_WORKLOAD
    pts = {k: v for k, v in sweep.items() if k.isdigit()}
    if len(pts) < 3:
        return None
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wl = predictor.Workload(M=cw["M"], N=cw["N"], K=cw["K"], coll="all_reduce", W=cw["W"], count=cw["count"])
    tk = next(t for t in predictor.TILE_KINDS if t.name == predictor.PREFERRED_TILE)
    pred = {k: predictor.simulate(wl, int(k), predictor.Machine(sms=sms), tk) / 1e3 for k in pts}
    keys = sorted(pts)

    def ranks(d):
        order = sorted(keys, key=lambda k: d[k])
        return {k: i for i, k in enumerate(order)}
    rp, rm = ranks(pred), ranks(pts)
    n = len(keys)
    rho = 1.0 - 6.0 * sum((rp[k] - rm[k]) ** 2 for k in keys) / (n * (n * n - 1))
    return {"predicted_ms": {k: round(v, 4) for k, v in pred.items()},
            "predicted_best": min(pred, key=pred.get), "measured_best": min(pts, key=pts.get),
            "rank_correlation": round(rho, 3)}


def sustained(prob, stream, peak_sustained, seconds=2.5):
    """The headline op back to back for about `seconds` (no flush between
    calls: the working set is several times the L2), one event pair around
    the whole loop, against the measured sustained peak."""
    for _ in range(20):
        prob.run(stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(50):
        prob.run(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    n = max(50, int(seconds * 1e3 / max(e0.elapsed_time(e1) / 50, 1e-3)))
    sampler = ClockSampler(0)
    sampler.start()
    e0.record(stream)
    for _ in range(n):
        prob.run(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / n
    tf = prob.flops() / (ms * 1e-3) / 1e12
    return {"value": tf, "unit": "TFLOP/s", "ms_per_step": ms, "steps": n, "peak": peak_sustained,
            "frac": tf / peak_sustained, "l2": "not flushed (back to back; working set > L2)",
            "clocks": short_clocks(clocks)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(synthetic.WORKLOADS) + ["concurrent_ar_w8", "ag_mm_shape_sweep"])
    ap.add_argument("--shapes", default="", help="ag_mm_shape_sweep: comma-separated labels (default all)")
    ap.add_argument("--sweep", action="store_true",
                    help="concurrent workload: also time gemm_ctas from 25%% to 90%% of the SMs")
    ap.add_argument("--config", default="{}", help="JSON dict of iris_b200_config fields")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads measured before the headline line")
    ap.add_argument("--e2e-steps", type=int, default=50)
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    cfg = json.loads(args.config)
    if args.workload == "concurrent_ar_w8":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the CPU oracle arm covers the fused-op workloads"}))
            return 0
        return run_concurrent(args, cfg)
    if args.workload == "ag_mm_shape_sweep":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the shape sweep compares against cuBLAS, not the oracle"}))
            return 0
        return run_shape_sweep(args, cfg)
    wl = dict(synthetic.WORKLOADS[args.workload])

    if args.impl == "reference":
        return run_reference(args, wl, args.workload, cfg)

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist

    from gemm_collective_tiles_gb300 import query_status
    from gemm_collective_tiles_gb300.runner import FusedProblem

    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    others = None
    if world == 1 and not args.headline_only and args.workload == DEFAULT_WORKLOAD:
        others = run_other_configs(args, cfg, stream, flush)

    wl, prob, x = make_problem(args.workload, cfg, "host")
    K = args.steps
    step_ms, clocks, wall = time_steps(prob, K, args.warmup, stream, flush, pg, local)
    total_ms = max_over_ranks(sum(step_ms), pg)
    flops = prob.flops()
    value = job_throughput(flops, world, K, total_ms)
    ms_per_step = total_ms / K

    # roofline of the one kernel per step
    peaks, peak_kind = measured_peaks()
    peak = float(peaks["bf16_tflops"])   # fp16 and bf16 share the nominal dense rate (ratio 1)
    achieved = flops / (statistics.mean(step_ms) * 1e-3) / 1e12
    traffic = recorded_traffic(args.workload)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peak_kind} bf16 burst (MEASURED_PEAKS.json) x 1.0 fp16/bf16 nominal ratio",
                "kernel": KERNEL_NAME, "median_ms": statistics.median(step_ms)}
    sus = None
    if world == 1 and not args.headline_only:
        sus = sustained(prob, stream, float(peaks.get("bf16_tflops_sustained", peak)))

    # end to end: pinned host inputs -> heap, fused op, outputs -> pinned host,
    # every step.  Two problem instances alternate so that step i's uploads
    # (copy stream) overlap step i-1's kernel and step i-2's download, the
    # way a serving loop double-buffers its inputs.
    pin_A = [a.pin_memory() for a in x.A]
    pin_B = [b.pin_memory() for b in x.B]
    pin_bias = x.bias.pin_memory() if x.bias is not None else None
    prob2 = FusedProblem(wl["op"], wl["W"], wl["M"], wl["N"], wl["K"], wl["dtype"], bias=wl.get("bias", False),
                         config=cfg)
    probs = [prob, prob2]

    def out_views(p):
        return [p.heap.view(p.out, r) for r in range(wl["W"])] if wl["op"] == "mm_rs" else [p.heap.view(p.out, 0)]
    host_out = [[torch.empty(v.shape, dtype=v.dtype).pin_memory() for v in out_views(p)] for p in probs]
    h2d = prob.input_bytes()
    d2h = sum(v.numel() * v.element_size() for v in out_views(prob))
    up_s, down_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in probs]
    ev_run = [torch.cuda.Event() for _ in probs]
    ev_down = [torch.cuda.Event() for _ in probs]
    for e in ev_run + ev_down:
        e.record(stream)
    E = max(3, args.e2e_steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    for i in range(3 + E):
        if i == 3:
            torch.cuda.synchronize()
            e0.record(up_s)
        j = i % 2
        p = probs[j]
        up_s.wait_event(ev_run[j])            # the kernel that read these inputs is done
        with torch.cuda.stream(up_s):
            p.upload(pin_A, pin_B, pin_bias, non_blocking=True)
        ev_up[j].record(up_s)
        stream.wait_event(ev_up[j])
        stream.wait_event(ev_down[j])         # the previous download of this output is done
        p.run(stream)
        ev_run[j].record(stream)
        down_s.wait_event(ev_run[j])
        with torch.cuda.stream(down_s):
            for h, v in zip(host_out[j], out_views(p)):
                h.copy_(v, non_blocking=True)
        ev_down[j].record(down_s)
    e1.record(down_s)                         # after the last step's download
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / E, pg)
    e2e = {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
           "pipelining": "two buffers; uploads, kernel and downloads on three streams"}
    rc2 = query_status(prob2.ws, stream)
    if rc2[0] != 0:
        raise RuntimeError(f"device status after e2e steps: {rc2}")
    del prob2
    rc = query_status(prob.ws, stream)
    if rc[0] != 0:
        raise RuntimeError(f"device status after e2e steps: {rc}")

    lib_ref = library_reference(prob, wl, stream, flush)
    if rank != 0:
        return 0
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        del flush
        cpu = cpu_baseline(wl, x)
    base = pages_tflops(wl["op"], wl["W"], wl["M"], wl["N"], wl["K"])
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": (value / world / base) if base else None, "dtype": wl["dtype"], "data": "synthetic",
            "config": bench_config(wl, args.workload, cfg, world),
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": K,
            "clocks": clocks, "wall_s_timed_region": wall, "library_reference": lib_ref}
    if sus is not None:
        line["sustained"] = sus
    if others is not None:
        line["other_configs"] = others
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
