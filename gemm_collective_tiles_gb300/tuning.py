"""Config selection for the fused ops: explicit config, else a measured
winner cached in a JSON file, else the measured winner of the nearest cached
shape, else the library's static default.

The shape of this subsystem follows ROCm/iris PR #544 ("Add iris.concurrent",
the autotune commit) and PR #506 (auto-config selection): candidates are ranked,
the top ones are benchmarked together with the static default, and the winner
is cached per (architecture, op, world size, shape, dtype -- and for the
concurrent mode the collective, its element count and type).  Because the
default is always measured, tuning never ends worse than the default.  A
shape with no entry of its own takes the winner of the nearest cached shape
of the same op, world size and types (PR #506, nearest-shape matching), but
only a winner that beat its own default, and only within a bounded distance
in log-space.  The cache is written atomically (a per-process temporary file,
then a rename).  The MI300X tables and rules on those pages do not carry
over; every value here is measured on the running GPU.
"""
from __future__ import annotations

import json
import math
import os
from typing import Callable, Dict, Iterable, List, Optional, Sequence

ENV_CACHE = "IRIS_B200_CACHE"

# knobs a cached entry may set (the rest stay at their defaults)
TUNABLE = ("tile_m", "tile_n", "group_m", "gemm_ctas", "reduce_mode", "rank_inner", "comm_block", "stages",
           "coll_ring", "coll_l2_hint", "coll_path", "gather_parts",
           "startup_gather", "gemm_l2_hint", "out_l2_hint",
           "sum_l2_hint", "k_split", "coll_out_stage")

# nearest-shape matching: largest accepted distance, in log2 units over the
# problem sizes (1.0 = one size off by a factor of 2, or two by 2^0.7 each)
NEAREST_MAX_DIST = 1.0


def cache_path() -> str:
    p = os.environ.get(ENV_CACHE)
    if p:
        return p
    return os.path.join(os.path.expanduser("~"), ".cache", "gemm_collective_tiles", "tuning.json")


def arch_key(device_name: str, sm_count: int, capability=(10, 3)) -> str:
    """Stable cache key of the device: name, compute capability, SM count."""
    return f"{device_name.strip()}|sm_{capability[0]}{capability[1]}|{int(sm_count)}sm"


def shape_key(op: str, W: int, M: int, N: int, K: int, dtype: str, coll: Optional[str] = None,
              count: int = 0, coll_dtype: str = "f32") -> str:
    """Cache key of one problem.  The concurrent mode's key also names the
    collective, its per-rank element count and element type: an all-reduce of
    64Mi elements and an all-gather of 1Mi want different splits."""
    k = f"{op}|W{int(W)}|{int(M)}x{int(N)}x{int(K)}|{dtype}"
    if op == "concurrent":
        k += f"|{coll or 'none'}|count{int(count)}|{coll_dtype}"
    return k


def shape_info(op: str, W: int, M: int, N: int, K: int, dtype: str, coll: Optional[str] = None,
               count: int = 0, coll_dtype: str = "f32") -> dict:
    """The fields of a problem that nearest-shape matching compares."""
    d = {"op": op, "W": int(W), "M": int(M), "N": int(N), "K": int(K), "dtype": dtype}
    if op == "concurrent":
        d.update(coll=coll or "none", count=int(count), coll_dtype=coll_dtype)
    return d


def shape_distance(a: dict, b: dict) -> Optional[float]:
    """Euclidean distance in log2 space over the sizes (M, N, K and, for the
    concurrent mode, count) of two problems of the same op, world size and
    types; None when they are not comparable."""
    for f in ("op", "W", "dtype", "coll", "coll_dtype"):
        if a.get(f) != b.get(f):
            return None
    d2 = 0.0
    for f in ("M", "N", "K", "count"):
        x, y = a.get(f, 0), b.get(f, 0)
        if (x > 0) != (y > 0):
            return None
        if x > 0:
            d2 += math.log2(x / y) ** 2
    return math.sqrt(d2)


def load_db(path: Optional[str] = None) -> Dict[str, Dict[str, dict]]:
    path = path or cache_path()
    try:
        with open(path) as f:
            db = json.load(f)
        return db if isinstance(db, dict) else {}
    except (OSError, ValueError):
        return {}


def save_db(db: Dict[str, Dict[str, dict]], path: Optional[str] = None) -> bool:
    """Atomic write: a per-process temporary file renamed over the cache, so a
    concurrent reader sees the old or the new file, never a torn one."""
    path = path or cache_path()
    try:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        tmp = f"{path}.{os.getpid()}.tmp"
        with open(tmp, "w") as f:
            json.dump(db, f, indent=1, sort_keys=True)
        os.replace(tmp, path)
        return True
    except OSError:
        return False


def lookup(arch: str, key: str, path: Optional[str] = None) -> Optional[dict]:
    entry = load_db(path).get(arch, {}).get(key)
    if not entry:
        return None
    return {k: v for k, v in entry.get("config", {}).items() if k in TUNABLE}


def record(arch: str, key: str, config: dict, ms: float, default_ms: float, path: Optional[str] = None,
           shape: Optional[dict] = None) -> bool:
    db = load_db(path)
    entry = {"config": {k: v for k, v in config.items() if k in TUNABLE}, "ms": ms, "default_ms": default_ms}
    if shape:
        entry["shape"] = shape
    db.setdefault(arch, {})[key] = entry
    return save_db(db, path)


def lookup_nearest(arch: str, shape: dict, path: Optional[str] = None,
                   max_dist: float = NEAREST_MAX_DIST) -> Optional[dict]:
    """The cached winner of the nearest comparable shape within max_dist,
    among entries whose winner beat their own static default (an entry
    whose best was the default carries no information for other shapes)."""
    best, best_d = None, None
    for entry in load_db(path).get(arch, {}).values():
        other = entry.get("shape")
        if not isinstance(other, dict):
            continue
        d = shape_distance(shape, other)
        if d is None or d > max_dist:
            continue
        ms, dms = entry.get("ms"), entry.get("default_ms")
        if ms is None or dms is None or not ms < dms or not entry.get("config"):
            continue
        if best_d is None or d < best_d:
            best, best_d = entry, d
    if best is None:
        return None
    return {k: v for k, v in best["config"].items() if k in TUNABLE}


def candidates(op: str, W: int, M: int, N: int, K: int, sm_count: int, top_k: int = 8,
               coll: str = "all_reduce", count: int = 0) -> List[dict]:
    """Ranked candidate configs (the static default, {}, is always first).

    Ranking rule (from the measurements behind the defaults): the swizzle
    group width matters most for operand reuse in L2, then one CTA per tile
    instead of a CTA pair where the pair tiles leave a wave badly filled,
    then the tile width for small N, then -- per op -- the reduce schedule or
    the concurrent CTA split.  The list is truncated to top_k."""
    out: List[dict] = [{}]
    # the CTA-pair pipeline the default does not pick for this K (three
    # 128-deep stages up to K = 98304, six 64-deep stages beyond)
    # (a split all_gather_matmul picks it by the K of one chunk)
    splits = op in ("all_gather_matmul", "matmul_reduce_scatter", "matmul_all_reduce",
                    "matmul_all_gather") and N % 32 == 0
    k_item = 16384 if (splits and K > 32768) else K
    out.append({"stages": 3 if k_item > 98304 else 6})
    # the swizzle widths the default does not use (32; 16 in the concurrent
    # mode and for the reduce ops when a rank's A exceeds 64 MB)
    reduce = op in ("matmul_reduce_scatter", "matmul_all_reduce")
    default_gm = 16 if op == "concurrent" or (reduce and M * K * 2 > (64 << 20)) else 32
    for gm in (64, 32, 16, 8):
        if gm != default_gm:
            out.append({"group_m": gm})
    pair_tiles = -(-M // 256) * -(-N // 256) * (W if op in ("matmul_reduce_scatter", "matmul_all_reduce") else 1)
    pairs = max(1, sm_count // 2)
    if pair_tiles % pairs and pair_tiles % pairs <= pairs // 2 or pair_tiles < pairs:
        out.insert(1, {"tile_m": 128})   # a short last wave of pair tiles
    else:
        out.append({"tile_m": 128})
    if N <= 4096:
        out.append({"tile_n": 128})
    if op in ("matmul_reduce_scatter", "matmul_all_reduce"):
        out += [{"reduce_mode": 2}, {"reduce_mode": 1}, {"group_m": 64, "reduce_mode": 3}]
    if splits and K > 16384:
        # split-K: the default splits above K = 32768 into chunks of ~16384
        out.insert(1, {"k_split": 1} if K > 32768 else {"k_split": 2})
    if op == "all_gather_matmul" and M <= 16384 and k_item <= 32768:
        # the default lets the TMA producer copy the start-up gathers up to
        # 16384 rows when an item's K is at most 32768 (0.4-2.4 % faster than
        # the worker threads on the PR #506 shapes of that size); the workers
        # remain the alternative
        out.insert(min(3, len(out)), {"startup_gather": 1})
    if op == "concurrent":
        if count > 0:
            # (tile, split) pairs ranked by the work-stealing makespan model
            return concurrent_candidates(M, N, K, coll, W, count, sm_count, top_k)
        else:
            for frac in (0.65, 0.55, 0.75, 0.45, 0.85):
                out.append({"gemm_ctas": max(1, int(round(frac * sm_count)))})
    # drop duplicates, keep order
    seen, uniq = set(), []
    for c in out:
        k = json.dumps(c, sort_keys=True)
        if k not in seen:
            seen.add(k)
            uniq.append(c)
    return uniq[:max(1, top_k)]


def tune(measure: Callable[[dict], float], cands: Sequence[dict], arch: str, key: str,
         path: Optional[str] = None, shape: Optional[dict] = None) -> dict:
    """Benchmark every candidate with ``measure(config) -> ms`` (the static
    default {} is added if missing), cache and return the fastest.  A
    candidate the library rejects (``measure`` raises) is skipped."""
    cands = list(cands)
    if {} not in cands:
        cands.insert(0, {})
    results = []
    default_ms = None
    for c in cands:
        try:
            ms = float(measure(dict(c)))
        except Exception:  # noqa: BLE001 -- an invalid candidate for this shape
            continue
        results.append((ms, c))
        if c == {}:
            default_ms = ms
    if not results:
        raise RuntimeError("no candidate config could run")
    best_ms, best = min(results, key=lambda t: t[0])
    if default_ms is not None and best_ms > default_ms:   # cannot happen; kept explicit
        best_ms, best = default_ms, {}
    record(arch, key, best, best_ms, default_ms if default_ms is not None else best_ms, path, shape)
    return {"config": best, "ms": best_ms, "default_ms": default_ms, "tried": len(results),
            "results": [{"config": c, "ms": ms} for ms, c in results]}


def select(arch: str, key: str, explicit: Optional[dict] = None, path: Optional[str] = None,
           shape: Optional[dict] = None) -> dict:
    """Explicit config, else the cached winner of this exact key, else (with
    `shape`) the winner of the nearest cached shape, else {} (the static
    default)."""
    if explicit:
        return dict(explicit)
    hit = lookup(arch, key, path)
    if hit is not None:
        return hit
    if shape is not None:
        near = lookup_nearest(arch, shape, path)
        if near is not None:
            return near
    return {}


def device_arch() -> str:
    import torch
    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    return arch_key(props.name, props.multi_processor_count, (props.major, props.minor))


def tune_fused(op: str, W: int, M: int, N: int, K: int, dtype: str, seed: int = 0, top_k: int = 8,
               reps: int = 10, path: Optional[str] = None) -> dict:
    """Measure the candidates of a fused op (runner.FusedProblem) on the
    current GPU with CUDA events and cache the winner."""
    import torch

    from .runner import FusedProblem
    short = {"all_gather_matmul": "ag_mm", "matmul_reduce_scatter": "mm_rs",
             "matmul_all_gather": "mm_ag", "matmul_all_reduce": "mm_ar"}[op]
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count

    def measure(cfg):
        prob = FusedProblem(short, W, M, N, K, dtype, config=cfg)
        for r in range(W):
            prob.heap.view(prob.A, r).normal_(0, 0.02)
            prob.heap.view(prob.B, r if prob.per_rank_b() else 0).normal_(0, 0.02)
        for _ in range(2):
            prob.run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            prob.run()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    return tune(measure, candidates(op, W, M, N, K, sms, top_k), device_arch(),
                shape_key(op, W, M, N, K, dtype), path, shape_info(op, W, M, N, K, dtype))


def concurrent_candidates(M: int, N: int, K: int, coll: str, W: int, count: int, sm_count: int,
                          top_k: int = 6, elem_bytes: int = 4, comm_block: int = 131072) -> List[dict]:
    """Ranked candidate configs of the concurrent mode: the static default
    first, then the default split with half and with 1.5x its collective
    items (the item size moved the step time by 2-8 % beside every
    collective), then the predictor's joint ranking of (tile kind,
    gemm_ctas)."""
    from . import predictor
    out: List[dict] = [{}]
    if count > 0 and M > 0 and N > 0:
        # collective items of other sizes, where the collective has items to spare
        if count >= 8 * comm_block:
            out += [{"comm_block": comm_block // 2}, {"comm_block": comm_block * 3 // 2}]
        wl = predictor.Workload(M=M, N=N, K=K, coll=coll, W=W, count=count, elem_bytes=elem_bytes,
                                comm_block=comm_block)
        for d in predictor.predict_split(wl, m=predictor.Machine(sms=sm_count), top_k=4 * top_k,
                                         tiles=predictor.TILE_KINDS):
            out.append(dict(d["config"]))
    seen, uniq = set(), []
    for c in out:
        k = json.dumps(c, sort_keys=True)
        if k not in seen:
            seen.add(k)
            uniq.append(c)
    return uniq[:max(1, top_k)]


def tune_concurrent(M: int, N: int, K: int, gemm_dtype: str, coll: str, W: int, count: int,
                    coll_dtype: str = "f32", top_k: int = 6, reps: int = 10, seed: int = 0,
                    path: Optional[str] = None) -> dict:
    """Measure the concurrent mode's candidates (runner.ConcurrentProblem:
    the GEMM and the collective in one launch) on the current GPU with CUDA
    events, the static default included, and cache the winner under the
    concurrent key."""
    import torch

    from .runner import ConcurrentProblem
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    esz = 4 if coll_dtype == "f32" else 2

    def measure(cfg):
        prob = ConcurrentProblem(M, N, K, gemm_dtype, coll, W, count, coll_dtype=coll_dtype, config=cfg or None)
        g = torch.Generator(device="cuda").manual_seed(seed)
        if prob.has_gemm:
            prob.A.normal_(0, 1, generator=g)
            prob.B.normal_(0, 1, generator=g)
        if count > 0:
            for r in range(W):
                prob.heap.view(prob.x_in, r).uniform_(-1, 1, generator=g)
        for _ in range(2):
            prob.run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            prob.run()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    cands = concurrent_candidates(M, N, K, coll, W, count, sms, top_k, esz)
    return tune(measure, cands, device_arch(),
                shape_key("concurrent", W, M, N, K, gemm_dtype, coll, count, coll_dtype), path,
                shape_info("concurrent", W, M, N, K, gemm_dtype, coll, count, coll_dtype))
