"""Analytical split predictor for the concurrent GEMM + collective mode.

ROCm/iris PR #544 ranks GEMM/comm work-group splits with a cost model and a
work-stealing makespan simulator before benchmarking the best few.  This is a
GB300 version written from that description: a per-tile cost model
(tensor-core rate per SM for GEMM tiles; per-SM copy bandwidth, capped by the
shared HBM bandwidth, for collective tiles) and a discrete-event simulation of
the persistent kernel's two queues with spill-over (a CTA whose preferred
queue is empty takes from the other).  All-reduce tiles read and write every
rank (2W transfers per tile), so they need the most CTAs to saturate memory;
the other collectives move fewer bytes per tile.

Constants are calibrated on GB300 measurements of this library (the GEMM and
the all-reduce of the concurrent path, each timed alone on 38 to 152 CTAs,
and the GEMM's DRAM bytes under ncu); they can be replaced by the caller.

The GEMM tile is ranked together with the split (PR #544 review excerpt of
predict_split: tile candidates, a preferred tile and a margin): each tile
kind of this library -- 256 x 256 tiles on CTA pairs with the six- or the
three-stage pipeline, or 128 x 256 tiles on one CTA -- has its own measured
per-CTA rate and its own cost for lending the pipeline stages to a
collective tile, and a tile other than the preferred one ranks above it only
when its predicted makespan is shorter by more than the margin.
"""
from __future__ import annotations

import dataclasses
import heapq
import math
from typing import Dict, List, Optional, Sequence


@dataclasses.dataclass
class Machine:
    sms: int = 152
    gemm_tflops_per_sm: float = 11.91     # CTA-pair GEMM 8192^3 bf16 (three-stage pipeline) over 152 SMs
    comm_gbs_per_sm: float = 78.0         # one CTA's collective engine, reads + writes (all-reduce, one box
                                          # of all sources per sub-chunk, on 38 CTAs)
    hbm_gbs: float = 6100.0               # reads + writes the all-reduce reaches alone on every SM
    gemm_hbm_share: float = 0.12          # HBM fraction the GEMM operands use when all SMs run it
    gemm_dram_bytes_per_flop: float = 1.27e-3  # the GEMM's DRAM reads per flop (8192^3 alone: 1.4 GB)
    tile_overhead_us: float = 1.0         # claim + pipeline fill per tile


@dataclasses.dataclass
class TileKind:
    """One GEMM tile / pipeline of the kernel, with its measured rate."""
    name: str
    tile_m: int                  # rows of one tile
    tile_n: int
    ctas: int                    # CTAs that compute one tile together (2 = a CTA pair)
    gemm_tflops_per_cta: float   # GEMM rate per CTA with every SM on the GEMM
    lease_us: float              # pipeline drain before a collective tile borrows the stages
    config: Dict[str, int]       # the iris_b200_config fields that select it


# Per-CTA rates measured on GB300 (bf16 8192^3 GEMM alone on 152 SMs:
# 0.640 ms six-stage pairs, 0.607 ms three-stage pairs, 0.694 ms one CTA per
# tile).  The lease cost is the pipeline's drain: the stages' bytes (192 KB
# either way) consumed at the tile's rate, about a third longer for the
# three-stage pipeline's deeper stages.
TILE_KINDS = (
    TileKind("pair6", 256, 256, 2, 11.30, 1.0, {"tile_m": 256, "stages": 6}),
    TileKind("pair3", 256, 256, 2, 11.91, 1.33, {"tile_m": 256, "stages": 3}),
    TileKind("cta128", 128, 256, 1, 10.43, 1.0, {"tile_m": 128}),
)
PREFERRED_TILE = "pair3"   # the library's default, beside a collective too


@dataclasses.dataclass
class Workload:
    M: int
    N: int
    K: int
    coll: str = "all_reduce"
    W: int = 8
    count: int = 64 * 1024 * 1024
    elem_bytes: int = 4
    tile_m: int = 128
    tile_n: int = 256
    comm_block: int = 131072

    def gemm_tiles(self) -> int:
        return math.ceil(self.M / self.tile_m) * math.ceil(self.N / self.tile_n)

    def gemm_tile_flops(self) -> float:
        return 2.0 * self.tile_m * self.tile_n * self.K

    def comm_tiles(self) -> int:
        chunks = math.ceil(self.count / self.comm_block)
        if self.coll == "all_gather":
            return chunks * self.W
        if self.coll == "all_to_all":
            return self.W * self.W * math.ceil(self.count / self.W / self.comm_block)
        return chunks

    def comm_tile_bytes(self) -> float:
        """Bytes one collective tile moves (reads + writes)."""
        e = self.elem_bytes
        if self.coll == "all_reduce":
            return 2.0 * self.W * self.comm_block * e          # read W, write W
        if self.coll == "reduce_scatter":
            return (self.W + 1.0) * self.comm_block * e        # read W, write 1
        if self.coll in ("all_gather", "broadcast"):
            return (1.0 + self.W) * self.comm_block * e        # read 1, write W
        return 2.0 * min(self.comm_block, self.count / self.W) * e  # all_to_all: one peer


def comm_floor(coll: str, base: int = 8, sms: int = 152) -> int:
    """Fewest CTAs worth giving the collective: an all-reduce tile does 2W
    transfers, the heaviest per tile, so it gets twice the base floor; the
    lighter collectives get no floor."""
    if coll == "all_reduce":
        return max(1, min(2 * base, sms))
    return 1


def simulate(wl: Workload, gemm_ctas: int, m: Optional[Machine] = None, tile: Optional[TileKind] = None) -> float:
    """Makespan (microseconds) of one launch with `gemm_ctas` CTAs preferring
    the GEMM queue and the rest the comm queue, both spilling when dry.

    Without `tile`, every CTA is a worker with the workload's tile at the
    machine's per-SM rate.  With a TileKind, the workers are its units (a CTA
    pair computes one tile and runs each collective tile on both CTAs), a
    unit prefers the GEMM when its first CTA is below gemm_ctas, and a unit
    that turns from GEMM to collective work first drains its pipeline.

    Both jobs draw on HBM: a collective tile moves its bytes at its engine's
    rate, capped by the bandwidth the GEMM leaves; a GEMM tile takes the
    longer of its tensor time and the time to read its DRAM bytes from what
    the running collective tiles leave, shared by the running GEMM tiles."""
    m = m or Machine()
    ctas = tile.ctas if tile else 1
    units = max(1, m.sms // ctas)
    gemm_ctas = max(0, min(m.sms, gemm_ctas))
    if tile:
        tiles = math.ceil(wl.M / tile.tile_m) * math.ceil(wl.N / tile.tile_n) if wl.M and wl.N else 0
        tile_flops = 2.0 * tile.tile_m * tile.tile_n * wl.K
        t_flop = tile_flops / (tile.gemm_tflops_per_cta * ctas * 1e12) * 1e6
        lease = tile.lease_us
    else:
        tiles = wl.gemm_tiles() if wl.M and wl.N else 0
        tile_flops = wl.gemm_tile_flops()
        t_flop = tile_flops / (m.gemm_tflops_per_sm * 1e12) * 1e6
        lease = 0.0
    tile_dram = tile_flops * m.gemm_dram_bytes_per_flop
    n_g, n_c = tiles, wl.comm_tiles()
    bytes_c = wl.comm_tile_bytes()
    # event queue of (time free, unit); greedy claims in time order
    free = [(0.0, u) for u in range(units)]
    heapq.heapify(free)
    last_gemm = [False] * units
    g_next = c_next = 0
    active_comm: List[float] = []   # end times of collective tiles in flight
    active_gemm: List[float] = []   # end times of GEMM tiles in flight
    end = 0.0
    while g_next < n_g or c_next < n_c:
        t, u = heapq.heappop(free)
        active_comm = [x for x in active_comm if x > t]
        active_gemm = [x for x in active_gemm if x > t]
        prefer_gemm = u * ctas < gemm_ctas
        take_gemm = (prefer_gemm and g_next < n_g) or (not prefer_gemm and c_next >= n_c)
        if take_gemm:
            g_next += 1
            comm_demand = len(active_comm) * m.comm_gbs_per_sm * ctas
            bw = max(1.0, (m.hbm_gbs - min(comm_demand, 0.9 * m.hbm_gbs)) / (len(active_gemm) + 1))
            done = t + max(t_flop, tile_dram / (bw * 1e9) * 1e6) + m.tile_overhead_us
            active_gemm.append(done)
        else:
            c_next += 1
            running = len(active_comm) + 1
            gemm_running = min(len(active_gemm), units - running) if g_next < n_g else len(active_gemm)
            hbm_left = m.hbm_gbs * (1.0 - m.gemm_hbm_share * gemm_running / units)
            bw = min(m.comm_gbs_per_sm * ctas, hbm_left / running)
            done = t + bytes_c / (bw * 1e9) * 1e6 + m.tile_overhead_us + (lease if last_gemm[u] else 0.0)
            active_comm.append(done)
        last_gemm[u] = take_gemm
        end = max(end, done)
        heapq.heappush(free, (done, u))
    return end


def predict_split(wl: Workload, candidates: Optional[Sequence[int]] = None, m: Optional[Machine] = None,
                  top_k: int = 4, tiles: Optional[Sequence[TileKind]] = None, prefer: str = PREFERRED_TILE,
                  margin: float = 0.20) -> List[Dict[str, object]]:
    """Rank GEMM/comm CTA splits by simulated makespan; the collective keeps
    at least comm_floor() CTAs.  Returns the top_k as dicts with "gemm_ctas"
    and "us".

    With `tiles`, each (tile kind, split) pair is simulated and ranked
    jointly; a tile other than `prefer` counts as if its makespan were
    1 / (1 - margin) times longer, so it wins only when it is faster by more
    than the margin.  Those dicts also hold "tile" (the kind's name), "key"
    (the ranking value) and "config" (the iris_b200_config fields)."""
    m = m or Machine()
    floor = comm_floor(wl.coll, sms=m.sms)
    if candidates is None:
        candidates = sorted({max(1, int(round(f * m.sms))) for f in
                             (0.25, 0.35, 0.45, 0.5, 0.55, 0.6, 0.65, 0.7, 0.75, 0.85, 0.9)})
    ranked = []
    for g in candidates:
        if wl.comm_tiles() > 0 and m.sms - g < floor:
            continue
        if tiles is None:
            ranked.append({"gemm_ctas": int(g), "us": simulate(wl, g, m)})
            continue
        for tk in tiles:
            us = simulate(wl, g, m, tk)
            key = us if tk.name == prefer else us / (1.0 - margin)
            ranked.append({"gemm_ctas": int(g), "us": us, "tile": tk.name, "key": key,
                           "config": {**tk.config, "gemm_ctas": int(g)}})
    ranked.sort(key=lambda d: d.get("key", d["us"]))
    return ranked[:max(1, top_k)]


def sequential_us(wl: Workload, m: Optional[Machine] = None) -> float:
    """GEMM alone on every SM, then the collective alone on every SM."""
    m = m or Machine()
    g = Workload(**{**dataclasses.asdict(wl), "count": 0})
    c = Workload(**{**dataclasses.asdict(wl), "M": 0, "N": 0})
    return simulate(g, m.sms, m) + simulate(c, 0, m)
