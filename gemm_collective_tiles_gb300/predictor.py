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
the all-reduce of the concurrent path, each timed alone on 8 to 152 CTAs);
they can be replaced by the caller.
"""
from __future__ import annotations

import dataclasses
import heapq
import math
from typing import Dict, List, Optional, Sequence


@dataclasses.dataclass
class Machine:
    sms: int = 152
    gemm_tflops_per_sm: float = 11.9      # CTA-pair GEMM 8192^3 bf16 at 1.81 PFLOP/s over 152 SMs
    comm_gbs_per_sm: float = 65.0         # one CTA's collective engine (all-reduce, linear up to ~96 CTAs)
    hbm_gbs: float = 6779.4               # measured copy bandwidth
    gemm_hbm_share: float = 0.12          # HBM fraction the GEMM operands use when all SMs run it
    tile_overhead_us: float = 1.0         # claim + pipeline fill per tile


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
    comm_block: int = 65536

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


def simulate(wl: Workload, gemm_ctas: int, m: Optional[Machine] = None) -> float:
    """Makespan (microseconds) of one launch with `gemm_ctas` CTAs preferring
    the GEMM queue and the rest the comm queue, both spilling when dry."""
    m = m or Machine()
    grid = m.sms
    gemm_ctas = max(0, min(grid, gemm_ctas))
    n_g, n_c = wl.gemm_tiles(), wl.comm_tiles()
    t_gemm = wl.gemm_tile_flops() / (m.gemm_tflops_per_sm * 1e12) * 1e6 + m.tile_overhead_us
    bytes_c = wl.comm_tile_bytes()
    # event queue of (time free, cta); greedy claims in time order
    free = [(0.0, c) for c in range(grid)]
    heapq.heapify(free)
    g_next = c_next = 0
    active_comm: List[float] = []   # end times of collective tiles in flight
    end = 0.0
    while g_next < n_g or c_next < n_c:
        t, cta = heapq.heappop(free)
        prefer_gemm = cta < gemm_ctas
        take_gemm = (prefer_gemm and g_next < n_g) or (not prefer_gemm and c_next >= n_c)
        if take_gemm:
            g_next += 1
            done = t + t_gemm
        else:
            c_next += 1
            active_comm = [x for x in active_comm if x > t]
            running = len(active_comm) + 1
            gemm_running = min(gemm_ctas, grid - running) if g_next < n_g else 0
            hbm_left = m.hbm_gbs * (1.0 - m.gemm_hbm_share * gemm_running / grid)
            bw = min(m.comm_gbs_per_sm, hbm_left / running)
            done = t + bytes_c / (bw * 1e9) * 1e6 + m.tile_overhead_us
            active_comm.append(done)
        end = max(end, done)
        heapq.heappush(free, (done, cta))
    return end


def predict_split(wl: Workload, candidates: Optional[Sequence[int]] = None, m: Optional[Machine] = None,
                  top_k: int = 4) -> List[Dict[str, float]]:
    """Rank GEMM/comm CTA splits by simulated makespan; the collective keeps
    at least comm_floor() CTAs.  Returns the top_k as dicts."""
    m = m or Machine()
    floor = comm_floor(wl.coll, sms=m.sms)
    if candidates is None:
        candidates = sorted({max(1, int(round(f * m.sms))) for f in
                             (0.25, 0.35, 0.45, 0.5, 0.55, 0.6, 0.65, 0.75, 0.85, 0.9)})
    ranked = []
    for g in candidates:
        if wl.comm_tiles() > 0 and m.sms - g < floor:
            continue
        ranked.append({"gemm_ctas": int(g), "us": simulate(wl, g, m)})
    ranked.sort(key=lambda d: d["us"])
    return ranked[:max(1, top_k)]


def sequential_us(wl: Workload, m: Optional[Machine] = None) -> float:
    """GEMM alone on every SM, then the collective alone on every SM."""
    m = m or Machine()
    g = Workload(**{**dataclasses.asdict(wl), "count": 0})
    c = Workload(**{**dataclasses.asdict(wl), "M": 0, "N": 0})
    return simulate(g, m.sms, m) + simulate(c, 0, m)
