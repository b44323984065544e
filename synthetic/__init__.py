"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module draws random numbers and casts them to the storage dtype; it holds
none of the fused operations' arithmetic (no matmul, no sum, no gather).  Both
the CUDA path and the CPU oracle receive exactly the host tensors built here,
so they see identical input bits whatever the generator.

Generator: ``torch.Generator('cpu').manual_seed(seed)``.  Uniform values are
``rand * 2 - 1`` (scaled), normal values ``randn * sigma``; each is drawn in
fp32 and then rounded to the storage dtype (round-to-nearest-even, torch's
``Tensor.to``).  Draw order for a workload: for rank r = 0..W-1 its A_r, then
its B_r (ops with per-rank B), then the shared B, then the bias.

The workload shapes are the five benchmark configurations of the fused
all-gather/matmul family ("Fused Communication and Compute Operations" API
pages for the ops; the ROCm/iris PR #506 performance table for the 131072 x
16384 x 16384 and 4096 x 14336 x 4096 shapes; ROCm/iris PR #544 for the
concurrent GEMM + all-reduce mode).
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def _draw(gen: torch.Generator, shape, dist: str, scale: float, dtype: torch.dtype,
          chunk_rows: int = 16384) -> torch.Tensor:
    """Draw a tensor of ``shape`` from ``dist`` ('uniform' in [-scale, scale] or
    'normal' with std ``scale``) in fp32, then round to ``dtype``.

    Rows are drawn ``chunk_rows`` at a time (part of the recipe) so the fp32
    temporary stays small for the multi-GB shards.
    """
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=dtype)
    if len(shape) == 0 or out.numel() == 0:
        return out
    rows = shape[0]
    rest = shape[1:]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        sub = (r1 - r0,) + rest
        if dist == "uniform":
            x = torch.rand(sub, generator=gen, dtype=torch.float32) * (2.0 * scale) - scale
        elif dist == "normal":
            x = torch.randn(sub, generator=gen, dtype=torch.float32) * scale
        elif dist == "int":
            # small integers in [-scale, scale]: every product and every fp32
            # partial sum is exact for modest K, so results are order-independent
            x = torch.randint(-int(scale), int(scale) + 1, sub, generator=gen).to(torch.float32)
        else:
            raise ValueError(dist)
        out[r0:r1] = x.to(dtype)
    return out


@dataclasses.dataclass
class FusedInputs:
    """Host tensors of one fused-op workload.

    ``A``: list of W per-rank A tensors (shard or full, per op).
    ``B``: list of W per-rank B tensors (ops with per-rank B) or a one-element
    list holding the shared B.  ``bias``: 1-D tensor or None.
    """
    op: str
    W: int
    M: int
    N: int
    K: int
    dtype: str
    A: List[torch.Tensor]
    B: List[torch.Tensor]
    bias: Optional[torch.Tensor]


def a_shape(op: str, W: int, M: int, N: int, K: int):
    """Per-rank A shape for each op (row-major, K contiguous)."""
    if op == "ag_mm":          # A shard is M x K_local, K = W * K_local
        return (M, K // W)
    if op == "mm_ag":          # M is the gathered M; each rank holds M / W rows
        return (M // W, K)
    return (M, K)              # mm_rs, mm_ar: full per-rank A


def b_per_rank(op: str) -> bool:
    return op in ("mm_rs", "mm_ar")


def make_fused_inputs(op: str, W: int, M: int, N: int, K: int, dtype: str, seed: int,
                      dist: str = "uniform", scale: float = 1.0, bias: bool = False,
                      bias_scale: float = 0.1, bias_len: Optional[int] = None) -> FusedInputs:
    """Build the host inputs of one fused op.  ``op`` is one of ag_mm, mm_rs,
    mm_ag, mm_ar.  The draw order is A_r (and B_r for per-rank-B ops) for each
    rank in order, then the shared B, then the bias (uniform in
    [-bias_scale, bias_scale]).  ``bias_len`` defaults to N (a per-column bias)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    dt = DTYPES[dtype]
    As, Bs = [], []
    ash = a_shape(op, W, M, N, K)
    for _r in range(W):
        As.append(_draw(g, ash, dist, scale, dt))
        if b_per_rank(op):
            Bs.append(_draw(g, (K, N), dist, scale, dt))
    if not b_per_rank(op):
        Bs.append(_draw(g, (K, N), dist, scale, dt))
    b = None
    if bias:
        n = N if bias_len is None else int(bias_len)
        b = _draw(g, (n,), "uniform" if dist != "int" else "int",
                  bias_scale if dist != "int" else max(1.0, bias_scale), dt)
    return FusedInputs(op, W, M, N, K, dtype, As, Bs, b)


def make_gemm_inputs(M: int, N: int, K: int, dtype: str, seed: int, dist: str = "normal",
                     scale: float = 1.0):
    """A (M x K) and B (K x N) of an independent GEMM, drawn A then B."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    dt = DTYPES[dtype]
    return _draw(g, (M, K), dist, scale, dt), _draw(g, (K, N), dist, scale, dt)


def make_coll_inputs(W: int, count: int, dtype: str, seed: int, dist: str = "uniform",
                     scale: float = 1.0) -> List[torch.Tensor]:
    """W per-rank 1-D buffers of ``count`` elements, drawn rank by rank."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    dt = DTYPES[dtype]
    return [_draw(g, (count,), dist, scale, dt, chunk_rows=1 << 24) for _ in range(W)]


def sample_indices(rows: int, cols: int, seed: int, n: int = 4096, tile_m: int = 128,
                   tile_n: int = 256):
    """Seeded output sample: ``n`` random (i, j) pairs from
    ``Generator('cpu').manual_seed(seed)``, plus the four corners and the first
    and last row and column of tile (0, 0).  Returns two int64 tensors."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    ii = torch.randint(0, rows, (n,), generator=g, dtype=torch.int64)
    jj = torch.randint(0, cols, (n,), generator=g, dtype=torch.int64)
    extra_i, extra_j = [], []
    for (i, j) in [(0, 0), (0, cols - 1), (rows - 1, 0), (rows - 1, cols - 1)]:
        extra_i.append(i)
        extra_j.append(j)
    tm, tn = min(tile_m, rows), min(tile_n, cols)
    for j in range(tn):
        extra_i += [0, tm - 1]
        extra_j += [j, j]
    for i in range(tm):
        extra_i += [i, i]
        extra_j += [0, tn - 1]
    ii = torch.cat([ii, torch.tensor(extra_i, dtype=torch.int64)])
    jj = torch.cat([jj, torch.tensor(extra_j, dtype=torch.int64)])
    return ii, jj


# The five benchmark workloads.  Each entry gives the op, world size W, the
# global problem (M, N, K) in the op's own convention, dtype, seed and the
# value distribution.  "ag_mm": A gathered along K; "mm_rs": per-rank A_r, B_r,
# output split along N; "mm_ag": A_r has M/W rows, output gathered along M;
# "mm_ar": per-rank A_r, B_r, summed output; "concurrent": independent GEMM
# beside an all-reduce of W fp32 buffers.
WORKLOADS = {
    "ag_mm_w2_256": dict(op="ag_mm", W=2, M=256, N=256, K=256, dtype="f16", seed=0,
                         dist="uniform", scale=1.0, bias=False),
    "mm_rs_w4_4096": dict(op="mm_rs", W=4, M=4096, N=4096, K=4096, dtype="f16", seed=1,
                          dist="uniform", scale=1.0, bias=True, bias_scale=0.1),
    "ag_mm_w8_4096x14336x4096": dict(op="ag_mm", W=8, M=4096, N=14336, K=4096, dtype="bf16",
                                     seed=2, dist="normal", scale=0.02, bias=False),
    "mm_ag_w8_4096x14336x4096": dict(op="mm_ag", W=8, M=4096, N=14336, K=4096, dtype="bf16",
                                     seed=2, dist="normal", scale=0.02, bias=False),
    "ag_mm_w8_131072x16384x16384": dict(op="ag_mm", W=8, M=131072, N=16384, K=16384,
                                        dtype="bf16", seed=5, dist="normal", scale=0.02,
                                        bias=False),
    "mm_ar_w8_8192": dict(op="mm_ar", W=8, M=8192, N=8192, K=8192, dtype="bf16", seed=5,
                          dist="normal", scale=0.02, bias=False),
}

CONCURRENT_WORKLOAD = dict(M=8192, N=8192, K=8192, gemm_dtype="bf16", gemm_seed=3,
                           coll="all_reduce", W=8, count=64 * 1024 * 1024, coll_dtype="f32",
                           coll_seed=4)

# The world-size-8 all_gather_matmul shape list of the ROCm/iris PR #506
# performance table (label, M, N, K; bf16).  Timing workloads only: their
# inputs are drawn on the device by ``fill_device_`` and never reach the oracle.
AG_MM_SHAPES = [
    ("g2", 131072, 16384, 16384),
    ("g14", 147456, 28672, 4096),
    ("g15", 327680, 28672, 4096),
    ("g16", 229376, 28672, 4096),
    ("g5", 8192, 8192, 262144),
    ("g6", 262144, 8192, 8192),
    ("g1", 16384, 16384, 131072),
    ("g8", 262144, 28672, 8192),
    ("g9", 196608, 18432, 16384),
    ("mixtral_gate", 4096, 14336, 4096),
    ("llama7b_gate", 4096, 11008, 4096),
    ("pow2_4k", 4096, 4096, 4096),
]


def fill_device_(t: torch.Tensor, seed: int, dist: str = "normal", scale: float = 0.02) -> torch.Tensor:
    """Fill a device tensor in place from ``torch.Generator(device).manual_seed(seed)``
    ('normal' with std ``scale`` or 'uniform' in [-scale, scale]), drawn in
    the tensor's own dtype.  For multi-GB timing inputs that would take
    minutes to draw on the host; parity inputs use the host generators above."""
    g = torch.Generator(device=t.device).manual_seed(int(seed))
    if dist == "normal":
        return t.normal_(0.0, scale, generator=g)
    if dist == "uniform":
        return t.uniform_(-scale, scale, generator=g)
    raise ValueError(dist)
