"""Plain CPU definitions of the fused GEMM + collective operations.

Test infrastructure only (see the package docstring).  Inputs are CPU torch
tensors of fp16/bf16 (GEMM operands) or fp32 (collective buffers); 16-bit
outputs are returned as numpy ``uint16`` bit patterns, fp32 outputs as numpy
``float32`` arrays.

Notation follows the iris docs page "Fused Communication and Compute
Operations": W ranks, A (M x K), B (K x N), optional bias of length N (or M),
K_local = K / W for ``all_gather_matmul``, M_local = M / W for
``matmul_all_gather``, N_local = N / W for ``matmul_reduce_scatter``.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np
import torch

_BF16 = "bf16"
_F16 = "f16"


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def _as_f64(t) -> np.ndarray:
    """Exact decode of a 16/32-bit float tensor to float64."""
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def _dtype_name(t) -> str:
    if isinstance(t, torch.Tensor):
        if t.dtype == torch.bfloat16:
            return _BF16
        if t.dtype == torch.float16:
            return _F16
    raise TypeError("expected a bf16 or fp16 torch tensor")


def round_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 with IEEE 754 roundTiesToEven, as 16-bit patterns.

    bf16 keeps the top 16 bits of the fp32 encoding.  Adding 0x7FFF plus the
    lowest kept bit to the full 32-bit pattern and truncating rounds to the
    nearest representable value with ties to the even pattern; a carry out of
    the mantissa moves to the next binade (or to infinity) as it should.  NaN
    stays NaN (quiet bit set, sign kept).
    """
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)).astype(np.uint16)
    nan = np.isnan(x32)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x0040)).astype(np.uint16)
    return r


def round_f16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 with roundTiesToEven (numpy's IEEE conversion, which
    handles subnormals and overflow to infinity), as 16-bit patterns."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        return x32.astype(np.float16).view(np.uint16)


def round16(x32: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to the 16-bit output type; returns bit patterns."""
    if dtype == _BF16:
        return round_bf16_bits(x32)
    if dtype == _F16:
        return round_f16_bits(x32)
    raise ValueError(dtype)


def decode16(bits: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit patterns -> float64 values (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == _F16:
        return bits.view(np.float16).astype(np.float64)
    if dtype == _BF16:
        with np.errstate(invalid="ignore"):
            return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


# --------------------------------------------------------------------------
# GEMM building blocks
# --------------------------------------------------------------------------

def accumulate(X64: np.ndarray, Y64: np.ndarray) -> np.ndarray:
    """The fp32 accumulator of X @ Y: every dot product sum_k X[i,k] Y[k,j]
    summed in fp64 and rounded once to fp32."""
    return np.matmul(X64, Y64).astype(np.float32)


def _bias32(bias, bias_on_m: bool, rows: np.ndarray, cols: np.ndarray):
    """Bias values to add to the accumulator entries at (rows, cols) (fp32)."""
    if bias is None:
        return None
    b = _as_f64(bias).astype(np.float32)
    return b[rows] if bias_on_m else b[cols]


def _epilogue(acc32: np.ndarray, bias, bias_on_m: bool) -> np.ndarray:
    """acc + bias in fp32 (one IEEE add per element); bias indexed by column
    (length N) or, with ``bias_on_m``, by row (length M)."""
    if bias is None:
        return acc32
    b = _as_f64(bias).astype(np.float32)
    if bias_on_m:
        return (acc32 + b[:, None]).astype(np.float32)
    return (acc32 + b[None, :]).astype(np.float32)


def gather_k(A_shards: Sequence[torch.Tensor]) -> np.ndarray:
    """all_gather of the K-shards: G[i, s*K_local + k] = A_s[i, k], built by an
    explicit copy of each shard into its column block.  Returns float64."""
    W = len(A_shards)
    M, K_l = A_shards[0].shape
    G = np.empty((M, W * K_l), dtype=np.float64)
    for s in range(W):
        G[:, s * K_l:(s + 1) * K_l] = _as_f64(A_shards[s])
    return G


# --------------------------------------------------------------------------
# Fused ops ("Fused Communication and Compute Operations")
# --------------------------------------------------------------------------

def all_gather_matmul(A_shards: Sequence[torch.Tensor], B: torch.Tensor, bias=None,
                      bias_on_m: bool = False):
    """``all_gather_matmul``: output = all_gather(A_sharded) @ B + bias, A
    gathered along K.  Returns (out bits M x N, gathered bits M x K)."""
    dt = _dtype_name(B)
    G = gather_k(A_shards)
    acc = accumulate(G, _as_f64(B))
    out = round16(_epilogue(acc, bias, bias_on_m), dt)
    gathered = round16(G.astype(np.float32), dt)   # exact: G holds 16-bit values
    return out, gathered


def all_gather_matmul_at(A_shards, B, bias, ii, jj, bias_on_m: bool = False):
    """``all_gather_matmul`` output at the sampled positions (ii[t], jj[t])."""
    dt = _dtype_name(B)
    ii = np.asarray(ii, dtype=np.int64)
    jj = np.asarray(jj, dtype=np.int64)
    W = len(A_shards)
    K_l = A_shards[0].shape[1]
    out = np.empty(len(ii), dtype=np.uint16)
    step = 512
    for t0 in range(0, len(ii), step):
        r = ii[t0:t0 + step]
        c = jj[t0:t0 + step]
        G_rows = np.empty((len(r), W * K_l), dtype=np.float64)
        for s in range(W):
            G_rows[:, s * K_l:(s + 1) * K_l] = _as_f64(A_shards[s][torch.from_numpy(r)])
        B_cols = _as_f64(B[:, torch.from_numpy(c)])           # K x n
        acc = np.einsum("tk,kt->t", G_rows, B_cols).astype(np.float32)
        b = _bias32(bias, bias_on_m, r, c)
        if b is not None:
            acc = (acc + b).astype(np.float32)
        out[t0:t0 + step] = round16(acc, dt)
    return out


def matmul_all_gather(A_ranks: Sequence[torch.Tensor], B: torch.Tensor, bias=None,
                      bias_on_m: bool = False):
    """``matmul_all_gather``: output = all_gather(A @ B + bias) along M.  Rank r
    computes C_r = A_r @ B + bias (M_local x N, rounded to 16 bits) and the
    output stacks C_0..C_{W-1} along M.  A per-row bias has length M_local and
    is the same on every rank.  Returns bits (W*M_local) x N."""
    dt = _dtype_name(B)
    Bf = _as_f64(B)
    W = len(A_ranks)
    M_l = A_ranks[0].shape[0]
    out = np.empty((W * M_l, Bf.shape[1]), dtype=np.uint16)
    for r in range(W):
        acc = accumulate(_as_f64(A_ranks[r]), Bf)
        out[r * M_l:(r + 1) * M_l] = round16(_epilogue(acc, bias, bias_on_m), dt)
    return out


def matmul_all_gather_at(A_ranks, B, bias, ii, jj, bias_on_m: bool = False):
    """``matmul_all_gather`` output at sampled global positions (ii, jj)."""
    dt = _dtype_name(B)
    ii = np.asarray(ii, dtype=np.int64)
    jj = np.asarray(jj, dtype=np.int64)
    M_l = A_ranks[0].shape[0]
    out = np.empty(len(ii), dtype=np.uint16)
    for t in range(len(ii)):
        r, i = divmod(int(ii[t]), M_l)
        a = _as_f64(A_ranks[r][i])
        bcol = _as_f64(B[:, int(jj[t])])
        acc = np.float32(np.dot(a, bcol))
        if bias is not None:
            bv = _as_f64(bias).astype(np.float32)
            acc = np.float32(acc + (bv[i] if bias_on_m else bv[int(jj[t])]))
        out[t] = round16(np.array([acc], dtype=np.float32), dt)[0]
    return out


def partial(A_r: torch.Tensor, B_r: torch.Tensor, bias=None, bias_on_m: bool = False):
    """Rank r's fp32 partial product P_r = A_r @ B_r + bias (fp32)."""
    return _epilogue(accumulate(_as_f64(A_r), _as_f64(B_r)), bias, bias_on_m)


def rank_order_sum(parts: Sequence[np.ndarray]) -> np.ndarray:
    """S = (((P_0 + P_1) + P_2) + ...) in fp32, ranks in order 0..W-1."""
    S = np.array(parts[0], dtype=np.float32, copy=True)
    for p in parts[1:]:
        S = (S + np.asarray(p, dtype=np.float32)).astype(np.float32)
    return S


def _partials(A_ranks, B_ranks, bias, bias_on_m, round_partials, dt):
    parts = []
    for r in range(len(A_ranks)):
        p = partial(A_ranks[r], B_ranks[r], bias, bias_on_m)
        if round_partials:
            p = decode16(round16(p, dt), dt).astype(np.float32)
        parts.append(p)
    return parts


def matmul_reduce_scatter(A_ranks, B_ranks, bias=None, bias_on_m: bool = False,
                          round_partials: bool = False) -> List[np.ndarray]:
    """``matmul_reduce_scatter``: output = reduce_scatter(A @ B + bias) along N.
    Every rank adds the bias to its own partial (so the sum holds it W times);
    rank r receives the columns [r*N_local, (r+1)*N_local) of the rank-order
    fp32 sum, rounded to 16 bits.  ``round_partials`` rounds each partial to
    16 bits first (the alternative reading; not the default)."""
    dt = _dtype_name(B_ranks[0])
    W = len(A_ranks)
    S = rank_order_sum(_partials(A_ranks, B_ranks, bias, bias_on_m, round_partials, dt))
    N_l = S.shape[1] // W
    return [round16(np.ascontiguousarray(S[:, r * N_l:(r + 1) * N_l]), dt) for r in range(W)]


def _sum_at(A_ranks, B_ranks, bias, ii, jj, bias_on_m):
    """Rank-order fp32 sum of the partials at sampled (ii, jj) (global cols)."""
    ii = np.asarray(ii, dtype=np.int64)
    jj = np.asarray(jj, dtype=np.int64)
    S = None
    for r in range(len(A_ranks)):
        a_rows = _as_f64(A_ranks[r][torch.from_numpy(ii)])          # n x K
        b_cols = _as_f64(B_ranks[r][:, torch.from_numpy(jj)])       # K x n
        p = np.einsum("tk,kt->t", a_rows, b_cols).astype(np.float32)
        b = _bias32(bias, bias_on_m, ii, jj)
        if b is not None:
            p = (p + b).astype(np.float32)
        S = p if S is None else (S + p).astype(np.float32)
    return S


def matmul_reduce_scatter_at(A_ranks, B_ranks, bias, rank, ii, jj_local,
                             bias_on_m: bool = False):
    """Rank ``rank``'s ``matmul_reduce_scatter`` output at (ii, jj_local)."""
    dt = _dtype_name(B_ranks[0])
    N = B_ranks[0].shape[1]
    N_l = N // len(A_ranks)
    jj = np.asarray(jj_local, dtype=np.int64) + rank * N_l
    return round16(_sum_at(A_ranks, B_ranks, bias, ii, jj, bias_on_m), dt)


def matmul_all_reduce(A_ranks, B_ranks, bias=None, bias_on_m: bool = False,
                      round_partials: bool = False) -> np.ndarray:
    """``matmul_all_reduce``: output = all_reduce(A @ B + bias); every rank's
    copy is the rank-order fp32 sum of the W partials, rounded to 16 bits."""
    dt = _dtype_name(B_ranks[0])
    S = rank_order_sum(_partials(A_ranks, B_ranks, bias, bias_on_m, round_partials, dt))
    return round16(S, dt)


def matmul_all_reduce_at(A_ranks, B_ranks, bias, ii, jj, bias_on_m: bool = False):
    dt = _dtype_name(B_ranks[0])
    return round16(_sum_at(A_ranks, B_ranks, bias, ii, jj, bias_on_m), dt)


# --------------------------------------------------------------------------
# Concurrent mode (ROCm/iris PR #544): an independent GEMM and a collective
# (all_gather / all_reduce / reduce_scatter / all_to_all / broadcast)
# --------------------------------------------------------------------------

def gemm(A: torch.Tensor, B: torch.Tensor) -> np.ndarray:
    """The independent GEMM of the concurrent mode: C = A @ B, fp32
    accumulator rounded to the input's 16-bit type.  Returns bits."""
    return round16(accumulate(_as_f64(A), _as_f64(B)), _dtype_name(A))


def gemm_at(A, B, ii, jj) -> np.ndarray:
    ii = np.asarray(ii, dtype=np.int64)
    jj = np.asarray(jj, dtype=np.int64)
    a = _as_f64(A[torch.from_numpy(ii)])
    b = _as_f64(B[:, torch.from_numpy(jj)])
    return round16(np.einsum("tk,kt->t", a, b).astype(np.float32), _dtype_name(A))


def all_reduce(X: Sequence[torch.Tensor]) -> np.ndarray:
    """all_reduce of W fp32 buffers: every rank receives the rank-order fp32
    sum X_0 + X_1 + ... + X_{W-1}."""
    return rank_order_sum([_as_f64(x).astype(np.float32) for x in X])


def all_gather(X: Sequence[torch.Tensor]) -> np.ndarray:
    """all_gather of W buffers of ``count`` elements: every rank receives the
    concatenation X_0 | X_1 | ... | X_{W-1} (rank s at offset s*count).
    Returned as raw bytes of the element type."""
    parts = [x.detach().contiguous().view(torch.uint8).numpy() for x in X]
    out = np.empty(sum(p.size for p in parts), dtype=np.uint8)
    off = 0
    for p in parts:
        out[off:off + p.size] = p
        off += p.size
    return out


def all_to_all(X: Sequence[torch.Tensor]) -> List[np.ndarray]:
    """all_to_all of W buffers of ``count`` elements (count divisible by W):
    each buffer is W contiguous chunks; rank r receives chunk r of every rank,
    rank s's chunk at position s: out_r[s*c + i] = X_s[r*c + i].  Returned as
    raw bytes of the element type."""
    W = len(X)
    parts = [x.detach().contiguous().view(torch.uint8).numpy() for x in X]
    cb = parts[0].size // W
    outs = []
    for r in range(W):
        o = np.empty(W * cb, dtype=np.uint8)
        for s in range(W):
            o[s * cb:(s + 1) * cb] = parts[s][r * cb:(r + 1) * cb]
        outs.append(o)
    return outs


def broadcast(X: Sequence[torch.Tensor], root: int = 0) -> List[np.ndarray]:
    """broadcast of rank ``root``'s buffer: every rank receives a copy of it.
    Returned as raw bytes of the element type."""
    src = X[root].detach().contiguous().view(torch.uint8).numpy()
    return [src.copy() for _ in X]


def reduce_scatter(X: Sequence[torch.Tensor]) -> List[np.ndarray]:
    """reduce_scatter of W fp32 buffers of ``count`` elements: rank r receives
    the r-th of W contiguous chunks of the rank-order fp32 sum."""
    S = all_reduce(X)
    W = len(X)
    c = S.size // W
    return [S[r * c:(r + 1) * c].copy() for r in range(W)]
