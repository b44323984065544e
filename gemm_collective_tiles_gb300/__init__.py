"""GB300 (sm_103a) fused GEMM + collective tiles.

Python face of the C ABI in ``include/gemm_collective_tiles.h``.  PyTorch is
used only to allocate device memory (the emulated symmetric heap and the
workspace) and to name the CUDA stream; every step of every op runs in the
library's own kernels.

Ops (iris docs "Fused Communication and Compute Operations"; ROCm/iris PR #544
"Add iris.concurrent"):

* ``all_gather_matmul``      out = all_gather(A_sharded along K) @ B + bias
* ``matmul_reduce_scatter``  out_r = reduce_scatter(A @ B + bias) along N
* ``matmul_all_gather``      out = all_gather(A @ B + bias) along M
* ``matmul_all_reduce``      out = all_reduce(A @ B + bias)
* ``concurrent_gemm_collective``  independent GEMM beside an all-gather /
  all-reduce / reduce-scatter, with an explicit GEMM/comm CTA split.

The W ranks live in W regions of one device allocation (``SymmetricHeap``);
a ``HeapTensor`` names the same byte offset in every region.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
from typing import Optional, Sequence

import torch

from . import _native
from ._native import (  # noqa: F401  (same-name C ABI wrappers)
    IrisError,
    iris_b200_all_gather_matmul,
    iris_b200_concurrent_gemm_collective,
    iris_b200_config,
    iris_b200_heap,
    iris_b200_matmul_all_gather,
    iris_b200_matmul_all_reduce,
    iris_b200_matmul_reduce_scatter,
    iris_b200_num_sms,
    iris_b200_query_status,
    iris_b200_strerror,
    iris_b200_workspace_size,
)

__all__ = [
    "SymmetricHeap", "HeapTensor", "Workspace", "make_config", "workspace_size",
    "all_gather_matmul", "matmul_reduce_scatter", "matmul_all_gather", "matmul_all_reduce",
    "concurrent_gemm_collective", "concurrent_two_stream", "query_status", "num_sms", "IrisError",
]

_DT = {torch.float16: _native.IRIS_F16, torch.bfloat16: _native.IRIS_BF16,
       torch.float32: _native.IRIS_F32}
_OPS = {
    "all_gather_matmul": _native.IRIS_OP_ALL_GATHER_MATMUL,
    "matmul_reduce_scatter": _native.IRIS_OP_MATMUL_REDUCE_SCATTER,
    "matmul_all_gather": _native.IRIS_OP_MATMUL_ALL_GATHER,
    "matmul_all_reduce": _native.IRIS_OP_MATMUL_ALL_REDUCE,
    "concurrent": _native.IRIS_OP_CONCURRENT,
}
_COLL = {"all_gather": _native.IRIS_COLL_ALL_GATHER, "all_reduce": _native.IRIS_COLL_ALL_REDUCE,
         "reduce_scatter": _native.IRIS_COLL_REDUCE_SCATTER, "all_to_all": _native.IRIS_COLL_ALL_TO_ALL,
         "broadcast": _native.IRIS_COLL_BROADCAST}


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


@dataclasses.dataclass(frozen=True)
class HeapTensor:
    """A tensor at byte ``offset`` of every heap region."""
    offset: int
    shape: tuple
    dtype: torch.dtype

    @property
    def nbytes(self) -> int:
        return math.prod(self.shape) * torch.empty((), dtype=self.dtype).element_size()


class SymmetricHeap:
    """W regions of ``rank_stride`` bytes in one device allocation: the
    single-GPU stand-in for W ranks' symmetric heaps (region r = rank r)."""

    def __init__(self, world: int, rank_bytes: int, device="cuda"):
        if not 1 <= world <= _native.IRIS_MAX_WORLD:
            raise ValueError("world size out of range")
        self.world = int(world)
        self.rank_stride = _round_up(max(int(rank_bytes), 256), 4096)
        self.buf = torch.empty(self.world * self.rank_stride, dtype=torch.uint8, device=device)
        self._top = 0

    def alloc(self, shape: Sequence[int], dtype: torch.dtype) -> HeapTensor:
        t = HeapTensor(_round_up(self._top, 256), tuple(int(s) for s in shape), dtype)
        if t.offset + t.nbytes > self.rank_stride:
            raise MemoryError("symmetric heap region exhausted")
        self._top = t.offset + t.nbytes
        return t

    def view(self, t: HeapTensor, rank: int) -> torch.Tensor:
        """Rank ``rank``'s copy of ``t`` as a device tensor (a view)."""
        start = rank * self.rank_stride + t.offset
        return self.buf[start:start + t.nbytes].view(t.dtype).view(t.shape)

    def c_heap(self) -> iris_b200_heap:
        return iris_b200_heap(self.buf.data_ptr(), self.rank_stride, self.world)

    @staticmethod
    def bytes_for(*tensors) -> int:
        """Region size holding the given (shape, dtype) pairs with 256-B alignment."""
        total = 0
        for shape, dtype in tensors:
            total = _round_up(total, 256) + math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        return total


def make_config(**kw) -> iris_b200_config:
    """Build a config struct; unknown keys raise, missing keys take defaults."""
    c = iris_b200_config()
    names = {f[0] for f in iris_b200_config._fields_}
    for k, v in kw.items():
        if k not in names:
            raise KeyError(k)
        setattr(c, k, int(v))
    return c


_DTN = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}


def _resolve(cfg, op: str, W: int, M: int, N: int, K: int, dtype: torch.dtype, coll: Optional[str] = None,
             count: int = 0, coll_dtype: Optional[torch.dtype] = None):
    """config="auto": the measured winner cached for this device and shape,
    else the winner of the nearest cached shape, else the static default
    (see tuning.py)."""
    if isinstance(cfg, str):
        if cfg != "auto":
            raise ValueError(f"unknown config {cfg!r}")
        from . import tuning
        cdt = _DTN[coll_dtype] if coll_dtype is not None else "f32"
        key = tuning.shape_key(op, W, M, N, K, _DTN[dtype], coll, count, cdt)
        shape = tuning.shape_info(op, W, M, N, K, _DTN[dtype], coll, count, cdt)
        hit = tuning.select(tuning.device_arch(), key, shape=shape)
        return hit or None
    return cfg


def _cfgp(cfg):
    if cfg is None:
        return None
    if isinstance(cfg, dict):
        cfg = make_config(**cfg)
    return ctypes.byref(cfg)


def workspace_size(op: str, M: int, N: int, K: int, world: int, dtype=torch.bfloat16, config=None) -> int:
    out = ctypes.c_size_t(0)
    _native.check("iris_b200_workspace_size", _native.load().iris_b200_workspace_size(
        _OPS[op], M, N, K, world, _DT[dtype], _cfgp(config), ctypes.byref(out)))
    return int(out.value)


class Workspace:
    """Zero-initialised device workspace, reusable across calls on one stream.

    The zero-fill is finished before the constructor returns, so the first
    call may run on any stream (a workspace is created once and reused)."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = max(256, _round_up(int(nbytes), 256))
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)
        if self.buf.is_cuda:
            torch.cuda.current_stream(self.buf.device).synchronize()

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()


def _ws(ws: Optional[Workspace], need: int, device) -> Workspace:
    if ws is None or ws.nbytes < need:
        ws = Workspace(need, device)
    return ws


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _bias_off(bias: Optional[HeapTensor]) -> int:
    return _native.IRIS_NO_BIAS if bias is None else bias.offset


def all_gather_matmul(heap: SymmetricHeap, A: HeapTensor, B: HeapTensor, out: HeapTensor,
                      gathered: HeapTensor, bias: Optional[HeapTensor] = None, config=None,
                      workspace: Optional[Workspace] = None, stream=None) -> Workspace:
    """out = all_gather(A_sharded) @ B + bias (A shards (M, K/W) in every region,
    B (K, N), bias and outputs in region 0).  Returns the workspace."""
    M, K_l = A.shape
    K, N = B.shape
    config = _resolve(config, "all_gather_matmul", heap.world, M, N, K, B.dtype)
    ws = _ws(workspace, workspace_size("all_gather_matmul", M, N, K, heap.world, B.dtype, config),
             heap.buf.device)
    _native.check("iris_b200_all_gather_matmul", _native.load().iris_b200_all_gather_matmul(
        ctypes.byref(heap.c_heap()), A.offset, B.offset, _bias_off(bias), out.offset,
        gathered.offset, M, N, K, _DT[B.dtype], _cfgp(config), ws.ptr, ws.nbytes, _stream(stream)))
    return ws


def _mm_coll(name, heap, A, B, out, bias, config, workspace, stream, M, N, K):
    config = _resolve(config, name, heap.world, M, N, K, B.dtype)
    ws = _ws(workspace, workspace_size(name, M, N, K, heap.world, B.dtype, config), heap.buf.device)
    fn = getattr(_native.load(), "iris_b200_" + name)
    _native.check("iris_b200_" + name, fn(
        ctypes.byref(heap.c_heap()), A.offset, B.offset, _bias_off(bias), out.offset, M, N, K,
        _DT[B.dtype], _cfgp(config), ws.ptr, ws.nbytes, _stream(stream)))
    return ws


def matmul_reduce_scatter(heap, A, B, out, bias=None, config=None, workspace=None, stream=None):
    """out_r = reduce_scatter(A_r @ B_r + bias_r) along N (A (M,K), B (K,N),
    out (M, N/W) in every region).  Returns the workspace."""
    M, K = A.shape
    N = B.shape[1]
    return _mm_coll("matmul_reduce_scatter", heap, A, B, out, bias, config, workspace, stream, M, N, K)


def matmul_all_reduce(heap, A, B, out, bias=None, config=None, workspace=None, stream=None):
    """out = all_reduce(A_r @ B_r + bias_r) (out (M, N) in region 0, or all
    regions with replicate_outputs).  Returns the workspace."""
    M, K = A.shape
    N = B.shape[1]
    return _mm_coll("matmul_all_reduce", heap, A, B, out, bias, config, workspace, stream, M, N, K)


def matmul_all_gather(heap, A, B, out, bias=None, config=None, workspace=None, stream=None):
    """out = all_gather(A_r @ B + bias) along M (A_r (M/W, K) per region, B in
    region 0, out (M, N) in region 0).  Returns the workspace."""
    M_l, K = A.shape
    N = B.shape[1]
    return _mm_coll("matmul_all_gather", heap, A, B, out, bias, config, workspace, stream,
                    M_l * heap.world, N, K)


def concurrent_gemm_collective(A: Optional[torch.Tensor], B: Optional[torch.Tensor],
                               C: Optional[torch.Tensor], coll: str, heap: Optional[SymmetricHeap],
                               x_in: Optional[HeapTensor], x_out: Optional[HeapTensor], config=None,
                               workspace: Optional[Workspace] = None, stream=None) -> Workspace:
    """C = A @ B (plain device tensors) concurrently with ``coll`` over the
    heap regions (x_in: count elements per region; x_out per the collective).
    Pass A = B = C = None to run the collective alone, heap = None for the
    GEMM alone.  Returns the workspace."""
    if C is not None:
        M, N = C.shape
        K = A.shape[1]
        gdt = C.dtype
        a_ptr, b_ptr, c_ptr = A.data_ptr(), B.data_ptr(), C.data_ptr()
        dev = C.device
    else:
        M = N = K = 0
        gdt = torch.bfloat16
        a_ptr = b_ptr = c_ptr = None
        dev = heap.buf.device
    W = heap.world if heap is not None else 1
    count = x_in.nbytes // torch.empty((), dtype=x_in.dtype).element_size() if x_in is not None else 0
    config = _resolve(config, "concurrent", W, M, N, K, gdt, coll if count else None, count,
                      x_in.dtype if x_in is not None else None)
    ws = _ws(workspace, workspace_size("concurrent", M, N, K, W, gdt, config), dev)
    hp = ctypes.byref(heap.c_heap()) if heap is not None else None
    _native.check("iris_b200_concurrent_gemm_collective",
                  _native.load().iris_b200_concurrent_gemm_collective(
                      a_ptr, b_ptr, c_ptr, M, N, K, _DT[gdt], _COLL[coll], hp,
                      x_in.offset if x_in is not None else 0,
                      x_out.offset if x_out is not None else 0, count,
                      _DT[x_in.dtype] if x_in is not None else _native.IRIS_F32,
                      _cfgp(config), ws.ptr, ws.nbytes, _stream(stream)))
    return ws


def concurrent_two_stream(A, B, C, coll: str, heap, x_in, x_out, gemm_workspace: Workspace,
                          comm_workspace: Workspace, gemm_stream, comm_stream, config=None):
    """The two-stream concurrent mode: the GEMM and the collective as two
    persistent kernels on two streams (disjoint SM sets; cfg gemm_ctas CTAs
    for the GEMM).  Workspaces are required (one per launch)."""
    if C is not None:
        M, N = C.shape
        K = A.shape[1]
        gdt = C.dtype
        a_ptr, b_ptr, c_ptr = A.data_ptr(), B.data_ptr(), C.data_ptr()
    else:
        M = N = K = 0
        gdt = torch.bfloat16
        a_ptr = b_ptr = c_ptr = None
    count = x_in.nbytes // torch.empty((), dtype=x_in.dtype).element_size() if x_in is not None else 0
    hp = ctypes.byref(heap.c_heap()) if heap is not None else None
    _native.check("iris_b200_concurrent_two_stream", _native.load().iris_b200_concurrent_two_stream(
        a_ptr, b_ptr, c_ptr, M, N, K, _DT[gdt], _COLL[coll], hp,
        x_in.offset if x_in is not None else 0, x_out.offset if x_out is not None else 0, count,
        _DT[x_in.dtype] if x_in is not None else _native.IRIS_F32, _cfgp(config),
        gemm_workspace.ptr, gemm_workspace.nbytes, comm_workspace.ptr, comm_workspace.nbytes,
        _stream(gemm_stream), _stream(comm_stream)))


def sm_partition_streams(gemm_sms: int):
    """Two streams on disjoint SM sets of the current device (CUDA green
    contexts, owned by the library): the first with at least `gemm_sms` SMs,
    the second with the rest.  Returns (gemm_stream, comm_stream, gemm_sms,
    comm_sms) with the streams as torch.cuda.ExternalStream.  For
    concurrent_two_stream pass config gemm_ctas=gemm_sms, grid=gemm_sms+comm_sms."""
    g, c = ctypes.c_void_p(), ctypes.c_void_p()
    gs, cs = ctypes.c_int(), ctypes.c_int()
    _native.check("iris_b200_sm_partition_streams", _native.load().iris_b200_sm_partition_streams(
        int(gemm_sms), ctypes.byref(g), ctypes.byref(c), ctypes.byref(gs), ctypes.byref(cs)))
    dev = torch.cuda.current_device()
    return (torch.cuda.ExternalStream(g.value, device=dev), torch.cuda.ExternalStream(c.value, device=dev),
            gs.value, cs.value)


def sm_partition_release():
    """Destroy the current device's SM partition (its streams must be idle)."""
    _native.check("iris_b200_sm_partition_release", _native.load().iris_b200_sm_partition_release())


def query_status(workspace: Workspace, stream=None):
    """Synchronise the stream and return (code, raw_status, where, index)."""
    st, wh, ix = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    rc = _native.load().iris_b200_query_status(ctypes.c_void_p(workspace.ptr), _stream(stream),
                                               ctypes.byref(st), ctypes.byref(wh), ctypes.byref(ix))
    return rc, st.value, wh.value, ix.value


def num_sms() -> int:
    n = ctypes.c_int(0)
    _native.check("iris_b200_num_sms", _native.load().iris_b200_num_sms(ctypes.byref(n)))
    return n.value
