"""Problem set-up helpers: allocate the emulated symmetric heap and the
workspace for one fused op, upload per-rank host tensors, launch, and read the
outputs back.  Used by the tests, the smoke check and the benchmark; a user
with tensors already on the heap calls the ops in ``__init__`` directly.
"""
from __future__ import annotations

from typing import Dict, List, Optional

import torch

from . import (HeapTensor, SymmetricHeap, Workspace, all_gather_matmul, concurrent_gemm_collective,
               concurrent_two_stream, make_config, matmul_all_gather, matmul_all_reduce,
               matmul_reduce_scatter, workspace_size)

_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}
OPS = ("ag_mm", "mm_rs", "mm_ag", "mm_ar")
_OPNAME = {"ag_mm": "all_gather_matmul", "mm_rs": "matmul_reduce_scatter",
           "mm_ag": "matmul_all_gather", "mm_ar": "matmul_all_reduce"}


def gemm_flops(op: str, W: int, M: int, N: int, K: int) -> float:
    """Distinct multiply-add work of one call, 2 flops per MAC.  all_gather_matmul
    and matmul_all_gather compute one M x N x K product; the reduce ops compute
    one per rank."""
    if op in ("mm_rs", "mm_ar"):
        return 2.0 * W * M * N * K
    return 2.0 * M * N * K


class FusedProblem:
    """Heap + workspace for one fused op at fixed sizes.

    Sizes follow the op's own convention (iris docs "Fused Communication and
    Compute Operations"): ag_mm A shards (M, K/W); mm_ag A_r (M/W, K) with M the
    gathered rows; mm_rs / mm_ar A_r (M, K), B_r (K, N).
    """

    def __init__(self, op: str, W: int, M: int, N: int, K: int, dtype: str, bias: bool = False,
                 bias_on_m: bool = False, config: Optional[dict] = None, device="cuda"):
        assert op in OPS
        self.op, self.W, self.M, self.N, self.K = op, W, M, N, K
        self.dt = _DT[dtype]
        self.device = device
        cfg = dict(config or {})
        if bias_on_m:
            cfg["bias_on_m"] = 1
        self.config = make_config(**cfg) if cfg else None
        self.replicate = bool(cfg.get("replicate_outputs", 0))
        dt = self.dt
        if op == "ag_mm":
            a_shape, b_shape, out_shape = (M, K // W), (K, N), (M, N)
        elif op == "mm_ag":
            a_shape, b_shape, out_shape = (M // W, K), (K, N), (M, N)
        elif op == "mm_rs":
            a_shape, b_shape, out_shape = (M, K), (K, N), (M, N // W)
        else:
            a_shape, b_shape, out_shape = (M, K), (K, N), (M, N)
        bias_len = (a_shape[0] if op == "mm_ag" else M) if bias_on_m else N
        parts = [(a_shape, dt), (b_shape, dt), (out_shape, dt)]
        if bias:
            parts.append(((bias_len,), dt))
        if op == "ag_mm":
            parts.append(((M, K), dt))
        self.heap = SymmetricHeap(W, SymmetricHeap.bytes_for(*parts), device=device)
        self.A = self.heap.alloc(a_shape, dt)
        self.B = self.heap.alloc(b_shape, dt)
        self.out = self.heap.alloc(out_shape, dt)
        self.bias = self.heap.alloc((bias_len,), dt) if bias else None
        self.gathered = self.heap.alloc((M, K), dt) if op == "ag_mm" else None
        M_ws = M if op != "mm_ag" else M
        self.ws = Workspace(workspace_size(_OPNAME[op], M_ws, N, K, W, dt, self.config), device)

    # ----------------------------------------------------------------- data
    def per_rank_b(self) -> bool:
        return self.op in ("mm_rs", "mm_ar")

    def upload(self, A: List[torch.Tensor], B: List[torch.Tensor], bias: Optional[torch.Tensor],
               non_blocking: bool = False):
        """Copy host tensors into the heap: A_r into region r; B_r into region
        r (reduce ops) or the shared B into region 0; the bias into region 0,
        or into every region for the reduce ops (each rank adds its own)."""
        for r in range(self.W):
            self.heap.view(self.A, r).copy_(A[r], non_blocking=non_blocking)
        if self.per_rank_b():
            for r in range(self.W):
                self.heap.view(self.B, r).copy_(B[r], non_blocking=non_blocking)
        else:
            self.heap.view(self.B, 0).copy_(B[0], non_blocking=non_blocking)
        if self.bias is not None:
            regions = range(self.W) if self.per_rank_b() else [0]
            for r in regions:
                self.heap.view(self.bias, r).copy_(bias, non_blocking=non_blocking)

    def input_bytes(self) -> int:
        nb = self.A.nbytes * self.W + self.B.nbytes * (self.W if self.per_rank_b() else 1)
        if self.bias is not None:
            nb += self.bias.nbytes * (self.W if self.per_rank_b() else 1)
        return nb

    def poison_outputs(self):
        """Fill every output copy with 0xFF bytes (NaN in fp16/bf16) so an
        element the kernel fails to write cannot pass a comparison."""
        for r in range(self.W):
            self.heap.view(self.out, r).view(torch.uint8).fill_(0xFF)
            if self.gathered is not None:
                self.heap.view(self.gathered, r).view(torch.uint8).fill_(0xFF)

    # ----------------------------------------------------------------- run
    def run(self, stream=None):
        if self.op == "ag_mm":
            all_gather_matmul(self.heap, self.A, self.B, self.out, self.gathered, self.bias,
                              self.config, self.ws, stream)
        elif self.op == "mm_rs":
            matmul_reduce_scatter(self.heap, self.A, self.B, self.out, self.bias, self.config,
                                  self.ws, stream)
        elif self.op == "mm_ar":
            matmul_all_reduce(self.heap, self.A, self.B, self.out, self.bias, self.config,
                              self.ws, stream)
        else:
            matmul_all_gather(self.heap, self.A, self.B, self.out, self.bias, self.config,
                              self.ws, stream)

    def outputs(self) -> Dict[str, object]:
        """Host copies: 'out' (list per region) and 'gathered' (region 0)."""
        res = {"out": [self.heap.view(self.out, r).cpu() for r in range(self.W)]}
        if self.gathered is not None:
            res["gathered"] = self.heap.view(self.gathered, 0).cpu()
        return res

    def flops(self) -> float:
        return gemm_flops(self.op, self.W, self.M, self.N, self.K)


class ConcurrentProblem:
    """Independent GEMM C = A @ B plus a collective over W heap regions."""

    def __init__(self, M: int, N: int, K: int, gemm_dtype: str, coll: str, W: int, count: int,
                 coll_dtype: str = "f32", in_place: bool = False, config: Optional[dict] = None,
                 device="cuda"):
        self.M, self.N, self.K, self.coll, self.W, self.count = M, N, K, coll, W, count
        self.gdt = _DT[gemm_dtype]
        self.cdt = _DT[coll_dtype]
        self.config = make_config(**config) if config else None
        self.has_gemm = M > 0 and N > 0
        if self.has_gemm:
            self.A = torch.empty((M, K), dtype=self.gdt, device=device)
            self.B = torch.empty((K, N), dtype=self.gdt, device=device)
            self.C = torch.empty((M, N), dtype=self.gdt, device=device)
        else:
            self.A = self.B = self.C = None
        self.heap = None
        self.x_in = self.x_out = None
        if count > 0:
            out_count = count * W if coll == "all_gather" else (count // W if coll == "reduce_scatter" else count)
            parts = [((count,), self.cdt)]
            if not in_place:
                parts.append(((out_count,), self.cdt))
            self.heap = SymmetricHeap(W, SymmetricHeap.bytes_for(*parts), device=device)
            self.x_in = self.heap.alloc((count,), self.cdt)
            self.x_out = self.x_in if in_place else self.heap.alloc((out_count,), self.cdt)
        self.ws = Workspace(workspace_size("concurrent", M, N, K, W, self.gdt, self.config), device)

    def upload(self, A=None, B=None, X: Optional[List[torch.Tensor]] = None, non_blocking=False):
        if A is not None:
            self.A.copy_(A, non_blocking=non_blocking)
            self.B.copy_(B, non_blocking=non_blocking)
        if X is not None:
            for r in range(self.W):
                self.heap.view(self.x_in, r).copy_(X[r], non_blocking=non_blocking)

    def poison_outputs(self):
        if self.C is not None:
            self.C.view(torch.uint8).fill_(0xFF)
        if self.x_out is not None and self.x_out is not self.x_in:
            for r in range(self.W):
                self.heap.view(self.x_out, r).view(torch.uint8).fill_(0xFF)

    def run(self, stream=None):
        concurrent_gemm_collective(self.A, self.B, self.C, self.coll, self.heap, self.x_in, self.x_out,
                                   self.config, self.ws, stream)

    def run_two_stream(self, gemm_stream, comm_stream):
        """The two-kernel mode: GEMM on gemm_stream, the collective on
        comm_stream (config gemm_ctas CTAs for the GEMM)."""
        if not hasattr(self, "ws2"):
            self.ws2 = Workspace(self.ws.nbytes, self.ws.buf.device)
        concurrent_two_stream(self.A, self.B, self.C, self.coll, self.heap, self.x_in, self.x_out,
                              self.ws, self.ws2, gemm_stream, comm_stream, self.config)

    def outputs(self):
        res = {}
        if self.C is not None:
            res["C"] = self.C.cpu()
        if self.x_out is not None:
            res["x"] = [self.heap.view(self.x_out, r).cpu() for r in range(self.W)]
        return res

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K if self.has_gemm else 0.0

    def coll_bytes(self) -> float:
        """Algorithmic collective traffic: W inputs read once, outputs written once."""
        esz = torch.empty((), dtype=self.cdt).element_size()
        if self.count == 0:
            return 0.0
        if self.coll == "all_reduce":
            return float(2 * self.W * self.count * esz)
        if self.coll == "reduce_scatter":
            return float(self.W * self.count * esz + self.count * esz)
        return float(self.W * self.count * esz + self.W * self.W * self.count * esz)
