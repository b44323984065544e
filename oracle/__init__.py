"""CPU oracle for the fused GEMM + collective operations.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call, link
or execute anything in this package: only the tests, the package smoke check
(``__graft_entry__.smoke``) and the benchmark's CPU-baseline leg use it.  It
shares no code with the CUDA path; the two meet only in the seeded input
generators of ``synthetic``.

Every function here is a plain definition written out, citing the page that
defines the operation:

* "Fused Communication and Compute Operations" (iris docs), sections
  ``all_gather_matmul``, ``matmul_all_gather``, ``matmul_reduce_scatter`` and
  ``matmul_all_reduce``: the four fused ops, their shapes and the bias.
* ROCm/iris PR #544 "Add iris.concurrent", description and commit messages:
  an independent GEMM beside an all-gather, all-reduce or reduce-scatter.

Arithmetic: 16-bit inputs are decoded exactly; each dot product is summed in
fp64 (exact products, fp64 adds) and rounded once to fp32, which stands for the
method's fp32 accumulator; bias adds and cross-rank sums are fp32 adds in rank
order 0..W-1; the result is rounded to fp16/bf16 with round-to-nearest-even.

Pins (``tests/test_oracle.py``, run with ``-m "not gpu"``): hand-derived
round-to-nearest-even cases and a sweep against torch's conversions; exact
integer brute force; the fp64 error bound against exact rational arithmetic;
the identity-B and bias-only special cases; the all-gather / per-shard-sum
identity; reduce-scatter slices against the all-reduce; a rank-order golden
case.  No function is unpinned.
"""
from .reference import (  # noqa: F401
    decode16,
    round16,
    round_bf16_bits,
    round_f16_bits,
    accumulate,
    gather_k,
    all_gather_matmul,
    all_gather_matmul_at,
    matmul_all_gather,
    matmul_all_gather_at,
    partial,
    rank_order_sum,
    matmul_reduce_scatter,
    matmul_reduce_scatter_at,
    matmul_all_reduce,
    matmul_all_reduce_at,
    gemm,
    gemm_at,
    all_reduce,
    all_gather,
    reduce_scatter,
    all_to_all,
    broadcast,
)
