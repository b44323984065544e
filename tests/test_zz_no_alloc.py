"""The no-allocation all_gather_matmul entry point.

Some callers cannot allocate device memory themselves (an allocator's own
bootstrap, a framework that owns every allocation, or a latency-critical path
that must not call cudaMalloc), so the library offers all_gather_matmul with its scratch
(queue counters, epoch, status and ready-flags) in a static device array
instead of a caller workspace.  This test calls it through the C ABI twice in
a row and checks each result against the workspace entry point's output on
the same inputs, within the GEMM tolerance the other tests use (the gathered
shards bit for bit).  It lives in its own file, collected last."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from gemm_collective_tiles_gb300 import _native
from gemm_collective_tiles_gb300.runner import FusedProblem

pytestmark = pytest.mark.gpu

TOL = 5e-3


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_noalloc_matches_workspace_entry_point():
    W, M, N, K = 4, 392, 520, 256
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "bf16", seed=91, dist="normal",
                                    scale=0.5, bias=True)
    prob = FusedProblem("ag_mm", W, M, N, K, "bf16", bias=True)
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    ref = prob.outputs()
    ref_out, ref_g = _bits(ref["out"][0]), _bits(ref["gathered"])

    lib = _native.load()
    heap = prob.heap.c_heap()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        prob.poison_outputs()
        torch.cuda.synchronize()
        rc = lib.iris_b200_all_gather_matmul_noalloc(
            ctypes.byref(heap), prob.A.offset, prob.B.offset, prob.bias.offset, prob.out.offset,
            prob.gathered.offset, M, N, K, _native.IRIS_BF16, None, stream)
        assert rc == _native.IRIS_OK, (call, rc, _native.strerror(rc))
        torch.cuda.synchronize()
        got = prob.outputs()
        assert np.array_equal(_bits(got["gathered"]), ref_g), f"call {call}: gathered A differs"
        g = oracle.decode16(_bits(got["out"][0]), "bf16")
        w = oracle.decode16(ref_out, "bf16")
        assert np.isfinite(g).all(), f"call {call}: unwritten output"
        assert np.max(np.abs(g - w)) <= TOL * np.max(np.abs(w)), f"call {call}"


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = _native.load()
    heap = _native.iris_b200_heap(1 << 20, 1 << 20, 8)
    too_many_rows = (_native.IRIS_NOALLOC_MAX_FLAGS // 8 + 1) * 128
    rc = lib.iris_b200_all_gather_matmul_noalloc(ctypes.byref(heap), 0, 0, _native.IRIS_NO_BIAS, 0, 0,
                                                 too_many_rows, 64, 64, _native.IRIS_BF16, None, None)
    assert rc == _native.IRIS_ENOWS
