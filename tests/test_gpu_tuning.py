"""Config selection on the GPU: tune a small fused op, the winner lands in
the JSON cache, config="auto" picks it up, and the auto-configured op still
matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import gemm_collective_tiles_gb300 as gct
from gemm_collective_tiles_gb300 import tuning

pytestmark = pytest.mark.gpu


def test_tune_then_auto(tmp_path, monkeypatch):
    path = str(tmp_path / "tuning.json")
    monkeypatch.setenv(tuning.ENV_CACHE, path)
    W, M, N, K = 4, 512, 1024, 512
    res = tuning.tune_fused("matmul_reduce_scatter", W, M, N, K, "bf16", top_k=4, reps=3)
    assert res["tried"] >= 2 and res["default_ms"] is not None
    assert res["ms"] <= res["default_ms"]
    key = tuning.shape_key("matmul_reduce_scatter", W, M, N, K, "bf16")
    assert tuning.select(tuning.device_arch(), key) == res["config"]

    x = synthetic.make_fused_inputs("mm_rs", W, M, N, K, "bf16", seed=95, dist="normal", scale=0.5,
                                    bias=True)
    dt = torch.bfloat16
    heap = gct.SymmetricHeap(W, gct.SymmetricHeap.bytes_for(((M, K), dt), ((K, N), dt), ((M, N // W), dt),
                                                            ((N,), dt)))
    A, B, out, bias = heap.alloc((M, K), dt), heap.alloc((K, N), dt), heap.alloc((M, N // W), dt), heap.alloc((N,), dt)
    for r in range(W):
        heap.view(A, r).copy_(x.A[r])
        heap.view(B, r).copy_(x.B[r])
        heap.view(bias, r).copy_(x.bias)
    gct.matmul_reduce_scatter(heap, A, B, out, bias, config="auto")
    torch.cuda.synchronize()
    want = oracle.matmul_reduce_scatter(x.A, x.B, x.bias)
    for r in range(W):
        got = oracle.decode16(heap.view(out, r).cpu().view(torch.int16).numpy().view(np.uint16), "bf16")
        w = oracle.decode16(want[r], "bf16")
        assert np.max(np.abs(got - w)) <= 5e-3 * np.max(np.abs(w))
