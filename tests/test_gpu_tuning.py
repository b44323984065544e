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


def test_tune_concurrent_then_auto(tmp_path, monkeypatch):
    """Tune a small concurrent GEMM + all-reduce (the static default, two
    other collective item sizes and the predictor's top (tile, split)
    candidates, measured on the device), the
    winner is cached under the concurrent key and never slower than the
    default; config="auto" then runs it: the GEMM exact on integer inputs and
    the all-reduce bit-exact against the oracle."""
    path = str(tmp_path / "tuning.json")
    monkeypatch.setenv(tuning.ENV_CACHE, path)
    W, count = 4, 1 << 22
    M, N, K = 1024, 1536, 512
    res = tuning.tune_concurrent(M, N, K, "bf16", "all_reduce", W, count, top_k=4, reps=3)
    assert res["tried"] >= 3 and res["default_ms"] is not None
    assert res["ms"] <= res["default_ms"]
    key = tuning.shape_key("concurrent", W, M, N, K, "bf16", "all_reduce", count, "f32")
    assert tuning.select(tuning.device_arch(), key) == res["config"]

    from gemm_collective_tiles_gb300.runner import ConcurrentProblem
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=96, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=97)
    prob = ConcurrentProblem(M, N, K, "bf16", "all_reduce", W, count)
    prob.upload(A, B, X)
    prob.poison_outputs()
    gct.concurrent_gemm_collective(prob.A, prob.B, prob.C, "all_reduce", prob.heap, prob.x_in, prob.x_out,
                                   config="auto", workspace=prob.ws)
    assert gct.query_status(prob.ws)[0] == 0
    out = prob.outputs()
    assert np.array_equal(out["C"].view(torch.int16).numpy().view(np.uint16), oracle.gemm(A, B))
    want = oracle.all_reduce(X)
    for r in range(W):
        assert np.array_equal(out["x"][r].numpy().view(np.uint32), want.view(np.uint32))


def test_nearest_shape_config_runs(tmp_path, monkeypatch):
    """A shape with no cache entry of its own takes the winner of the nearest
    cached shape (here one whose winner beat its default with one CTA per
    tile and a narrow swizzle group); the op runs with it and matches the
    oracle bit for bit on integer inputs."""
    path = str(tmp_path / "tuning.json")
    monkeypatch.setenv(tuning.ENV_CACHE, path)
    arch = tuning.device_arch()
    W, M, N, K = 4, 512, 768, 512
    near = {"tile_m": 128, "group_m": 8}
    tuning.record(arch, tuning.shape_key("all_gather_matmul", W, 1024, N, K, "f16"), near, 1.0, 1.5, path,
                  tuning.shape_info("all_gather_matmul", W, 1024, N, K, "f16"))
    key = tuning.shape_key("all_gather_matmul", W, M, N, K, "f16")
    assert tuning.select(arch, key, shape=tuning.shape_info("all_gather_matmul", W, M, N, K, "f16")) == near

    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "f16", seed=98, dist="int", scale=2, bias=True,
                                    bias_scale=2)
    dt = torch.float16
    heap = gct.SymmetricHeap(W, gct.SymmetricHeap.bytes_for(((M, K // W), dt), ((K, N), dt), ((M, N), dt),
                                                            ((N,), dt), ((M, K), dt)))
    A, B, out = heap.alloc((M, K // W), dt), heap.alloc((K, N), dt), heap.alloc((M, N), dt)
    bias, gathered = heap.alloc((N,), dt), heap.alloc((M, K), dt)
    for r in range(W):
        heap.view(A, r).copy_(x.A[r])
    heap.view(B, 0).copy_(x.B[0])
    heap.view(bias, 0).copy_(x.bias)
    ws = gct.all_gather_matmul(heap, A, B, out, gathered, bias, config="auto")
    assert gct.query_status(ws)[0] == 0
    want_out, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    assert np.array_equal(heap.view(gathered, 0).cpu().view(torch.int16).numpy().view(np.uint16), want_g)
    assert np.array_equal(heap.view(out, 0).cpu().view(torch.int16).numpy().view(np.uint16), want_out)
