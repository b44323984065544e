"""The fused calls captured in a CUDA graph and replayed.

A serving loop that launches the same fused op many times can capture the
call once and replay it, so no host work (argument checks, tensor-map
encoding, the launch itself) is repeated.  That is safe because every call
keeps its state on the device: each launch reads the workspace epoch, tags
its ready flags and chain counters with the next one and publishes it when
its last CTA leaves, and resets the queue counters for the next launch.
These tests capture one call of each kind, replay it three times with the
outputs poisoned in between, and need the oracle's bits after every replay
(small-integer inputs, so every fp32 sum is exact)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gemm_collective_tiles_gb300 import query_status
from gemm_collective_tiles_gb300.runner import ConcurrentProblem, FusedProblem

pytestmark = pytest.mark.gpu


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_exact(got, want):
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def fused_want(x):
    if x.op == "ag_mm":
        out, g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
        return [out], g
    if x.op == "mm_rs":
        return oracle.matmul_reduce_scatter(x.A, x.B, x.bias), None
    if x.op == "mm_ar":
        return [oracle.matmul_all_reduce(x.A, x.B, x.bias)], None
    return [oracle.matmul_all_gather(x.A, x.B[0], x.bias)], None


def capture(run):
    """Warm up outside the capture (first-call set-up), then capture one call."""
    run()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    torch.cuda.synchronize()
    return g


# (op, W, M, N, K, config): the gather flags, the chained reduce, the reduce
# parts schedule, the queue schedule, split-K chains and replicated outputs
CASES = [
    ("ag_mm", 4, 300, 512, 256, {}),
    ("ag_mm", 2, 256, 256, 65536, {"k_split": 4}),
    ("mm_rs", 4, 300, 512, 256, {}),
    ("mm_rs", 4, 256, 512, 128, {"tile_m": 128, "reduce_mode": 2}),
    ("mm_ar", 4, 256, 256, 128, {"tile_m": 128, "reduce_mode": 1, "replicate_outputs": 1}),
    ("mm_ar", 2, 130, 256, 8192, {"k_split": 3}),
    ("mm_ag", 4, 4 * 100, 256, 128, {"replicate_outputs": 1}),
]


@pytest.mark.parametrize("op,W,M,N,K,cfg", CASES)
def test_fused_op_graph_replays_exact(op, W, M, N, K, cfg):
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=6100 + M + K, dist="int", scale=1, bias=True,
                                    bias_scale=3)
    want, want_g = fused_want(x)
    prob = FusedProblem(op, W, M, N, K, "bf16", bias=True, config=cfg)
    prob.upload(x.A, x.B, x.bias)
    g = capture(prob.run)
    replicated = cfg.get("replicate_outputs") and op != "mm_rs"
    for replay in range(3):
        prob.poison_outputs()
        g.replay()
        torch.cuda.synchronize()
        assert query_status(prob.ws)[0] == 0, replay
        outs = prob.outputs()
        for r in range(W if (op == "mm_rs" or replicated) else 1):
            assert_exact(bits(outs["out"][r]), want[r if op == "mm_rs" else 0])
        if want_g is not None:
            assert_exact(bits(outs["gathered"]), want_g)


@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter", "all_gather"])
def test_concurrent_graph_replays_exact(coll):
    W, count = 8, 8 * 16384
    M, N, K = 384, 256, 256
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=6200, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=6201)
    prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count, config={"comm_block": 8192})
    prob.upload(A, B, X)
    g = capture(prob.run)
    want = {"all_reduce": lambda: [oracle.all_reduce(X)] * W,
            "reduce_scatter": lambda: oracle.reduce_scatter(X),
            "all_gather": lambda: [oracle.all_gather(X)] * W}[coll]()
    for replay in range(3):
        prob.poison_outputs()
        g.replay()
        torch.cuda.synchronize()
        assert query_status(prob.ws)[0] == 0, replay
        out = prob.outputs()
        assert_exact(bits(out["C"]), oracle.gemm(A, B))
        for r in range(W):
            got = out["x"][r].contiguous().view(torch.uint8).numpy()
            exp = want[r] if want[r].dtype == np.uint8 else want[r].view(np.uint8)
            assert np.array_equal(got, exp), (replay, r)
