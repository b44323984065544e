"""The largest world size the library accepts (IRIS_MAX_WORLD = 16 regions).

Every fused op, every reduce schedule, split-K and every concurrent
collective at W = 16 on small-integer inputs: the fp32 sums are exact, so
the outputs must equal the oracle's bit for bit.  At this W an all_gather
shard is 64 columns wide (K = 1024), a reduce-scatter slice 32 columns
(N = 512), and one 1 KB row of all 16 sources fills a collective ring
buffer."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gemm_collective_tiles_gb300 import _native, query_status
from gemm_collective_tiles_gb300.runner import ConcurrentProblem, FusedProblem

pytestmark = pytest.mark.gpu

W = 16


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_exact(got, want):
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def test_max_world_is_sixteen():
    assert _native.IRIS_MAX_WORLD == W


def fused_want(x):
    if x.op == "ag_mm":
        out, g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
        return [out], g
    if x.op == "mm_rs":
        return oracle.matmul_reduce_scatter(x.A, x.B, x.bias), None
    if x.op == "mm_ar":
        return [oracle.matmul_all_reduce(x.A, x.B, x.bias)], None
    return [oracle.matmul_all_gather(x.A, x.B[0], x.bias)], None


def run_fused(x, cfg):
    prob = FusedProblem(x.op, x.W, x.M, x.N, x.K, x.dtype, bias=x.bias is not None, config=cfg)
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    return prob.outputs()


# (op, M, N, K, config): CTA pairs (the default) and one-CTA tiles; for the
# reduce ops also the parts and queue schedules; all_gather_matmul and the
# reduce ops also split along K
CASES = [
    ("ag_mm", 300, 512, 1024, {}),
    ("ag_mm", 300, 512, 1024, {"tile_m": 128}),
    ("ag_mm", 256, 256, 16 * 2048, {"k_split": 4}),
    ("mm_rs", 200, 512, 128, {}),
    ("mm_rs", 200, 512, 128, {"tile_m": 128, "reduce_mode": 2}),
    ("mm_rs", 200, 512, 128, {"tile_m": 128, "reduce_mode": 1}),
    ("mm_rs", 256, 512, 4096, {"k_split": 2}),
    ("mm_ar", 256, 256, 192, {}),
    ("mm_ar", 256, 256, 192, {"replicate_outputs": 1}),
    ("mm_ar", 130, 256, 2048, {"k_split": 3}),
    ("mm_ag", 16 * 40, 264, 128, {}),
    ("mm_ag", 16 * 40, 264, 128, {"replicate_outputs": 1}),
    ("mm_ag", 16 * 64, 256, 4096, {"k_split": 2}),
]


@pytest.mark.parametrize("op,M,N,K,cfg", CASES)
def test_fused_ops_at_max_world_exact(op, M, N, K, cfg):
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=5100 + M + K, dist="int", scale=1, bias=True,
                                    bias_scale=3)
    want, want_g = fused_want(x)
    outs = run_fused(x, cfg)
    replicated = cfg.get("replicate_outputs") and op != "mm_rs"
    for r in range(W if (op == "mm_rs" or replicated) else 1):
        assert_exact(bits(outs["out"][r]), want[r if op == "mm_rs" else 0])
    if want_g is not None:
        assert_exact(bits(outs["gathered"]), want_g)


@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter", "all_gather", "all_to_all", "broadcast"])
def test_concurrent_collectives_at_max_world_exact(coll):
    """A GEMM beside each collective over 16 regions: the GEMM exact on
    integers, the collective bit for bit (the fp32 sums in rank order)."""
    count = W * (2 * 4096 + 256)
    M, N, K = 384, 256, 256
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=5200, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=5201)
    prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count, config={"comm_block": 4096, "gemm_ctas": 60})
    prob.upload(A, B, X)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    assert query_status(prob.ws)[0] == 0
    out = prob.outputs()
    assert_exact(bits(out["C"]), oracle.gemm(A, B))
    want = {"all_reduce": lambda: [oracle.all_reduce(X)] * W,
            "reduce_scatter": lambda: oracle.reduce_scatter(X),
            "all_gather": lambda: [oracle.all_gather(X)] * W,
            "all_to_all": lambda: oracle.all_to_all(X),
            "broadcast": lambda: oracle.broadcast(X, 11)}
    if coll == "broadcast":
        prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count, config={"comm_block": 4096, "root": 11})
        prob.upload(A, B, X)
        prob.poison_outputs()
        prob.run()
        torch.cuda.synchronize()
        assert query_status(prob.ws)[0] == 0
        out = prob.outputs()
    w = want[coll]()
    for r in range(W):
        got = out["x"][r].contiguous().view(torch.uint8).numpy()
        exp = w[r] if w[r].dtype == np.uint8 else w[r].view(np.uint8)
        assert np.array_equal(got, exp), r


def test_two_stream_all_reduce_at_max_world_exact():
    count = W * 4096
    M, N, K = 256, 256, 128
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=5300, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=5301)
    prob = ConcurrentProblem(M, N, K, "bf16", "all_reduce", W, count, config={"comm_block": 4096, "gemm_ctas": 40})
    prob.upload(A, B, X)
    prob.poison_outputs()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    prob.run_two_stream(s1, s2)
    torch.cuda.synchronize()
    assert query_status(prob.ws)[0] == 0 and query_status(prob.ws2)[0] == 0
    out = prob.outputs()
    assert_exact(bits(out["C"]), oracle.gemm(A, B))
    want = oracle.all_reduce(X)
    for r in range(W):
        assert np.array_equal(out["x"][r].numpy().view(np.uint32), want.view(np.uint32)), r
