"""Split-K for every fused op against the oracle.

With k_split > 1 (by default above K = 32768) every output tile's K range is
cut into chunks; chunk j of a tile is a GEMM item of its own, and the chunks'
fp32 partials are summed in chunk order (for the reduce ops in (rank, chunk)
order) through the chained reduce's running sum before the one rounding to
16 bits.  On small-integer inputs every
partial and every sum is exact, so the output must equal the oracle's bits
whatever the chunking; the gathered A is a copy and must always match.  Row
counts leave the last pair tile full, partial or half empty; N = 288 leaves a
partial last 64-column chunk of B."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gemm_collective_tiles_gb300 import query_status
from gemm_collective_tiles_gb300.runner import FusedProblem

pytestmark = pytest.mark.gpu


def bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_exact(got, want):
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def run(x, cfg, bias_on_m=False):
    prob = FusedProblem("ag_mm", x.W, x.M, x.N, x.K, x.dtype, bias=x.bias is not None, bias_on_m=bias_on_m,
                        config=cfg)
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    return prob.outputs()


# (W, M, N, K, k_split): chunks of whole shards, chunks inside a shard,
# chunks across shard boundaries, an odd K-block count, and more chunks than
# shards
CASES = [
    (4, 300, 256, 8192, 4), (2, 512, 288, 4096, 3), (8, 200, 512, 8192, 2),
    (4, 640, 256, 4160, 5), (2, 129, 320, 2048, 16), (8, 256, 256, 16384, 8),
]


@pytest.mark.parametrize("W,M,N,K,ks", CASES)
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_split_k_exact_integer(W, M, N, K, ks, dt):
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, dt, seed=4100 + M + N + ks, dist="int", scale=1,
                                    bias=True, bias_scale=3)
    want, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    outs = run(x, {"k_split": ks})
    assert_exact(bits(outs["gathered"]), want_g)
    assert_exact(bits(outs["out"][0]), want)


@pytest.mark.parametrize("extra", [{"grid": 2}, {"grid": 6, "group_m": 2}, {"replicate_outputs": 1},
                                   {"gather_parts": 4}, {"startup_gather": 2}, {"stages": 6}])
def test_split_k_schedules_exact(extra):
    """A grid of one or three pairs (the rings wrap many times), narrow
    swizzle groups, replicated outputs, gathers cut into row parts or copied
    by the TMA producer, and the six-stage pipeline."""
    W, M, N, K = 4, 520, 256, 8192
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "bf16", seed=4200, dist="int", scale=1, bias=True,
                                    bias_scale=3)
    want, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    outs = run(x, {"k_split": 4, **extra})
    assert_exact(bits(outs["gathered"]), want_g)
    for r in range(W if extra.get("replicate_outputs") else 1):
        assert_exact(bits(outs["out"][r]), want)


def test_split_k_row_bias_exact():
    W, M, N, K = 2, 300, 256, 4096
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "f16", seed=4300, dist="int", scale=1, bias=True,
                                    bias_scale=3, bias_len=M)
    want, _ = oracle.all_gather_matmul(x.A, x.B[0], x.bias, bias_on_m=True)
    assert_exact(bits(run(x, {"k_split": 4}, bias_on_m=True)["out"][0]), want)


def test_split_k_random_within_tolerance_of_unsplit():
    """Random inputs: the chunked sum rounds differently from one fp32
    accumulation over all of K, within the GEMM tolerance of the oracle.
    fp16 outputs, whose rounding step (2^-11 relative) is well below the
    tolerance; a bf16 step (up to 2^-7) is above it, so there a single
    legitimate rounding flip at the largest output could fail the bound."""
    W, M, N, K = 8, 512, 512, 16384
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "f16", seed=4400, dist="normal", scale=0.5, bias=True)
    want, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    ref = torch.from_numpy(want.view(np.int16)).view(torch.float16).float()
    for ks in (1, 4, 8):
        outs = run(x, {"k_split": ks})
        assert_exact(bits(outs["gathered"]), want_g)
        got = outs["out"][0].float()
        err = float((got - ref).abs().max() / ref.abs().max())
        assert err <= 5e-3, (ks, err)


@pytest.mark.parametrize("W,M,N,K,extra", [(4, 300, 256, 8192, {"tile_m": 128}), (2, 256, 264, 4096, {}),
                                           (2, 256, 136, 65536, {"k_split": 0})])
def test_split_k_where_it_does_not_apply(W, M, N, K, extra):
    """A split asked for (or, above K = 32768, the default one) on one-CTA
    tiles or with N not a multiple of 32 runs unsplit: exact all the same."""
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "bf16", seed=4500 + N, dist="int", scale=1, bias=True,
                                    bias_scale=3)
    want, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    outs = run(x, {"k_split": 4, **extra})
    assert_exact(bits(outs["gathered"]), want_g)
    assert_exact(bits(outs["out"][0]), want)


def reduce_want(x):
    if x.op == "mm_rs":
        return oracle.matmul_reduce_scatter(x.A, x.B, x.bias)
    return [oracle.matmul_all_reduce(x.A, x.B, x.bias)]


def run_reduce(x, cfg):
    prob = FusedProblem(x.op, x.W, x.M, x.N, x.K, x.dtype, bias=x.bias is not None, config=cfg)
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    return prob.outputs()


# (op, W, M, N, K, k_split): the chained reduce then runs over (rank, chunk);
# each rank's bias is added once, with its first chunk
REDUCE_CASES = [
    ("mm_rs", 4, 300, 512, 4096, 3), ("mm_rs", 2, 256, 256, 8192, 4), ("mm_rs", 2, 129, 1024, 2048, 16),
    ("mm_ar", 2, 520, 256, 4160, 5), ("mm_ar", 3, 256, 320, 8192, 2), ("mm_ar", 8, 100, 256, 4096, 4),
]


@pytest.mark.parametrize("op,W,M,N,K,ks", REDUCE_CASES)
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_split_k_reduce_ops_exact_integer(op, W, M, N, K, ks, dt):
    x = synthetic.make_fused_inputs(op, W, M, N, K, dt, seed=4600 + M + N + ks, dist="int", scale=1, bias=True,
                                    bias_scale=3)
    want = reduce_want(x)
    outs = run_reduce(x, {"k_split": ks})
    for r in range(W if op == "mm_rs" else 1):
        assert_exact(bits(outs["out"][r]), want[r])


@pytest.mark.parametrize("op", ["mm_rs", "mm_ar"])
def test_split_k_reduce_ops_schedules(op):
    """Replicated outputs, a grid of one pair, and random inputs within the
    GEMM tolerance of the oracle (fp16 outputs, as in the test above)."""
    W, M, N, K = 4, 300, 512, 8192
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=4700, dist="int", scale=1, bias=True, bias_scale=3)
    want = reduce_want(x)
    for extra in ({"replicate_outputs": 1}, {"grid": 2}):
        outs = run_reduce(x, {"k_split": 4, **extra})
        n = W if (op == "mm_rs" or extra.get("replicate_outputs")) else 1
        for r in range(n):
            assert_exact(bits(outs["out"][r]), want[r if op == "mm_rs" else 0])
    y = synthetic.make_fused_inputs(op, W, M, N, K, "f16", seed=4701, dist="normal", scale=0.5, bias=True)
    want = reduce_want(y)
    outs = run_reduce(y, {"k_split": 4})
    for r in range(W if op == "mm_rs" else 1):
        ref = torch.from_numpy(want[r].view(np.int16)).view(torch.float16).float()
        err = float((outs["out"][r].float() - ref).abs().max() / ref.abs().max())
        assert err <= 5e-3, (r, err)


@pytest.mark.parametrize("op", ["mm_rs", "mm_ar"])
def test_split_k_reduce_ops_row_bias_and_rank_inner(op):
    """Per-row bias (each rank's, added with its first chunk) and a request
    for the rank-fastest item order, which a split overrides: exact."""
    W, M, N, K = 2, 300, 256, 4096
    x = synthetic.make_fused_inputs(op, W, M, N, K, "f16", seed=4800, dist="int", scale=1, bias=True, bias_scale=3,
                                    bias_len=M)
    want = (oracle.matmul_reduce_scatter(x.A, x.B, x.bias, bias_on_m=True) if op == "mm_rs"
            else [oracle.matmul_all_reduce(x.A, x.B, x.bias, bias_on_m=True)])
    prob = FusedProblem(op, W, M, N, K, "f16", bias=True, bias_on_m=True, config={"k_split": 3, "rank_inner": 1})
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    outs = prob.outputs()
    for r in range(W if op == "mm_rs" else 1):
        assert_exact(bits(outs["out"][r]), want[r])


# matmul_all_gather: rank r's M_l rows land at rows r * M_l of the output; with
# split-K every rank's tiles chain over the K chunks through a running sum of
# all W x M_l rows.  M_l = 100 and 300 leave the last pair tile of every rank
# half or partly empty.
MM_AG_CASES = [(4, 4 * 100, 256, 4096, 4), (2, 2 * 300, 512, 8192, 3), (8, 8 * 256, 288, 2048, 16)]


@pytest.mark.parametrize("W,M,N,K,ks", MM_AG_CASES)
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_split_k_matmul_all_gather_exact_integer(W, M, N, K, ks, dt):
    x = synthetic.make_fused_inputs("mm_ag", W, M, N, K, dt, seed=4900 + M + N + ks, dist="int", scale=1,
                                    bias=True, bias_scale=3)
    want = oracle.matmul_all_gather(x.A, x.B[0], x.bias)
    outs = run_reduce(x, {"k_split": ks})
    assert_exact(bits(outs["out"][0]), want)


def test_split_k_matmul_all_gather_schedules():
    """Replicated outputs, per-row bias, a grid of one pair, and random inputs
    within the GEMM tolerance (fp16 outputs)."""
    W, M, N, K = 2, 2 * 300, 256, 8192
    x = synthetic.make_fused_inputs("mm_ag", W, M, N, K, "f16", seed=4950, dist="int", scale=1, bias=True,
                                    bias_scale=3)
    want = oracle.matmul_all_gather(x.A, x.B[0], x.bias)
    for extra in ({"replicate_outputs": 1}, {"grid": 2}):
        outs = run_reduce(x, {"k_split": 4, **extra})
        for r in range(W if extra.get("replicate_outputs") else 1):
            assert_exact(bits(outs["out"][r]), want)
    y = synthetic.make_fused_inputs("mm_ag", W, M, N, K, "f16", seed=4951, dist="int", scale=1, bias=True,
                                    bias_scale=3, bias_len=M // W)
    want = oracle.matmul_all_gather(y.A, y.B[0], y.bias, bias_on_m=True)
    prob = FusedProblem("mm_ag", W, M, N, K, "f16", bias=True, bias_on_m=True, config={"k_split": 4})
    prob.upload(y.A, y.B, y.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    assert_exact(bits(prob.outputs()["out"][0]), want)
    z = synthetic.make_fused_inputs("mm_ag", W, M, N, K, "f16", seed=4952, dist="normal", scale=0.5, bias=True)
    want = oracle.matmul_all_gather(z.A, z.B[0], z.bias)
    ref = torch.from_numpy(want.view(np.int16)).view(torch.float16).float()
    got = run_reduce(z, {"k_split": 4})["out"][0].float()
    err = float((got - ref).abs().max() / ref.abs().max())
    assert err <= 5e-3, err
