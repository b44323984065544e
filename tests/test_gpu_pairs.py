"""CTA-pair tiles against one-CTA tiles and the oracle.

With tile_m 256 a 2-CTA cluster shares one tensor-core instruction per
256 x 256 tile: each CTA stages 128 rows of A and 128 columns of B and drains
its own 128 accumulator rows.  With tile_m 128 every CTA owns a 128 x 256
tile.  Both must give the same bits (each output element is the same
K-ordered fp32 accumulation) and, on small-integer inputs, exactly the
oracle's values.  Row counts are chosen so the odd CTA's half of the last
pair tile is full, partly below the last row, or wholly below it."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gemm_collective_tiles_gb300 import query_status
from gemm_collective_tiles_gb300.runner import FusedProblem

pytestmark = pytest.mark.gpu


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_exact(got, want):
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def run(x, tile_m, extra=None, bias_on_m=False):
    cfg = {"tile_m": tile_m}
    cfg.update(extra or {})
    prob = FusedProblem(x.op, x.W, x.M, x.N, x.K, x.dtype, bias=x.bias is not None, bias_on_m=bias_on_m,
                        config=cfg)
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    return prob.outputs()


def oracle_outputs(x, bias_on_m=False):
    if x.op == "ag_mm":
        out, g = oracle.all_gather_matmul(x.A, x.B[0], x.bias, bias_on_m=bias_on_m)
        return [out], g
    if x.op == "mm_rs":
        return oracle.matmul_reduce_scatter(x.A, x.B, x.bias, bias_on_m=bias_on_m), None
    if x.op == "mm_ar":
        return [oracle.matmul_all_reduce(x.A, x.B, x.bias, bias_on_m=bias_on_m)], None
    return [oracle.matmul_all_gather(x.A, x.B[0], x.bias, bias_on_m=bias_on_m)], None


# (op, W, M, N, K): M (or M / W for matmul_all_gather) ends a pair tile with
# the odd half full (256, 512), partial (200, 300, 129) or empty (100, 60)
CASES = [
    ("ag_mm", 4, 100, 512, 256), ("ag_mm", 4, 200, 520, 128), ("ag_mm", 8, 640, 256, 512),
    ("ag_mm", 2, 129, 264, 64),
    ("mm_rs", 4, 100, 512, 256), ("mm_rs", 4, 300, 1024, 128), ("mm_rs", 2, 512, 256, 192),
    ("mm_ar", 2, 60, 256, 128), ("mm_ar", 4, 300, 512, 64), ("mm_ar", 8, 256, 256, 256),
    ("mm_ag", 4, 4 * 100, 256, 128), ("mm_ag", 2, 2 * 300, 512, 64), ("mm_ag", 8, 8 * 256, 264, 128),
]


@pytest.mark.parametrize("op,W,M,N,K", CASES)
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_pair_tiles_exact_integer(op, W, M, N, K, dt):
    x = synthetic.make_fused_inputs(op, W, M, N, K, dt, seed=900 + W * 7 + M, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    pair = run(x, 256)
    single = run(x, 128)
    want, want_g = oracle_outputs(x)
    n_out = W if op == "mm_rs" else 1
    for r in range(n_out):
        assert_exact(bits(pair["out"][r]), want[r])
        assert_exact(bits(single["out"][r]), want[r])
    if want_g is not None:
        assert_exact(bits(pair["gathered"]), want_g)


@pytest.mark.parametrize("op", ["ag_mm", "mm_rs", "mm_ar", "mm_ag"])
def test_pair_tiles_match_single_cta_random(op):
    """Random inputs: tile_m 256 and tile_m 128 agree bit for bit."""
    W = 4
    M = 4 * 384 if op == "mm_ag" else 640
    x = synthetic.make_fused_inputs(op, W, M, 768, 512, "bf16", seed=77, dist="normal", scale=0.5,
                                    bias=True)
    pair = run(x, 256)
    single = run(x, 128)
    for a, b in zip(pair["out"], single["out"]):
        assert_exact(bits(a), bits(b))


def test_pair_tiles_replicated_and_small_grid():
    """Replicated outputs and a grid of one pair (every tile through the
    same two CTAs, so both rings wrap many times)."""
    x = synthetic.make_fused_inputs("mm_ar", 4, 520, 512, 128, "bf16", seed=78, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    want = oracle.matmul_all_reduce(x.A, x.B, x.bias)
    for extra in ({"replicate_outputs": 1}, {"grid": 2}, {"grid": 3, "group_m": 2}):
        outs = run(x, 256, extra)
        for r in range(4 if extra.get("replicate_outputs") else 1):
            assert_exact(bits(outs["out"][r]), want)


def test_pair_tiles_rejected_where_they_do_not_apply():
    from gemm_collective_tiles_gb300 import _native
    x = synthetic.make_fused_inputs("mm_rs", 2, 256, 256, 64, "bf16", seed=79, dist="int", scale=2)
    for extra in ({"tile_n": 128}, {"reduce_mode": 1}, {"reduce_mode": 2}):
        with pytest.raises(_native.IrisError) as e:
            run(x, 256, extra)
        assert e.value.code == _native.IRIS_EINVAL


@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter", "all_gather", "all_to_all", "broadcast"])
def test_pair_tiles_concurrent_mode(coll):
    """Concurrent mode with CTA pairs: both CTAs of a pair run each collective
    item (one slice per worker warp of either CTA) on their leased stages.
    GEMM bits equal the one-CTA run's; the collective is bit-exact."""
    from gemm_collective_tiles_gb300.runner import ConcurrentProblem
    W, count = 4, 5 * 16384 + 4096
    M, N, K = 520, 768, 256   # ragged M: the last pair tile's odd half is partial
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=95, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=96)
    outs = {}
    for tile_m in (256, 128):
        prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count,
                                 config={"tile_m": tile_m, "comm_block": 16384, "gemm_ctas": 60})
        prob.upload(A, B, X)
        prob.poison_outputs()
        prob.run()
        assert query_status(prob.ws)[0] == 0
        outs[tile_m] = prob.outputs()
    assert_exact(bits(outs[256]["C"]), oracle.gemm(A, B))
    assert_exact(bits(outs[256]["C"]), bits(outs[128]["C"]))
    if coll == "all_reduce":
        want = [oracle.all_reduce(X)] * W
    elif coll == "reduce_scatter":
        want = oracle.reduce_scatter(X)
    elif coll == "all_gather":
        want = [oracle.all_gather(X)] * W
    elif coll == "all_to_all":
        want = oracle.all_to_all(X)
    else:
        want = oracle.broadcast(X, 0)
    for r in range(W):
        got = outs[256]["x"][r].contiguous().view(torch.uint8).numpy()
        assert np.array_equal(got, np.ascontiguousarray(want[r]).view(np.uint8).reshape(-1)), f"rank {r}"


@pytest.mark.parametrize("tile_m", [256, 128])
def test_ag_mm_large_shards(tile_m):
    """Shards of K/W = 4096 columns (1 MB per 128-row block, 64 K-blocks per
    shard flag): gathered A is bit-exact and the output exact on integer
    inputs; ragged M leaves a partial last block."""
    W, M, N, K = 4, 300, 256, 16384
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "bf16", seed=97, dist="int", scale=1,
                                    bias=True, bias_scale=2)
    outs = run(x, tile_m)
    want, want_g = oracle_outputs(x)
    assert_exact(bits(outs["gathered"]), want_g)
    assert_exact(bits(outs["out"][0]), want[0])


# (op, W, M, N, K, grid): with `grid` CTAs (grid/2 pairs) the tile count leaves
# a last wave at most half full, so its tiles run as two 256 x 128 column
# halves (for the reduce ops: the last rank's final tiles only)
TAIL_CASES = [
    ("mm_rs", 2, 640, 768, 128, 8),     # 9 tiles per rank, 18 items, 4 pairs: 2 tail tiles of rank 1
    ("mm_ar", 3, 520, 512, 64, 8),      # 6 tiles per rank, 18 items: 2 tail tiles of rank 2
    ("ag_mm", 4, 600, 768, 256, 8),     # 9 tiles, 4 pairs: 1 tail tile
    ("mm_ag", 2, 2 * 300, 520, 128, 10),  # 12 tiles, 5 pairs: 2 tail tiles (ragged M and N)
    ("mm_ag", 2, 2 * 300, 784, 128, 8),   # 16 tiles, 4 pairs: no split (a control)
]


@pytest.mark.parametrize("op,W,M,N,K,grid", TAIL_CASES)
def test_tail_split_exact(op, W, M, N, K, grid):
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=700 + M + N, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    want, want_g = oracle_outputs(x)
    for extra in ({"grid": grid}, {"grid": 2 * grid}):
        pair = run(x, 256, extra)
        single = run(x, 128, extra)
        for r in range(W if op == "mm_rs" else 1):
            assert_exact(bits(pair["out"][r]), want[r])
            assert_exact(bits(single["out"][r]), want[r])
        if want_g is not None:
            assert_exact(bits(pair["gathered"]), want_g)


# (op, W, M, N, K): empty M, empty K (the output is the bias alone: zeros + bias,
# summed over the ranks for the reduce ops), a single row, and N = 8 per rank
DEGENERATE = [
    ("ag_mm", 4, 0, 256, 256), ("ag_mm", 4, 200, 136, 0), ("ag_mm", 2, 1, 8, 16),
    ("mm_rs", 4, 0, 512, 128), ("mm_rs", 2, 130, 256, 0), ("mm_rs", 4, 1, 32, 64),
    ("mm_ar", 3, 0, 256, 64), ("mm_ar", 2, 77, 264, 0), ("mm_ar", 2, 1, 8, 8),
    ("mm_ag", 4, 0, 256, 64), ("mm_ag", 2, 2 * 100, 136, 0), ("mm_ag", 4, 4 * 1, 8, 24),
]


@pytest.mark.parametrize("op,W,M,N,K", DEGENERATE)
@pytest.mark.parametrize("tile_m", [0, 128])   # 0: the default (pairs wherever they apply)
def test_degenerate_shapes(op, W, M, N, K, tile_m):
    x = synthetic.make_fused_inputs(op, W, M, N, K, "f16", seed=800 + M + N + K, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    outs = run(x, tile_m)
    want, want_g = oracle_outputs(x)
    for r in range(W if op == "mm_rs" else 1):
        assert_exact(bits(outs["out"][r]), want[r])
    if want_g is not None:
        assert_exact(bits(outs["gathered"]), want_g)


# Both bias layouts through every epilogue: a per-row bias on pair tiles (with
# the split tail halves at `grid`) and on one-CTA tiles, and a per-column bias
# on one-CTA 128 x 128 tiles, where a warp's 128 columns of bias sit in half
# its lanes.  Small-integer inputs: every output must equal the oracle's bits.
@pytest.mark.parametrize("op,W,M,N,K,grid", TAIL_CASES)
@pytest.mark.parametrize("layout", ["row", "col_128x128"])
def test_bias_layouts_exact(op, W, M, N, K, grid, layout):
    bias_on_m = layout == "row"
    bias_len = (M // W if op == "mm_ag" else M) if bias_on_m else N
    x = synthetic.make_fused_inputs(op, W, M, N, K, "f16", seed=1700 + M + N + K, dist="int", scale=2,
                                    bias=True, bias_scale=3, bias_len=bias_len)
    want, want_g = oracle_outputs(x, bias_on_m)
    if bias_on_m:
        runs = [(256, {"grid": grid}), (256, {}), (128, {"grid": grid})]
    else:
        runs = [(128, {"tile_n": 128}), (128, {"tile_n": 128, "grid": grid})]
    for tile_m, extra in runs:
        outs = run(x, tile_m, extra, bias_on_m=bias_on_m)
        for r in range(W if op == "mm_rs" else 1):
            assert_exact(bits(outs["out"][r]), want[r])
        if want_g is not None:
            assert_exact(bits(outs["gathered"]), want_g)


# Both CTA-pair pipelines (3 stages of two K blocks, 6 stages of one) on
# small-integer inputs: K not a multiple of 64 (A loaded chunk by chunk), an
# odd number of K blocks (the last 3-stage slot half past K), a single K
# block, N not a multiple of 64 (B loaded chunk by chunk) and split tails.
STAGE_CASES = [
    ("ag_mm", 2, 300, 512, 208, 0), ("ag_mm", 4, 256, 256, 192, 0),
    ("mm_rs", 4, 300, 512, 64, 0), ("mm_rs", 2, 640, 768, 192, 8),
    ("mm_ar", 2, 260, 256, 320, 0), ("mm_ag", 2, 2 * 200, 520, 136, 0),
    ("mm_ag", 4, 4 * 256, 768, 512, 10),
]


@pytest.mark.parametrize("op,W,M,N,K,grid", STAGE_CASES)
@pytest.mark.parametrize("stages", [3, 6])
def test_pair_pipelines_exact(op, W, M, N, K, grid, stages):
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=2100 + M + N + K, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    want, want_g = oracle_outputs(x)
    extra = {"stages": stages}
    if grid:
        extra["grid"] = grid
    outs = run(x, 256, extra)
    for r in range(W if op == "mm_rs" else 1):
        assert_exact(bits(outs["out"][r]), want[r])
    if want_g is not None:
        assert_exact(bits(outs["gathered"]), want_g)


@pytest.mark.parametrize("stages", [3, 6])
def test_pair_pipelines_concurrent_gemm(stages):
    from gemm_collective_tiles_gb300.runner import ConcurrentProblem
    M, N, K = 520, 776, 328
    A, B = synthetic.make_gemm_inputs(M, N, K, "f16", seed=2200, dist="int", scale=2)
    prob = ConcurrentProblem(M, N, K, "f16", "all_reduce", 2, 0, config={"stages": stages})
    prob.upload(A, B)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    assert_exact(bits(prob.outputs()["C"]), oracle.gemm(A, B))


def test_pair_pipeline_choice_rejected_for_one_cta_tiles():
    from gemm_collective_tiles_gb300 import _native
    x = synthetic.make_fused_inputs("mm_ag", 2, 256, 256, 64, "bf16", seed=2300, dist="int", scale=2)
    with pytest.raises(_native.IrisError) as e:
        run(x, 128, {"stages": 6})
    assert e.value.code == _native.IRIS_EINVAL


# K > 98304: the default config runs the six-stage pipeline.  Inputs in
# {-1, 0, 1} keep every fp32 sum exact (|sum| <= K < 2^24).
@pytest.mark.parametrize("op,W,M,N,K", [("ag_mm", 2, 300, 256, 131072), ("mm_rs", 2, 256, 512, 106496)])
def test_long_k_default_pipeline_exact(op, W, M, N, K):
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=2400 + M, dist="int", scale=1)
    want, want_g = oracle_outputs(x)
    outs = run(x, 0)
    for r in range(W if op == "mm_rs" else 1):
        assert_exact(bits(outs["out"][r]), want[r])
    if want_g is not None:
        assert_exact(bits(outs["gathered"]), want_g)


@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter", "all_gather", "all_to_all", "broadcast"])
@pytest.mark.parametrize("ring,hint,store", [(3, 0, 1), (4, 1, 0), (2, 1, 0), (4, 2, 0), (2, 0, 2), (3, 1, 2),
                                             (0, 0, 3), (3, 1, 3), (1, 0, 1), (1, 1, 3)])
def test_concurrent_collective_paths(coll, ring, hint, store):
    """The collective tiles' buffer ring (1-4 buffers per worker warp), the
    L2 evict-first policy on their bulk copies, the way results leave the SM
    (TMA bulk stores or stores from registers) and the way sources arrive
    (one 1-D copy per source, or one 3-D box of all sources for the summing
    collectives) change only the schedule of the copies: the collective stays
    bit-exact against the oracle and the GEMM exact on integer inputs, with
    CTA pairs and with one CTA per tile."""
    from gemm_collective_tiles_gb300 import _native
    from gemm_collective_tiles_gb300.runner import ConcurrentProblem
    W, count = 8, 3 * 16384 + 4096 + 256   # a ragged last item of 17 one-KB rows
    M, N, K = 392, 512, 192
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=97, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=98)
    if store == 3 and coll not in ("all_reduce", "reduce_scatter"):
        # one box of all W sources per sub-chunk is a summing collective's path
        prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count,
                                 config={"comm_block": 16384, "coll_path": 3})
        with pytest.raises(_native.IrisError) as e:
            prob.run()
        assert e.value.code == _native.IRIS_EINVAL
        return
    if coll == "all_reduce":
        want = [oracle.all_reduce(X)] * W
    elif coll == "reduce_scatter":
        want = oracle.reduce_scatter(X)
    elif coll == "all_gather":
        want = [oracle.all_gather(X)] * W
    elif coll == "all_to_all":
        want = oracle.all_to_all(X)
    else:
        want = oracle.broadcast(X, 0)
    for tile_m in (256, 128):
        prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count,
                                 config={"tile_m": tile_m, "comm_block": 16384, "gemm_ctas": 50,
                                         "coll_ring": ring, "coll_l2_hint": hint, "coll_path": store})
        prob.upload(A, B, X)
        prob.poison_outputs()
        prob.run()
        assert query_status(prob.ws)[0] == 0
        out = prob.outputs()
        assert_exact(bits(out["C"]), oracle.gemm(A, B))
        for r in range(W):
            got = out["x"][r].contiguous().view(torch.uint8).numpy()
            assert np.array_equal(got, np.ascontiguousarray(want[r]).view(np.uint8).reshape(-1)), f"rank {r}"


@pytest.mark.parametrize("parts", [1, 3, 4, 16])
@pytest.mark.parametrize("tile_m", [256, 128])
def test_ag_mm_gather_parts_exact(parts, tile_m):
    """all_gather_matmul with each (row block, shard) copy cut into `parts`
    row parts (ragged: 392 rows leave a last block of 8 rows, fewer rows than
    parts): the gathered A is bit-exact and the output exact on integer
    inputs, for CTA pairs and one CTA per tile."""
    W, M, N, K = 4, 392, 520, 256
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "bf16", seed=99, dist="int", scale=2, bias=True,
                                    bias_scale=2)
    prob = FusedProblem("ag_mm", W, M, N, K, "bf16", bias=True, config={"gather_parts": parts, "tile_m": tile_m})
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    outs = prob.outputs()
    want_out, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    assert_exact(bits(outs["gathered"]), want_g)
    assert_exact(bits(outs["out"][0]), want_out)


@pytest.mark.parametrize("W,M,N,K", [(2, 256, 256, 256), (4, 392, 520, 256), (8, 200, 136, 576),
                                     (2, 1, 8, 16), (4, 640, 512, 4 * 2048)])
@pytest.mark.parametrize("tile_m", [0, 128])   # 0: the default (CTA pairs wherever they apply)
@pytest.mark.parametrize("startup", [1, 2])
def test_ag_mm_startup_gather_by_producer_exact(W, M, N, K, tile_m, startup):
    """The gathers claimed before a CTA's first GEMM tile copied by its TMA
    producer (2, the default at these sizes: boxes of up to 256 columns x 128
    rows through the idle stages; ragged rows, shards 8 to 2048 columns wide,
    one box or several batches) or by the worker threads (1): gathered A
    bit-exact, output exact on integer inputs."""
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "f16", seed=100 + M, dist="int", scale=2, bias=True,
                                    bias_scale=2)
    prob = FusedProblem("ag_mm", W, M, N, K, "f16", bias=True, config={"startup_gather": startup, "tile_m": tile_m})
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    outs = prob.outputs()
    want_out, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    assert_exact(bits(outs["gathered"]), want_g)
    assert_exact(bits(outs["out"][0]), want_out)


def test_ag_mm_startup_gather_stopped_then_exact():
    """A start-up gather whose ready counter is never completed (test hook)
    makes the waiting tile's bounded wait give up; the producer's copies
    drain, IRIS_ETIMEOUT is reported, and the next call on the same
    workspace is exact."""
    from gemm_collective_tiles_gb300 import _native
    W, M, N, K = 4, 256, 512, 256
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "bf16", seed=104, dist="int", scale=2)
    bad = FusedProblem("ag_mm", W, M, N, K, "bf16", config={"startup_gather": 2, "debug_skip_flag": 2,
                                                            "wait_ns": 50_000_000})
    bad.upload(x.A, x.B, x.bias)
    bad.run()
    assert query_status(bad.ws)[0] == _native.IRIS_ETIMEOUT
    good = FusedProblem("ag_mm", W, M, N, K, "bf16", config={"startup_gather": 2})
    good.ws = bad.ws
    good.upload(x.A, x.B, x.bias)
    good.poison_outputs()
    good.run()
    assert query_status(good.ws)[0] == 0
    want_out, want_g = oracle.all_gather_matmul(x.A, x.B[0], None)
    outs = good.outputs()
    assert_exact(bits(outs["gathered"]), want_g)
    assert_exact(bits(outs["out"][0]), want_out)


@pytest.mark.parametrize("op", ["ag_mm", "mm_rs", "mm_ag", "mm_ar"])
@pytest.mark.parametrize("hints", [{"gemm_l2_hint": 2}, {"out_l2_hint": 1}, {"sum_l2_hint": 1}, {"sum_l2_hint": 2}])
def test_gemm_l2_policies_exact(op, hints):
    """CTA-pair operand loads without the default L2 evict-last policy,
    final output stores with an evict-first policy, or running-sum stores
    and reduce-adds with either policy change only the cache state: outputs
    stay exact on integer inputs."""
    W, M, N, K = 4, 520, 512, 256
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=105, dist="int", scale=2, bias=True,
                                    bias_scale=2)
    prob = FusedProblem(op, W, M, N, K, "bf16", bias=True, config=hints)
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    outs = prob.outputs()
    if op == "ag_mm":
        want = [oracle.all_gather_matmul(x.A, x.B[0], x.bias)[0]]
    elif op == "mm_ag":
        want = [oracle.matmul_all_gather(x.A, x.B[0], x.bias)]
    elif op == "mm_ar":
        want = [oracle.matmul_all_reduce(x.A, x.B, x.bias)]
    else:
        want = oracle.matmul_reduce_scatter(x.A, x.B, x.bias)
    for r, w in enumerate(want):
        assert_exact(bits(outs["out"][r]), w)


def test_concurrent_gemm_evict_last_exact():
    from gemm_collective_tiles_gb300.runner import ConcurrentProblem
    W, count = 8, 2 * 16384 + 2048
    M, N, K = 520, 768, 256
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=106, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=107)
    prob = ConcurrentProblem(M, N, K, "bf16", "all_reduce", W, count,
                             config={"gemm_l2_hint": 1, "coll_l2_hint": 1, "comm_block": 16384, "gemm_ctas": 60})
    prob.upload(A, B, X)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    out = prob.outputs()
    assert_exact(bits(out["C"]), oracle.gemm(A, B))
    want = oracle.all_reduce(X)
    for r in range(W):
        assert np.array_equal(out["x"][r].numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("op,W,M,N,K", [("ag_mm", 2, 256, 256, 256), ("mm_rs", 2, 256, 512, 128),
                                        ("mm_ag", 2, 2 * 128, 256, 64), ("mm_ar", 2, 300, 256, 64)])
def test_small_problem_runs_one_pair_per_item(op, W, M, N, K):
    """A launch with fewer work items than CTA pairs starts one pair per item
    (the kernel-entry events of the device timeline count the CTAs that ran),
    and the result is exact."""
    x = synthetic.make_fused_inputs(op, W, M, N, K, "f16", seed=2500 + M + N, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    want, want_g = oracle_outputs(x)
    cap = 64
    tb = torch.zeros(152 * 4 * cap * 2, dtype=torch.int64, device="cuda")
    outs = run(x, 0, {"trace_buf": tb.data_ptr(), "trace_cap": cap})
    ran = int((tb.view(152, 4, cap, 2)[:, 0, 0, 0] > 0).sum().item())
    assert 2 <= ran <= 16 and ran % 2 == 0, ran
    for r in range(W if op == "mm_rs" else 1):
        assert_exact(bits(outs["out"][r]), want[r])
    if want_g is not None:
        assert_exact(bits(outs["gathered"]), want_g)
