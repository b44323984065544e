"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element
by element, at sizes that span several tiles plus ragged tails.

Bars: data-movement outputs (gathered A, fp32 collectives) bit-exact; GEMM
outputs bit-exact on small-integer inputs (every fp32 sum exact, so the
accumulation order cannot matter) and within max|gpu - oracle| <= 5e-3 *
max|oracle| on random inputs (tensor-core fp32 accumulation is not a
sequential IEEE sum)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gemm_collective_tiles_gb300.runner import ConcurrentProblem, FusedProblem

pytestmark = pytest.mark.gpu

TOL = 5e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def assert_close(got_bits, want_bits, dt, tol=TOL):
    g = oracle.decode16(got_bits, dt)
    w = oracle.decode16(want_bits, dt)
    assert g.shape == w.shape
    assert np.isfinite(g).all(), "unwritten or non-finite output elements"
    err = np.max(np.abs(g - w)) if g.size else 0.0
    scale = np.max(np.abs(w)) if w.size else 0.0
    assert err <= tol * scale + 1e-30, f"max err {err} vs scale {scale}"


def assert_exact(got_bits, want_bits):
    assert got_bits.shape == want_bits.shape
    bad = np.argwhere(got_bits != want_bits)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def run_fused(x: synthetic.FusedInputs, config=None, bias_on_m=False):
    prob = FusedProblem(x.op, x.W, x.M, x.N, x.K, x.dtype, bias=x.bias is not None,
                        bias_on_m=bias_on_m, config=config)
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    return prob, prob.outputs()


# ------------------------------------------------------------------ GEMM tile

GEMM_SHAPES = [(128, 256, 64), (256, 512, 256), (200, 136, 72), (1, 8, 8), (384, 384, 512),
               (130, 264, 1024)]


@pytest.mark.parametrize("tile_n", [256, 128])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("shape", GEMM_SHAPES)
def test_gemm_exact_integer(shape, dt, tile_n):
    M, N, K = shape
    A, B = synthetic.make_gemm_inputs(M, N, K, dt, seed=100 + M + N + K, dist="int", scale=3)
    prob = ConcurrentProblem(M, N, K, dt, "all_reduce", 1, 0, config={"tile_n": tile_n})
    prob.upload(A, B)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    assert_exact(bits(prob.outputs()["C"]), oracle.gemm(A, B))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_gemm_random_tolerance(dt):
    M, N, K = 512, 768, 1024
    A, B = synthetic.make_gemm_inputs(M, N, K, dt, seed=7, dist="normal", scale=1.0)
    prob = ConcurrentProblem(M, N, K, dt, "all_reduce", 1, 0)
    prob.upload(A, B)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    assert_close(bits(prob.outputs()["C"]), oracle.gemm(A, B), dt)


def test_gemm_k_zero_writes_zeros():
    M, N = 130, 200
    A = torch.zeros((M, 0), dtype=torch.bfloat16)
    B = torch.zeros((0, N), dtype=torch.bfloat16)
    prob = ConcurrentProblem(M, N, 0, "bf16", "all_reduce", 1, 0)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    assert_exact(bits(prob.outputs()["C"]), np.zeros((M, N), dtype=np.uint16))


# ------------------------------------------------------------------ all_gather_matmul

def check_ag_mm(x, prob, outs, exact):
    want_out, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    assert_exact(bits(outs["gathered"]), want_g)
    if exact:
        assert_exact(bits(outs["out"][0]), want_out)
    else:
        assert_close(bits(outs["out"][0]), want_out, x.dtype)
    if prob.replicate:
        for r in range(1, x.W):
            assert_exact(bits(outs["out"][r]), bits(outs["out"][0]))


def test_ag_mm_w2_256_full_oracle():
    """The W=2 256x256x256 fp16 workload, checked on every element."""
    x = synthetic.make_fused_inputs(**synthetic.WORKLOADS["ag_mm_w2_256"])
    prob, outs = run_fused(x)
    check_ag_mm(x, prob, outs, exact=False)


@pytest.mark.parametrize("W,M,N,K,dt", [(2, 256, 256, 256, "f16"), (4, 200, 136, 96, "bf16"),
                                         (8, 300, 520, 512, "bf16"), (3, 129, 64, 48, "f16")])
@pytest.mark.parametrize("replicate", [0, 1])
def test_ag_mm_exact_integer(W, M, N, K, dt, replicate):
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, dt, seed=W * 1000 + M, dist="int",
                                    scale=2, bias=True, bias_scale=3)
    prob, outs = run_fused(x, config={"replicate_outputs": replicate})
    check_ag_mm(x, prob, outs, exact=True)


def test_ag_mm_bias_on_m_random():
    x = synthetic.make_fused_inputs("ag_mm", 4, 384, 256, 512, "bf16", seed=5, dist="normal",
                                    scale=0.5, bias=True, bias_len=384)
    prob, outs = run_fused(x, bias_on_m=True)
    want_out, want_g = oracle.all_gather_matmul(x.A, x.B[0], x.bias, bias_on_m=True)
    assert_exact(bits(outs["gathered"]), want_g)
    assert_close(bits(outs["out"][0]), want_out, "bf16")


# ------------------------------------------------------------------ reduce ops

@pytest.mark.parametrize("W,M,N,K,dt", [(4, 256, 512, 128, "f16"), (4, 200, 160, 72, "bf16"),
                                         (2, 128, 256, 64, "f16"), (8, 384, 1024, 256, "bf16"),
                                         (1, 136, 264, 64, "bf16")])
@pytest.mark.parametrize("exact", [True, False])
@pytest.mark.parametrize("reduce_mode", [0, 1, 2])
def test_mm_reduce_scatter(W, M, N, K, dt, exact, reduce_mode):
    kw = dict(dist="int", scale=2, bias_scale=3) if exact else dict(dist="uniform", scale=1.0)
    x = synthetic.make_fused_inputs("mm_rs", W, M, N, K, dt, seed=31 + W + M, bias=True, **kw)
    prob, outs = run_fused(x, config={"reduce_mode": reduce_mode})
    want = oracle.matmul_reduce_scatter(x.A, x.B, x.bias)
    for r in range(W):
        if exact:
            assert_exact(bits(outs["out"][r]), want[r])
        else:
            assert_close(bits(outs["out"][r]), want[r], dt)


@pytest.mark.parametrize("W,M,N,K,dt", [(8, 256, 256, 128, "bf16"), (3, 200, 136, 72, "f16")])
@pytest.mark.parametrize("replicate", [0, 1])
@pytest.mark.parametrize("reduce_mode", [0, 1, 2])
def test_mm_all_reduce_exact_integer(W, M, N, K, dt, replicate, reduce_mode):
    x = synthetic.make_fused_inputs("mm_ar", W, M, N, K, dt, seed=41 + W, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    prob, outs = run_fused(x, config={"replicate_outputs": replicate, "reduce_mode": reduce_mode})
    want = oracle.matmul_all_reduce(x.A, x.B, x.bias)
    assert_exact(bits(outs["out"][0]), want)
    if replicate:
        for r in range(1, W):
            assert_exact(bits(outs["out"][r]), want)


def test_mm_all_reduce_random_bias_on_m():
    x = synthetic.make_fused_inputs("mm_ar", 4, 256, 384, 256, "bf16", seed=43, dist="normal",
                                    scale=0.5, bias=True, bias_len=256)
    prob, outs = run_fused(x, bias_on_m=True)
    assert_close(bits(outs["out"][0]), oracle.matmul_all_reduce(x.A, x.B, x.bias, bias_on_m=True),
                 "bf16")


@pytest.mark.parametrize("tile_m", [256, 128])
def test_mm_reduce_scatter_subnormal_partials(tile_m):
    """Partials that are fp32 subnormals (entries +-{0,1,2} x 2^-70, products
    near 2^-140): the tensor-core accumulation, the middle ranks' reduce-adds
    at the L2 and the last rank's add all keep them, so the outputs (bf16, which
    shares fp32's exponent range) equal the oracle's bit for bit."""
    W, M, N, K = 4, 256, 256, 64
    g = torch.Generator().manual_seed(5)

    def tiny(shape):
        sign = torch.randint(0, 2, shape, generator=g).float() * 2 - 1
        mag = torch.randint(0, 3, shape, generator=g).float()
        return (sign * mag * 2.0 ** -70).to(torch.bfloat16)
    A = [tiny((M, K)) for _ in range(W)]
    B = [tiny((K, N)) for _ in range(W)]
    x = synthetic.FusedInputs("mm_rs", W, M, N, K, "bf16", A, B, None)
    _, outs = run_fused(x, config={"tile_m": tile_m})
    want = oracle.matmul_reduce_scatter(A, B, None)
    assert sum(int((w & 0x7FFF != 0).sum()) for w in want) > 500   # the case is not all zeros
    for r in range(W):
        assert_exact(bits(outs["out"][r]), want[r])


def test_rs_slices_concatenate_to_ar():
    """The two reduce ops agree bit for bit (same partials, same order)."""
    x = synthetic.make_fused_inputs("mm_rs", 4, 256, 512, 128, "bf16", seed=44, dist="normal",
                                    scale=0.5, bias=True)
    _, rs = run_fused(x)
    y = synthetic.FusedInputs("mm_ar", x.W, x.M, x.N, x.K, x.dtype, x.A, x.B, x.bias)
    _, ar = run_fused(y)
    assert_exact(np.concatenate([bits(t) for t in rs["out"]], axis=1), bits(ar["out"][0]))


# ------------------------------------------------------------------ matmul_all_gather

@pytest.mark.parametrize("W,M,N,K,dt", [(4, 384, 264, 128, "bf16"), (8, 4096 // 8 * 2, 512, 64, "f16"),
                                         (2, 250, 128, 72, "bf16")])
@pytest.mark.parametrize("replicate", [0, 1])
def test_mm_all_gather_exact_integer(W, M, N, K, dt, replicate):
    x = synthetic.make_fused_inputs("mm_ag", W, M, N, K, dt, seed=51 + W, dist="int", scale=2,
                                    bias=True, bias_scale=3)
    prob, outs = run_fused(x, config={"replicate_outputs": replicate})
    want = oracle.matmul_all_gather(x.A, x.B[0], x.bias)
    assert_exact(bits(outs["out"][0]), want)
    if replicate:
        for r in range(1, W):
            assert_exact(bits(outs["out"][r]), want)


# ------------------------------------------------------------------ concurrent mode

@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter", "all_gather"])
@pytest.mark.parametrize("gemm_ctas", [-1, 0, 40, 151])
def test_concurrent_collective_bit_exact(coll, gemm_ctas):
    W, count = 8, 3 * 65536 + 4096
    M, N, K = 384, 512, 256
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=61, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=62)
    prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count,
                             config={"gemm_ctas": gemm_ctas, "comm_block": 16384})
    prob.upload(A, B, X)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    out = prob.outputs()
    assert_exact(bits(out["C"]), oracle.gemm(A, B))
    if coll == "all_reduce":
        want = oracle.all_reduce(X)
        for r in range(W):
            assert np.array_equal(out["x"][r].numpy().view(np.uint32), want.view(np.uint32))
    elif coll == "reduce_scatter":
        want = oracle.reduce_scatter(X)
        for r in range(W):
            assert np.array_equal(out["x"][r].numpy().view(np.uint32), want[r].view(np.uint32))
    else:
        want = oracle.all_gather(X)
        for r in range(W):
            assert np.array_equal(out["x"][r].contiguous().view(torch.uint8).numpy(), want)


@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter"])
@pytest.mark.parametrize("W", [4, 8, 16])
@pytest.mark.parametrize("stage", [1, 2])
def test_concurrent_sum_in_place_or_staged_bit_exact(coll, W, stage):
    """The summing collectives with the sums in the load buffer (1) or in the
    warp's staging halves (2; applies where a sub-chunk fits 4 KB: W = 8 and
    16 with the default ring, not W = 4), over several items per warp so
    both staging halves and both load buffers are reused; with one and three
    ring buffers too."""
    count = W * (5 * 16384 + 1024)   # items of 64Ki elements cross the reduce-scatter slices
    M, N, K = 256, 256, 128
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=69, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=70 + W)
    want = oracle.all_reduce(X) if coll == "all_reduce" else oracle.reduce_scatter(X)
    for ring in (2, 1, 3):
        prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count,
                                 config={"comm_block": 65536, "gemm_ctas": 30, "coll_out_stage": stage,
                                         "coll_ring": ring})
        prob.upload(A, B, X)
        prob.poison_outputs()
        prob.run()
        torch.cuda.synchronize()
        from gemm_collective_tiles_gb300 import query_status
        assert query_status(prob.ws)[0] == 0
        out = prob.outputs()
        assert_exact(bits(out["C"]), oracle.gemm(A, B))
        for r in range(W):
            w = want if coll == "all_reduce" else want[r]
            assert np.array_equal(out["x"][r].numpy().view(np.uint32), w.view(np.uint32)), (ring, r)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_concurrent_all_to_all_and_broadcast_bit_exact(dt):
    W = 8
    count = W * (3 * 4096 + 512)     # per-rank slices of 12800 elements
    M, N, K = 256, 384, 192
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=65, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, dt, seed=66)
    want_a2a = oracle.all_to_all(X)
    prob = ConcurrentProblem(M, N, K, "bf16", "all_to_all", W, count, coll_dtype=dt,
                             config={"comm_block": 4096, "gemm_ctas": 60})
    prob.upload(A, B, X)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    out = prob.outputs()
    assert_exact(bits(out["C"]), oracle.gemm(A, B))
    for r in range(W):
        assert np.array_equal(out["x"][r].contiguous().view(torch.uint8).numpy(), want_a2a[r]), r
    for root in (0, 5):
        prob = ConcurrentProblem(0, 0, 0, "bf16", "broadcast", W, count, coll_dtype=dt,
                                 config={"comm_block": 8192, "root": root})
        prob.upload(X=X)
        prob.poison_outputs()
        prob.run()
        torch.cuda.synchronize()
        want = oracle.broadcast(X, root)
        for r in range(W):
            assert np.array_equal(prob.outputs()["x"][r].contiguous().view(torch.uint8).numpy(), want[r])


@pytest.mark.parametrize("coll", ["all_reduce", "reduce_scatter", "all_gather", "all_to_all", "broadcast"])
def test_two_stream_mode_bit_exact(coll):
    """The GEMM and the collective as two kernels on two streams."""
    W, count = 8, 8 * 16384
    M, N, K = 384, 512, 256
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=67, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=68)
    prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count, config={"comm_block": 8192, "gemm_ctas": 40})
    prob.upload(A, B, X)
    prob.poison_outputs()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    prob.run_two_stream(s1, s2)
    torch.cuda.synchronize()
    from gemm_collective_tiles_gb300 import query_status
    assert query_status(prob.ws)[0] == 0 and query_status(prob.ws2)[0] == 0
    out = prob.outputs()
    assert_exact(bits(out["C"]), oracle.gemm(A, B))
    want = {"all_reduce": lambda: [oracle.all_reduce(X)] * W,
            "reduce_scatter": lambda: oracle.reduce_scatter(X),
            "all_gather": lambda: [oracle.all_gather(X)] * W,
            "all_to_all": lambda: oracle.all_to_all(X),
            "broadcast": lambda: oracle.broadcast(X, 0)}[coll]()
    for r in range(W):
        got = out["x"][r].contiguous().view(torch.uint8).numpy()
        w = want[r] if want[r].dtype == np.uint8 else want[r].view(np.uint8)
        assert np.array_equal(got, w), r


@pytest.mark.parametrize("coll", ["all_reduce", "all_gather", "all_to_all"])
def test_two_stream_mode_on_sm_partition(coll):
    """The two-stream mode on streams of two green contexts with disjoint SM
    sets (the split enforced by the CUDA driver, not by occupancy): results bit for
    bit as before."""
    from gemm_collective_tiles_gb300 import query_status, sm_partition_release, sm_partition_streams
    W, count = 8, 8 * 16384
    M, N, K = 520, 512, 256
    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=71, dist="int", scale=3)
    X = synthetic.make_coll_inputs(W, count, "f32", seed=72)
    s_gemm, s_comm, gs, cs = sm_partition_streams(80)
    try:
        assert gs >= 80 and cs >= 1
        prob = ConcurrentProblem(M, N, K, "bf16", coll, W, count,
                                 config={"comm_block": 8192, "gemm_ctas": gs, "grid": gs + cs})
        prob.upload(A, B, X)
        prob.poison_outputs()
        torch.cuda.synchronize()
        prob.run_two_stream(s_gemm, s_comm)
        s_gemm.synchronize()
        s_comm.synchronize()
        assert query_status(prob.ws)[0] == 0 and query_status(prob.ws2)[0] == 0
        out = prob.outputs()
    finally:
        torch.cuda.synchronize()
        sm_partition_release()
    assert_exact(bits(out["C"]), oracle.gemm(A, B))
    want = {"all_reduce": lambda: [oracle.all_reduce(X)] * W,
            "all_gather": lambda: [oracle.all_gather(X)] * W,
            "all_to_all": lambda: oracle.all_to_all(X)}[coll]()
    for r in range(W):
        got = out["x"][r].contiguous().view(torch.uint8).numpy()
        w = want[r] if want[r].dtype == np.uint8 else want[r].view(np.uint8)
        assert np.array_equal(got, w), r


def test_concurrent_all_reduce_in_place_and_alone():
    W, count = 4, 100000
    X = synthetic.make_coll_inputs(W, count, "f32", seed=63)
    prob = ConcurrentProblem(0, 0, 0, "bf16", "all_reduce", W, count, in_place=True)
    prob.upload(X=X)
    prob.run()
    torch.cuda.synchronize()
    want = oracle.all_reduce(X)
    for r in range(W):
        assert np.array_equal(prob.outputs()["x"][r].numpy().view(np.uint32), want.view(np.uint32))


def test_concurrent_all_gather_16bit():
    W, count = 4, 24576 + 8
    X = synthetic.make_coll_inputs(W, count, "bf16", seed=64)
    prob = ConcurrentProblem(0, 0, 0, "bf16", "all_gather", W, count, coll_dtype="bf16",
                             config={"comm_block": 4096})
    prob.upload(X=X)
    prob.poison_outputs()
    prob.run()
    torch.cuda.synchronize()
    want = oracle.all_gather(X)
    for r in range(W):
        assert np.array_equal(prob.outputs()["x"][r].contiguous().view(torch.uint8).numpy(), want)


# ------------------------------------------------------------------ workspace reuse / config sweep

@pytest.mark.parametrize("op", ["ag_mm", "mm_rs", "mm_ar"])
def test_workspace_reuse_and_schedule_invariance(op):
    """Repeated launches on one workspace (epoch-tagged flags, self-resetting
    queues) and different CTA splits / grids give identical bits."""
    W, M, N, K = 4, 384, 512, 256
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=71, dist="normal", scale=0.5,
                                    bias=True)
    prob = FusedProblem(op, W, M, N, K, "bf16", bias=True)
    prob.upload(x.A, x.B, x.bias)
    ref = None
    for _ in range(3):
        prob.poison_outputs()
        prob.run()
        torch.cuda.synchronize()
        cur = [bits(t) for t in prob.outputs()["out"][: (W if op == "mm_rs" else 1)]]
        if ref is None:
            ref = cur
        for a, b in zip(ref, cur):
            assert_exact(a, b)
    for cfg in ({"gemm_ctas": 20}, {"grid": 7}, {"group_m": 1}, {"tile_n": 128}, {"gemm_ctas": -1},
                {"reduce_mode": 1}, {"reduce_mode": 1, "gemm_ctas": 30}, {"rank_inner": 1},
                {"rank_inner": 1, "reduce_mode": 1}, {"group_m": 3, "reduce_mode": 1}, {"reduce_mode": 2},
                {"reduce_mode": 2, "grid": 5}, {"reduce_mode": 3, "grid": 3}, {"reduce_mode": 3, "rank_inner": 1}):
        p2 = FusedProblem(op, W, M, N, K, "bf16", bias=True, config=cfg)
        p2.upload(x.A, x.B, x.bias)
        p2.poison_outputs()
        p2.run()
        torch.cuda.synchronize()
        cur = [bits(t) for t in p2.outputs()["out"][: (W if op == "mm_rs" else 1)]]
        for a, b in zip(ref, cur):
            if cfg.get("tile_n") == 128:
                assert_close(b, a, "bf16")   # different tile -> different MMA grouping
            else:
                assert_exact(a, b)


# ------------------------------------------------------------------ bounded waits

@pytest.mark.parametrize("op,skip", [("ag_mm", 3), ("mm_rs", 5)])
def test_missing_flag_times_out_and_context_survives(op, skip):
    """A ready-flag that is never released (test hook) makes the waiting tile's
    bounded wait give up: the kernel stops, status reports IRIS_ETIMEOUT, and
    the next call on the same workspace and context runs correctly."""
    from gemm_collective_tiles_gb300 import query_status, _native
    W, M, N, K = 4, 256, 512, 256
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=81, dist="int", scale=2)
    # the reduce op's flag waits belong to its comm-queue schedule
    bad = FusedProblem(op, W, M, N, K, "bf16", config={"debug_skip_flag": skip, "wait_ns": 50_000_000,
                                                       "reduce_mode": 1 if op == "mm_rs" else 0})
    bad.upload(x.A, x.B, x.bias)
    bad.run()
    rc, status, where, index = query_status(bad.ws)
    assert rc == _native.IRIS_ETIMEOUT and status != 0
    assert index == skip - 1 or where != 0
    good = FusedProblem(op, W, M, N, K, "bf16")
    good.ws = bad.ws            # same workspace, next epoch
    good.upload(x.A, x.B, x.bias)
    good.poison_outputs()
    good.run()
    assert query_status(good.ws)[0] == 0
    outs = good.outputs()
    if op == "ag_mm":
        assert_exact(bits(outs["out"][0]), oracle.all_gather_matmul(x.A, x.B[0], None)[0])
    else:
        want = oracle.matmul_reduce_scatter(x.A, x.B, None)
        for r in range(W):
            assert_exact(bits(outs["out"][r]), want[r])


@pytest.mark.parametrize("op", ["ag_mm", "mm_rs"])
def test_one_workspace_many_launches_varying_schedules(op):
    """Forty launches on one workspace, cycling through grids of 2 to 152
    CTAs, one-CTA and pair tiles and different splits: the last CTA of each
    launch resets the queues and publishes the epoch with one store, and the
    flags of earlier launches (other layouts) carry older epochs, so every
    launch must still give the oracle's bits (small-integer inputs)."""
    W, M, N, K = 4, 300, 512, 256
    x = synthetic.make_fused_inputs(op, W, M, N, K, "bf16", seed=72, dist="int", scale=1, bias=True, bias_scale=3)
    if op == "ag_mm":
        out, g = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
        want, want_g = [out], g
    else:
        want, want_g = oracle.matmul_reduce_scatter(x.A, x.B, x.bias), None
    # sized for the schedule that needs the most workspace (W fp32 partials)
    big = {"tile_m": 128, "reduce_mode": 2} if op == "mm_rs" else {"tile_m": 128}
    prob = FusedProblem(op, W, M, N, K, "bf16", bias=True, config=big)
    prob.upload(x.A, x.B, x.bias)
    from gemm_collective_tiles_gb300 import make_config, query_status
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cfgs = [{}, {"grid": 2}, {"grid": 6, "group_m": 2}, {"tile_m": 128}, {"tile_m": 128, "grid": 3},
            {"gemm_ctas": 20}, {"grid": sms - sms % 2}, {"tile_m": 128, "gemm_ctas": -1}]
    if op == "mm_rs":
        cfgs += [{"tile_m": 128, "reduce_mode": 2}, {"tile_m": 128, "reduce_mode": 1, "grid": 5}]
    for launch in range(40):
        cfg = cfgs[launch % len(cfgs)]
        prob.config = make_config(**cfg) if cfg else None
        prob.poison_outputs()
        prob.run()
        torch.cuda.synchronize()
        assert query_status(prob.ws)[0] == 0, (launch, cfg)
        outs = prob.outputs()
        for r in range(W if op == "mm_rs" else 1):
            assert_exact(bits(outs["out"][r]), want[r])
        if want_g is not None:
            assert_exact(bits(outs["gathered"]), want_g)
