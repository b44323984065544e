"""Pins for the CPU oracle: each test ties the oracle to something other than
itself (hand-derived values, exact arithmetic, error bounds, identities that
link different oracle functions, library routines).  CPU only."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _t(x, dt):
    return torch.tensor(x, dtype=torch.float32).to(synthetic.DTYPES[dt])


def _hex_bits(rows):
    return np.array([[int(v, 16) for v in r] for r in rows], dtype=np.uint16)


# ----------------------------------------------------------------- rounding

def test_rne16_golden_cases():
    g = _load("rne16_cases.json")
    for src, dt, want, why in g["cases"]:
        x = np.array([int(src, 16)], dtype=np.uint32).view(np.float32)
        got = oracle.round16(x, dt)[0]
        assert got == int(want, 16), (src, dt, hex(got), want, why)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_rne16_matches_torch_on_random_bits(dt):
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # add every pattern near a rounding boundary of the low 16 bits
    edge = (rng.integers(0, 2**16, size=4096, dtype=np.uint64).astype(np.uint32) << 16)
    bits = np.concatenate([bits, edge | 0x8000, edge | 0x7FFF, edge | 0x8001,
                           edge | 0x1000, edge | 0x0FFF, edge | 0x1001])
    x = bits.view(np.float32)
    ours = oracle.round16(x, dt)
    ref = torch.from_numpy(x.copy()).to(synthetic.DTYPES[dt]).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN
    dec = oracle.decode16(ours[nan], dt)
    assert np.isnan(dec).all()


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_decode16_roundtrip(dt):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    v = oracle.decode16(bits, dt)
    ok = ~np.isnan(v)
    back = oracle.round16(v[ok].astype(np.float32), dt)
    assert np.array_equal(back, bits[ok])
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(synthetic.DTYPES[dt]).to(torch.float64).numpy()
    assert np.array_equal(v[ok], ref[ok])


# ---------------------------------------------------------- hand-derived ops

def test_golden_fused_small():
    g = _load("fused_small.json")
    dt = g["dtype"]
    c = g["all_gather_matmul"]
    out, gathered = oracle.all_gather_matmul([_t(a, dt) for a in c["A_shards"]], _t(c["B"], dt),
                                             _t(c["bias"], dt))
    assert np.array_equal(out, _hex_bits(c["out_bits"]))
    assert np.array_equal(gathered, _hex_bits(c["gathered_bits"]))

    c = g["matmul_reduce_scatter"]
    outs = oracle.matmul_reduce_scatter([_t(a, dt) for a in c["A"]], [_t(b, dt) for b in c["B"]],
                                        _t(c["bias"], dt))
    for r, want in enumerate(c["out_bits"]):
        assert np.array_equal(outs[r], _hex_bits(want))

    c = g["matmul_all_reduce"]
    out = oracle.matmul_all_reduce([_t(a, dt) for a in c["A"]], [_t(b, dt) for b in c["B"]],
                                   _t(c["bias"], dt))
    assert np.array_equal(out, _hex_bits(c["out_bits"]))

    c = g["matmul_all_gather"]
    out = oracle.matmul_all_gather([_t(a, dt) for a in c["A"]], _t(c["B"], dt))
    assert np.array_equal(out, _hex_bits(c["out_bits"]))


def test_rank_order_golden():
    g = _load("rank_order_sum.json")
    X = [torch.tensor(b, dtype=torch.float32) for b in g["buffers"]]
    got = oracle.all_reduce(X)
    assert got.tolist() == g["expected"]


# ---------------------------------------------------------- brute force

def _int_inputs(op, W, M, N, K, dt, seed, bias=True):
    return synthetic.make_fused_inputs(op, W, M, N, K, dt, seed, dist="int", scale=3,
                                       bias=bias, bias_scale=2)


def _brute_int(A, B):
    """Exact integer matmul with Python ints (tiny shapes)."""
    A = [[int(v) for v in row] for row in A.to(torch.float64).tolist()]
    B = [[int(v) for v in row] for row in B.to(torch.float64).tolist()]
    M, K, N = len(A), len(B), len(B[0])
    return [[sum(A[i][k] * B[k][j] for k in range(K)) for j in range(N)] for i in range(M)]


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_ag_mm_exact_integer_brute_force(dt):
    W, M, N, K = 2, 5, 7, 6
    x = _int_inputs("ag_mm", W, M, N, K, dt, seed=11)
    out, gathered = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    # brute force: per-shard products against the matching row block of B,
    # summed over shards -- the all-gather along K written as a sum
    K_l = K // W
    want = [[0] * N for _ in range(M)]
    for s in range(W):
        part = _brute_int(x.A[s], x.B[0][s * K_l:(s + 1) * K_l])
        for i in range(M):
            for j in range(N):
                want[i][j] += part[i][j]
    bias = [int(v) for v in x.bias.to(torch.float64).tolist()]
    want = np.array([[want[i][j] + bias[j] for j in range(N)] for i in range(M)], dtype=np.float64)
    assert np.array_equal(oracle.decode16(out, dt), want)
    # gathered: shard s occupies columns [s*K_l, (s+1)*K_l)
    for s in range(W):
        blk = oracle.decode16(gathered[:, s * K_l:(s + 1) * K_l], dt)
        assert np.array_equal(blk, x.A[s].to(torch.float64).numpy())


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_mm_rs_ar_exact_integer_brute_force(dt):
    W, M, N, K = 4, 3, 8, 5
    x = _int_inputs("mm_rs", W, M, N, K, dt, seed=12)
    bias = [int(v) for v in x.bias.to(torch.float64).tolist()]
    S = np.zeros((M, N))
    for r in range(W):
        S += np.array(_brute_int(x.A[r], x.B[r]), dtype=np.float64) + np.array(bias)[None, :]
    outs = oracle.matmul_reduce_scatter(x.A, x.B, x.bias)
    N_l = N // W
    for r in range(W):
        assert np.array_equal(oracle.decode16(outs[r], dt), S[:, r * N_l:(r + 1) * N_l])
    ar = oracle.matmul_all_reduce(x.A, x.B, x.bias)
    assert np.array_equal(oracle.decode16(ar, dt), S)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_mm_ag_exact_integer_brute_force(dt):
    W, M, N, K = 2, 6, 5, 4      # M is the gathered M: 3 rows per rank
    x = _int_inputs("mm_ag", W, M, N, K, dt, seed=13)
    out = oracle.matmul_all_gather(x.A, x.B[0], x.bias)
    bias = np.array([int(v) for v in x.bias.to(torch.float64).tolist()], dtype=np.float64)
    M_l = M // W
    for r in range(W):
        want = np.array(_brute_int(x.A[r], x.B[0]), dtype=np.float64) + bias[None, :]
        assert np.array_equal(oracle.decode16(out[r * M_l:(r + 1) * M_l], dt), want)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_accumulator_within_fp64_error_bound(dt):
    """fp32 accumulator vs the exact rational dot product: the fp64 sum is
    within gamma_K * sum|a||b| of the exact value (Higham, Accuracy and
    Stability of Numerical Algorithms, section 3.1), then one fp32 rounding
    adds at most half an fp32 ulp."""
    M, N, K = 3, 4, 37
    A, B = synthetic.make_gemm_inputs(M, N, K, dt, seed=21, dist="uniform")
    acc = oracle.accumulate(A.to(torch.float64).numpy(), B.to(torch.float64).numpy())
    Af = [[Fraction(float(v)) for v in row] for row in A.to(torch.float64).tolist()]
    Bf = [[Fraction(float(v)) for v in row] for row in B.to(torch.float64).tolist()]
    u = 2.0 ** -53
    gamma = K * u / (1 - K * u)
    for i in range(M):
        for j in range(N):
            exact = sum(Af[i][k] * Bf[k][j] for k in range(K))
            mag = float(sum(abs(Af[i][k] * Bf[k][j]) for k in range(K)))
            half_ulp = float(np.spacing(np.float32(abs(float(exact))))) / 2
            err = abs(Fraction(float(acc[i, j])) - exact)
            assert float(err) <= gamma * mag + half_ulp + 1e-300


def test_accumulator_matches_numpy_fp64_matmul_rounded():
    """Special case reducing to a library routine: float64 matmul then fp32."""
    A, B = synthetic.make_gemm_inputs(17, 9, 33, "bf16", seed=22)
    a = A.to(torch.float64).numpy()
    b = B.to(torch.float64).numpy()
    want = (a @ b).astype(np.float32)
    assert np.array_equal(oracle.accumulate(a, b), want)
    assert np.array_equal(oracle.gemm(A, B), oracle.round16(want, "bf16"))


# ---------------------------------------------------------- identities / special cases

@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_identity_B_returns_gathered_A(dt):
    W, M, K = 4, 9, 16
    x = synthetic.make_fused_inputs("ag_mm", W, M, K, K, dt, seed=31, dist="uniform")
    eye = torch.eye(K, dtype=torch.float32).to(synthetic.DTYPES[dt])
    out, gathered = oracle.all_gather_matmul(x.A, eye)
    assert np.array_equal(out, gathered)
    # and the gathered block of shard s is shard s, bit for bit
    K_l = K // W
    for s in range(W):
        ref = x.A[s].contiguous().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(gathered[:, s * K_l:(s + 1) * K_l], ref)


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_bias_only(dt):
    """A = 0: all_gather_matmul gives RNE16(bias); the reduce ops sum the bias
    once per rank, so they give RNE16(W * bias) (exact for W a power of 2)."""
    W, M, N, K = 4, 5, 8, 8
    x = synthetic.make_fused_inputs("mm_rs", W, M, N, K, dt, seed=41, bias=True, bias_scale=0.7)
    zA = [torch.zeros_like(a) for a in x.A]
    bias64 = x.bias.to(torch.float64).numpy()
    bias_bits = x.bias.contiguous().view(torch.int16).numpy().view(np.uint16)
    y = synthetic.make_fused_inputs("ag_mm", W, M, N, K, dt, seed=42, bias=True)
    out, _ = oracle.all_gather_matmul([torch.zeros_like(a) for a in y.A], y.B[0], y.bias)
    ybits = y.bias.contiguous().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, np.broadcast_to(ybits, (M, N)))
    ar = oracle.matmul_all_reduce(zA, x.B, x.bias)
    assert np.array_equal(oracle.decode16(ar, dt), np.broadcast_to(W * bias64, (M, N)))
    outs = oracle.matmul_reduce_scatter(zA, x.B, x.bias)
    N_l = N // W
    for r in range(W):
        assert np.array_equal(oracle.decode16(outs[r], dt),
                              np.broadcast_to(W * bias64[r * N_l:(r + 1) * N_l], (M, N_l)))
    ag = oracle.matmul_all_gather([torch.zeros(2, K).to(synthetic.DTYPES[dt])] * W, x.B[0], x.bias)
    assert np.array_equal(ag, np.broadcast_to(bias_bits, (2 * W, N)))


def test_bias_on_m():
    W, M, N, K = 2, 6, 4, 4
    x = synthetic.make_fused_inputs("mm_ar", W, M, N, K, "f16", seed=43, dist="int", scale=2,
                                    bias=True, bias_scale=3, bias_len=M)
    zA = [torch.zeros_like(a) for a in x.A]
    out = oracle.matmul_all_reduce(zA, x.B, x.bias, bias_on_m=True)
    b = x.bias.to(torch.float64).numpy()
    assert np.array_equal(oracle.decode16(out, "f16"), np.broadcast_to(W * b[:, None], (M, N)))


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_rs_concat_is_ar(dt):
    W, M, N, K = 4, 7, 16, 24
    x = synthetic.make_fused_inputs("mm_rs", W, M, N, K, dt, seed=51, bias=True)
    outs = oracle.matmul_reduce_scatter(x.A, x.B, x.bias)
    ar = oracle.matmul_all_reduce(x.A, x.B, x.bias)
    assert np.array_equal(np.concatenate(outs, axis=1), ar)


def test_collectives_agree():
    W, count = 8, 64
    X = synthetic.make_coll_inputs(W, count, "f32", seed=61)
    ar = oracle.all_reduce(X)
    rs = oracle.reduce_scatter(X)
    assert np.array_equal(np.concatenate(rs), ar)
    ag = oracle.all_gather(X).view(np.float32)
    # summing the gathered blocks in rank order reproduces the all-reduce
    blocks = [ag[s * count:(s + 1) * count] for s in range(W)]
    assert np.array_equal(oracle.rank_order_sum(blocks), ar)
    # each block is that rank's buffer
    for s in range(W):
        assert np.array_equal(blocks[s], X[s].numpy())


def test_all_reduce_of_identical_buffers_is_W_times():
    # values with 8 significant bits: every partial sum k*x (k <= 8) is exact
    # in fp32, so any order gives W*x
    for W in (2, 3, 4, 8):
        x = synthetic.make_coll_inputs(1, 1000, "bf16", seed=62)[0].to(torch.float32)
        got = oracle.all_reduce([x] * W)
        assert np.array_equal(got, (x.numpy().astype(np.float64) * W).astype(np.float32))


def test_round_partials_variant_is_close():
    W, M, N, K = 4, 8, 8, 64
    x = synthetic.make_fused_inputs("mm_ar", W, M, N, K, "bf16", seed=71, dist="normal",
                                    scale=0.5, bias=True)
    a = oracle.decode16(oracle.matmul_all_reduce(x.A, x.B, x.bias), "bf16")
    b = oracle.decode16(oracle.matmul_all_reduce(x.A, x.B, x.bias, round_partials=True), "bf16")
    assert np.max(np.abs(a - b)) <= 5e-3 * np.max(np.abs(a)) + 1e-6


# ---------------------------------------------------------- sampled == full

def test_sampled_variants_match_full():
    W, M, N, K = 4, 40, 48, 32
    x = synthetic.make_fused_inputs("ag_mm", W, M, N, K, "bf16", seed=81, dist="normal",
                                    bias=True)
    out, _ = oracle.all_gather_matmul(x.A, x.B[0], x.bias)
    ii, jj = synthetic.sample_indices(M, N, seed=1081, n=300, tile_m=16, tile_n=16)
    got = oracle.all_gather_matmul_at(x.A, x.B[0], x.bias, ii.numpy(), jj.numpy())
    assert np.array_equal(got, out[ii.numpy(), jj.numpy()])

    y = synthetic.make_fused_inputs("mm_rs", W, M, N, K, "f16", seed=82, bias=True)
    outs = oracle.matmul_reduce_scatter(y.A, y.B, y.bias)
    N_l = N // W
    ii, jj = synthetic.sample_indices(M, N_l, seed=1082, n=200, tile_m=8, tile_n=8)
    for r in range(W):
        got = oracle.matmul_reduce_scatter_at(y.A, y.B, y.bias, r, ii.numpy(), jj.numpy())
        assert np.array_equal(got, outs[r][ii.numpy(), jj.numpy()])
    ar = oracle.matmul_all_reduce(y.A, y.B, y.bias)
    ii, jj = synthetic.sample_indices(M, N, seed=1083, n=200, tile_m=8, tile_n=8)
    assert np.array_equal(oracle.matmul_all_reduce_at(y.A, y.B, y.bias, ii.numpy(), jj.numpy()),
                          ar[ii.numpy(), jj.numpy()])

    z = synthetic.make_fused_inputs("mm_ag", W, M, N, K, "bf16", seed=83, bias=True)
    ag = oracle.matmul_all_gather(z.A, z.B[0], z.bias)
    ii, jj = synthetic.sample_indices(M, N, seed=1084, n=200, tile_m=8, tile_n=8)
    assert np.array_equal(oracle.matmul_all_gather_at(z.A, z.B[0], z.bias, ii.numpy(), jj.numpy()),
                          ag[ii.numpy(), jj.numpy()])

    A, B = synthetic.make_gemm_inputs(M, N, K, "bf16", seed=84)
    c = oracle.gemm(A, B)
    assert np.array_equal(oracle.gemm_at(A, B, ii.numpy(), jj.numpy()), c[ii.numpy(), jj.numpy()])


# ---------------------------------------------------------- the independent GEMM

@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_gemm_golden(dt):
    g = _load("gemm_small.json")
    C = oracle.gemm(_t(g["A"], dt), _t(g["B"], dt))
    assert C.dtype == np.uint16 and C.shape == (2, 4)
    assert np.array_equal(C, _hex_bits(g[dt]["C_bits"]))
    ii, jj = np.array([0, 1, 0, 1]), np.array([0, 3, 3, 1])
    assert np.array_equal(oracle.gemm_at(_t(g["A"], dt), _t(g["B"], dt), ii, jj),
                          _hex_bits(g[dt]["C_bits"])[ii, jj])


@pytest.mark.parametrize("dt", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(5, 7, 9), (3, 11, 4), (8, 2, 13)])
def test_gemm_exact_integer_brute_force(dt, shape):
    """C = A @ B on integers in [-8, 8]: every dot product is an exact integer
    (|C| <= 13 * 64), computed here with Python ints, so the only rounding is
    the final one to the 16-bit type, taken from torch's own conversion of the
    exact value (exact in fp32).  bf16 results above 256 do round."""
    M, N, K = shape
    A, B = synthetic.make_gemm_inputs(M, N, K, dt, seed=17 + M, dist="int", scale=8)
    exact = _brute_int(A, B)
    want = torch.tensor(exact, dtype=torch.float32).to(synthetic.DTYPES[dt]).view(torch.int16).numpy().view(np.uint16)
    got = oracle.gemm(A, B)
    assert got.dtype == np.uint16 and got.shape == (M, N)
    assert np.array_equal(got, want)
    ii = np.array([i for i in range(M) for _ in range(N)])
    jj = np.array([j for _ in range(M) for j in range(N)])
    assert np.array_equal(oracle.gemm_at(A, B, ii, jj), want[ii, jj])


# ---------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes(monkeypatch):
    """Plant plausible mistakes in the oracle and check that a pin fails."""
    from oracle import reference as ref

    def fails(fn):
        try:
            fn()
        except AssertionError:
            return True
        return False

    # 1. reversed reduction order
    orig = ref.rank_order_sum
    monkeypatch.setattr(ref, "rank_order_sum", lambda parts: orig(list(parts)[::-1]))
    monkeypatch.setattr(oracle, "all_reduce", lambda X: ref.rank_order_sum(
        [x.numpy().astype(np.float32) for x in X]))
    assert fails(test_rank_order_golden)
    monkeypatch.undo()

    # 2. shards gathered in the wrong order
    orig_g = ref.gather_k
    monkeypatch.setattr(ref, "gather_k", lambda A: orig_g(list(A)[::-1]))
    assert fails(lambda: test_ag_mm_exact_integer_brute_force("f16"))
    monkeypatch.undo()

    # 3. bias added once in total instead of once per rank
    orig_p = ref._partials

    def once(A, B, bias, bias_on_m, rp, dt):
        parts = orig_p(A, B, None, bias_on_m, rp, dt)
        parts[0] = ref._epilogue(parts[0], bias, bias_on_m)
        return parts
    monkeypatch.setattr(ref, "_partials", once)
    assert fails(lambda: test_mm_rs_ar_exact_integer_brute_force("f16"))
    monkeypatch.undo()

    # 4. transposed B operand (square shapes hide it; the pins use non-square)
    orig_acc = ref.accumulate
    monkeypatch.setattr(ref, "accumulate", lambda X, Y: orig_acc(X, Y.T.copy()) if Y.shape[0] == Y.shape[1] else orig_acc(X, Y))
    assert fails(test_golden_fused_small)
    monkeypatch.undo()

    # 5. round-to-nearest with ties away from zero instead of to even
    def away(x32):
        u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32).astype(np.uint64)
        return ((u + np.uint64(0x8000)) >> np.uint64(16)).astype(np.uint16)
    monkeypatch.setattr(ref, "round_bf16_bits", away)
    assert fails(test_rne16_golden_cases)
    monkeypatch.undo()

    # 6. fp16 GEMM inputs taken as bf16: the output rounded to the wrong type
    monkeypatch.setattr(ref, "_dtype_name", lambda t: "bf16")
    assert fails(lambda: test_gemm_golden("f16"))
    assert fails(lambda: test_gemm_exact_integer_brute_force("f16", (5, 7, 9)))
    monkeypatch.undo()

    # 7. the last term of every dot product dropped (an off-by-one K loop)
    monkeypatch.setattr(ref, "accumulate", lambda X, Y: orig_acc(X[:, :-1], Y[:-1, :]))
    assert fails(lambda: test_gemm_golden("bf16"))
    assert fails(lambda: test_gemm_exact_integer_brute_force("bf16", (5, 7, 9)))
    monkeypatch.undo()


def test_all_to_all_golden_and_involution():
    g = _load("all_to_all_small.json")
    X = [torch.tensor(b, dtype=torch.float32) for b in g["buffers"]]
    outs = oracle.all_to_all(X)
    for o, want in zip(outs, g["expected"]):
        assert o.view(np.float32).tolist() == [float(v) for v in want]
    # applying all_to_all twice gives the inputs back (a block transpose)
    Y = synthetic.make_coll_inputs(4, 64, "bf16", seed=91)
    once = [torch.from_numpy(o.copy()).view(torch.bfloat16) for o in oracle.all_to_all(Y)]
    twice = oracle.all_to_all(once)
    for a, b in zip(twice, Y):
        assert np.array_equal(a, b.view(torch.uint8).numpy())


def test_broadcast_matches_gather_block():
    W, count = 4, 40
    X = synthetic.make_coll_inputs(W, count, "f32", seed=92)
    for root in range(W):
        outs = oracle.broadcast(X, root)
        ag = oracle.all_gather(X)
        blk = ag[root * count * 4:(root + 1) * count * 4]
        for o in outs:
            assert np.array_equal(o, blk)
