"""GPU parity at the benchmark workloads' full sizes, in the default launch
configuration the benchmark times.

GEMM outputs: 4096 seeded sample positions (plus the corners and the first /
last row and column of tile (0, 0)) compared with the oracle's value at each
position, max |gpu - oracle| <= 5e-3 * max |oracle| over the sample.
Data-movement outputs (gathered A, the concurrent all-reduce) are compared
bit for bit in full."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gemm_collective_tiles_gb300 import query_status
from gemm_collective_tiles_gb300.runner import ConcurrentProblem, FusedProblem

pytestmark = pytest.mark.gpu

TOL = 5e-3


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_sample(got_bits, want_bits, dt):
    g = oracle.decode16(got_bits, dt)
    w = oracle.decode16(want_bits, dt)
    assert np.isfinite(g).all()
    err = float(np.max(np.abs(g - w)))
    scale = float(np.max(np.abs(w)))
    assert err <= TOL * scale, f"max err {err} vs scale {scale}"


def _run(name):
    wl = synthetic.WORKLOADS[name]
    x = synthetic.make_fused_inputs(**wl)
    prob = FusedProblem(wl["op"], wl["W"], wl["M"], wl["N"], wl["K"], wl["dtype"], bias=wl.get("bias", False))
    prob.upload(x.A, x.B, x.bias)
    prob.poison_outputs()
    prob.run()
    rc = query_status(prob.ws)
    assert rc[0] == 0, rc
    return wl, x, prob


def _gather_sample(prob, view, ii, jj):
    t = view[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()]
    return _bits(t)


def test_mm_rs_w4_4096_sampled():
    wl, x, prob = _run("mm_rs_w4_4096")
    N_l = wl["N"] // wl["W"]
    for r in range(wl["W"]):
        ii, jj = synthetic.sample_indices(wl["M"], N_l, seed=wl["seed"] + 1000 + r)
        ii, jj = ii.numpy(), jj.numpy()
        got = _gather_sample(prob, prob.heap.view(prob.out, r), ii, jj)
        want = oracle.matmul_reduce_scatter_at(x.A, x.B, x.bias, r, ii, jj)
        _check_sample(got, want, wl["dtype"])


def _check_gathered_full(prob, wl):
    """gathered A, block s == shard s, bit for bit (compared on the device)."""
    W, K_l = wl["W"], wl["K"] // wl["W"]
    g = prob.heap.view(prob.gathered, 0).view(torch.int16)
    for s in range(W):
        shard = prob.heap.view(prob.A, s).view(torch.int16)
        assert torch.equal(g[:, s * K_l:(s + 1) * K_l], shard), f"shard {s}"


def test_ag_mm_w8_4096x14336x4096_sampled():
    wl, x, prob = _run("ag_mm_w8_4096x14336x4096")
    _check_gathered_full(prob, wl)
    # the gathered buffer also matches the oracle's gather on sampled rows
    ii, jj = synthetic.sample_indices(wl["M"], wl["N"], seed=wl["seed"] + 1000)
    ii, jj = ii.numpy(), jj.numpy()
    got = _gather_sample(prob, prob.heap.view(prob.out, 0), ii, jj)
    want = oracle.all_gather_matmul_at(x.A, x.B[0], x.bias, ii, jj)
    _check_sample(got, want, wl["dtype"])


def test_mm_ag_w8_4096x14336x4096_sampled():
    wl, x, prob = _run("mm_ag_w8_4096x14336x4096")
    ii, jj = synthetic.sample_indices(wl["M"], wl["N"], seed=wl["seed"] + 1001)
    ii, jj = ii.numpy(), jj.numpy()
    got = _gather_sample(prob, prob.heap.view(prob.out, 0), ii, jj)
    want = oracle.matmul_all_gather_at(x.A, x.B[0], x.bias, ii, jj)
    _check_sample(got, want, wl["dtype"])


def test_mm_ar_w8_8192_sampled():
    wl, x, prob = _run("mm_ar_w8_8192")
    ii, jj = synthetic.sample_indices(wl["M"], wl["N"], seed=wl["seed"] + 1000)
    ii, jj = ii.numpy(), jj.numpy()
    got = _gather_sample(prob, prob.heap.view(prob.out, 0), ii, jj)
    want = oracle.matmul_all_reduce_at(x.A, x.B, x.bias, ii, jj)
    _check_sample(got, want, wl["dtype"])


def test_concurrent_gemm_8192_allreduce_w8_64mi():
    """GEMM sampled; the all-reduce over 8 x 64Mi fp32, in place, bit for bit."""
    cw = synthetic.CONCURRENT_WORKLOAD
    A, B = synthetic.make_gemm_inputs(cw["M"], cw["N"], cw["K"], cw["gemm_dtype"], cw["gemm_seed"],
                                      dist="normal", scale=1.0)
    X = synthetic.make_coll_inputs(cw["W"], cw["count"], cw["coll_dtype"], cw["coll_seed"])
    prob = ConcurrentProblem(cw["M"], cw["N"], cw["K"], cw["gemm_dtype"], "all_reduce", cw["W"], cw["count"],
                             in_place=True)
    prob.upload(A, B, X)
    prob.poison_outputs()
    prob.run()
    assert query_status(prob.ws)[0] == 0
    want = oracle.all_reduce(X).view(np.uint32)
    for r in range(cw["W"]):
        got = prob.heap.view(prob.x_out, r).cpu().numpy().view(np.uint32)
        assert np.array_equal(got, want), f"rank {r}"
    ii, jj = synthetic.sample_indices(cw["M"], cw["N"], seed=cw["gemm_seed"] + 1000)
    ii, jj = ii.numpy(), jj.numpy()
    got = _bits(prob.C[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()])
    _check_sample(got, oracle.gemm_at(A, B, ii, jj), cw["gemm_dtype"])


@pytest.mark.slow
def test_ag_mm_w8_131072x16384x16384_sampled():
    wl, x, prob = _run("ag_mm_w8_131072x16384x16384")
    _check_gathered_full(prob, wl)
    ii, jj = synthetic.sample_indices(wl["M"], wl["N"], seed=wl["seed"] + 1000)
    ii, jj = ii.numpy(), jj.numpy()
    got = _gather_sample(prob, prob.heap.view(prob.out, 0), ii, jj)
    want = oracle.all_gather_matmul_at(x.A, x.B[0], x.bias, ii, jj)
    _check_sample(got, want, wl["dtype"])
