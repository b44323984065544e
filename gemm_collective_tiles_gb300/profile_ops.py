"""Run one benchmark workload's fused kernel a few times (for an ncu capture).

    python -m gemm_collective_tiles_gb300.profile_ops WORKLOAD [LAUNCHES] [CONFIG_JSON]

WORKLOAD is a fused-op workload name of ``synthetic.WORKLOADS``,
``concurrent_ar_w8`` or ``gemm_bf16_8192`` (the concurrent workload's GEMM
alone), with inputs drawn as the benchmark draws them; or an
all_gather_matmul shape ``ag_mm_w<W>_<M>x<N>x<K>`` (bf16, N(0, 0.02) drawn on
the device, as the shape sweep draws them).  CONFIG_JSON (fused ops) is a
dict of ``iris_b200_config`` fields.  Used by the profiling commands recorded
under ``profiles/``.
"""
from __future__ import annotations

import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


def main(argv):
    import json

    import torch

    import synthetic
    from gemm_collective_tiles_gb300 import query_status
    from gemm_collective_tiles_gb300.runner import ConcurrentProblem, FusedProblem
    name = argv[0]
    launches = int(argv[1]) if len(argv) > 1 else 6
    cfg = json.loads(argv[2]) if len(argv) > 2 else None
    torch.cuda.set_device(0)
    if name in ("concurrent_ar_w8", "gemm_bf16_8192"):
        cw = synthetic.CONCURRENT_WORKLOAD
        coll = name == "concurrent_ar_w8"
        A, B = synthetic.make_gemm_inputs(cw["M"], cw["N"], cw["K"], cw["gemm_dtype"], cw["gemm_seed"],
                                          dist="normal", scale=1.0)
        X = synthetic.make_coll_inputs(cw["W"], cw["count"], cw["coll_dtype"], cw["coll_seed"]) if coll else None
        prob = ConcurrentProblem(cw["M"], cw["N"], cw["K"], cw["gemm_dtype"], "all_reduce", cw["W"],
                                 cw["count"] if coll else 0, coll_dtype=cw["coll_dtype"])
        prob.upload(A, B, X)
    elif name not in synthetic.WORKLOADS and name.startswith("ag_mm_w"):
        w_part, shape = name[len("ag_mm_w"):].split("_", 1)
        W = int(w_part)
        M, N, K = (int(v) for v in shape.split("x"))
        prob = FusedProblem("ag_mm", W, M, N, K, "bf16", config=cfg)
        for r in range(W):
            synthetic.fill_device_(prob.heap.view(prob.A, r), 7 + r)
        synthetic.fill_device_(prob.heap.view(prob.B, 0), 99)
    else:
        wl = synthetic.WORKLOADS[name]
        x = synthetic.make_fused_inputs(**wl)
        prob = FusedProblem(wl["op"], wl["W"], wl["M"], wl["N"], wl["K"], wl["dtype"], bias=wl.get("bias", False),
                            config=cfg)
        prob.upload(x.A, x.B, x.bias)
    for _ in range(launches):
        prob.run()
    torch.cuda.synchronize()
    rc = query_status(prob.ws)
    if rc[0] != 0:
        raise RuntimeError(f"device status {rc}")
    print(f"{name}: {launches} launches ok")
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
