"""The C ABI library builds for sm_103a, loads, exports every entry point the
header declares, and rejects bad arguments before touching the GPU.  CPU only."""
import ctypes
import os
import re
import subprocess

import pytest

import gemm_collective_tiles_gb300 as gct
from gemm_collective_tiles_gb300 import _native as N

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm_collective_tiles.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(iris_b200_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = N.load()
    names = _declared()
    assert set(names) == set(N.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", N.lib_path()], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (iris_b200_\w+)", out.stdout))
    assert exported == set(names)


def test_strerror_and_codes():
    for code in (0, -1, -2, -3, -4, -5, -6, 123):
        assert isinstance(N.strerror(code), str) and N.strerror(code)
    assert N.strerror(N.IRIS_ETIMEOUT).startswith("a bounded")


def test_workspace_size_layout():
    lib = N.load()
    out = ctypes.c_size_t(0)
    # all_gather_matmul: header + W * m_blocks 8-byte ready counters
    assert lib.iris_b200_workspace_size(N.IRIS_OP_ALL_GATHER_MATMUL, 4096, 14336, 4096, 8, N.IRIS_BF16,
                                        None, ctypes.byref(out)) == 0
    assert out.value == 256 + ((8 * 32 * 8 + 255) // 256) * 256
    # reduce-scatter, default (chained) schedule: flags / tile counters + one
    # fp32 running sum of M x N
    assert lib.iris_b200_workspace_size(N.IRIS_OP_MATMUL_REDUCE_SCATTER, 4096, 4096, 4096, 4, N.IRIS_F16,
                                        None, ctypes.byref(out)) == 0
    flags = 4 * 32 * 16 * 4
    assert out.value == 256 + flags + 4096 * 4096 * 4
    # queue and parts schedules keep one fp32 partial per rank
    for mode in (1, 2):
        cfg = gct.make_config(reduce_mode=mode)
        assert lib.iris_b200_workspace_size(N.IRIS_OP_MATMUL_REDUCE_SCATTER, 4096, 4096, 4096, 4, N.IRIS_F16,
                                            ctypes.byref(cfg), ctypes.byref(out)) == 0
        assert out.value == 256 + flags + 4 * 4096 * 4096 * 4
    # chained needs whole 32-column slices: N/W = 8 does not qualify -> parts
    assert lib.iris_b200_workspace_size(N.IRIS_OP_MATMUL_REDUCE_SCATTER, 64, 32, 64, 4, N.IRIS_F16,
                                        None, ctypes.byref(out)) == 0
    assert out.value == 256 + 256 + 4 * 64 * 32 * 4
    cfg = gct.make_config(reduce_mode=3)
    assert lib.iris_b200_workspace_size(N.IRIS_OP_MATMUL_REDUCE_SCATTER, 64, 32, 64, 4, N.IRIS_F16,
                                        ctypes.byref(cfg), ctypes.byref(out)) == N.IRIS_EINVAL
    cfg = gct.make_config(tile_n=128)
    assert lib.iris_b200_workspace_size(N.IRIS_OP_MATMUL_ALL_REDUCE, 256, 256, 64, 2, N.IRIS_F16,
                                        ctypes.byref(cfg), ctypes.byref(out)) == 0
    assert out.value == 256 + 256 + 256 * 256 * 4
    assert lib.iris_b200_workspace_size(N.IRIS_OP_CONCURRENT, 8192, 8192, 8192, 8, N.IRIS_BF16,
                                        None, ctypes.byref(out)) == 0
    assert out.value == 256
    # bad arguments
    assert lib.iris_b200_workspace_size(N.IRIS_OP_CONCURRENT, -1, 8, 8, 1, 0, None, ctypes.byref(out)) == N.IRIS_EINVAL
    assert lib.iris_b200_workspace_size(N.IRIS_OP_CONCURRENT, 8, 8, 8, 0, 0, None, ctypes.byref(out)) == N.IRIS_EINVAL
    assert lib.iris_b200_workspace_size(N.IRIS_OP_CONCURRENT, 8, 8, 8, 17, 0, None, ctypes.byref(out)) == N.IRIS_EINVAL
    assert lib.iris_b200_workspace_size(9, 8, 8, 8, 1, 0, None, ctypes.byref(out)) == N.IRIS_EINVAL
    assert lib.iris_b200_workspace_size(0, 8, 8, 8, 1, 0, None, None) == N.IRIS_EINVAL
    bad = gct.make_config(tile_n=96)
    assert lib.iris_b200_workspace_size(0, 8, 8, 8, 1, 0, ctypes.byref(bad), ctypes.byref(out)) == N.IRIS_EINVAL
    for stages in (1, 4, 5, 7):   # CTA-pair pipelines: 3 or 6 stages (0 = by K)
        bad = gct.make_config(stages=stages)
        assert lib.iris_b200_workspace_size(0, 8, 8, 8, 1, 0, ctypes.byref(bad), ctypes.byref(out)) == N.IRIS_EINVAL
    for stages in (0, 3, 6):
        ok = gct.make_config(stages=stages)
        assert lib.iris_b200_workspace_size(0, 8, 8, 8, 1, 0, ctypes.byref(ok), ctypes.byref(out)) == N.IRIS_OK


def _heap(world=2, stride=1 << 20, base=1 << 20):
    return N.iris_b200_heap(base, stride, world)


def test_argument_checks_before_any_gpu_work():
    lib = N.load()
    h = _heap()
    hp = ctypes.byref(h)
    # null heap
    assert lib.iris_b200_all_gather_matmul(None, 0, 0, N.IRIS_NO_BIAS, 0, 0, 8, 8, 16, 0, None, None, 0, None) == N.IRIS_EINVAL
    # world out of range
    bad = _heap(world=0)
    assert lib.iris_b200_matmul_all_reduce(ctypes.byref(bad), 0, 0, N.IRIS_NO_BIAS, 0, 8, 8, 8, 0, None, None, 0, None) == N.IRIS_EINVAL
    # misaligned heap stride / base
    bad = _heap(stride=(1 << 20) + 8)
    assert lib.iris_b200_matmul_all_reduce(ctypes.byref(bad), 0, 0, N.IRIS_NO_BIAS, 0, 8, 8, 8, 0, None, None, 0, None) == N.IRIS_EALIGN
    bad = _heap(base=(1 << 20) + 4)
    assert lib.iris_b200_matmul_all_reduce(ctypes.byref(bad), 0, 0, N.IRIS_NO_BIAS, 0, 8, 8, 8, 0, None, None, 0, None) == N.IRIS_EALIGN
    # K not divisible by W; K_local not a multiple of 8; N not a multiple of 8
    assert lib.iris_b200_all_gather_matmul(hp, 0, 0, N.IRIS_NO_BIAS, 0, 0, 8, 8, 15, 0, None, None, 0, None) == N.IRIS_EINVAL
    assert lib.iris_b200_all_gather_matmul(hp, 0, 0, N.IRIS_NO_BIAS, 0, 0, 8, 8, 12, 0, None, None, 0, None) == N.IRIS_EALIGN
    assert lib.iris_b200_all_gather_matmul(hp, 0, 0, N.IRIS_NO_BIAS, 0, 0, 8, 12, 16, 0, None, None, 0, None) == N.IRIS_EALIGN
    # unsupported dtype for a GEMM operand
    assert lib.iris_b200_all_gather_matmul(hp, 0, 0, N.IRIS_NO_BIAS, 0, 0, 8, 8, 16, 2, None, None, 0, None) == N.IRIS_EINVAL
    # reduce-scatter: N not divisible by W, N/W not a multiple of 8
    assert lib.iris_b200_matmul_reduce_scatter(hp, 0, 0, N.IRIS_NO_BIAS, 0, 8, 12, 8, 0, None, None, 0, None) in (N.IRIS_EINVAL, N.IRIS_EALIGN)
    assert lib.iris_b200_matmul_reduce_scatter(hp, 0, 0, N.IRIS_NO_BIAS, 0, 8, 8, 8, 0, None, None, 0, None) == N.IRIS_EALIGN
    # all-gather along M: M not divisible by W
    assert lib.iris_b200_matmul_all_gather(hp, 0, 0, N.IRIS_NO_BIAS, 0, 7, 8, 8, 0, None, None, 0, None) == N.IRIS_EINVAL
    # negative sizes
    assert lib.iris_b200_matmul_all_reduce(hp, 0, 0, N.IRIS_NO_BIAS, 0, -8, 8, 8, 0, None, None, 0, None) == N.IRIS_EINVAL
    # concurrent: misaligned GEMM pointer, bad collective sizes
    assert lib.iris_b200_concurrent_gemm_collective(8, 16, 32, 8, 8, 8, 0, 1, None, 0, 0, 0, 2, None, None, 0, None) == N.IRIS_EALIGN
    assert lib.iris_b200_concurrent_gemm_collective(None, None, None, 0, 0, 0, 0, 1, hp, 0, 0, 3, 2, None, None, 0, None) == N.IRIS_EALIGN
    assert lib.iris_b200_concurrent_gemm_collective(None, None, None, 0, 0, 0, 0, 1, hp, 0, 0, 8, 1, None, None, 0, None) == N.IRIS_EUNSUPPORTED
    assert lib.iris_b200_concurrent_gemm_collective(None, None, None, 0, 0, 0, 0, 7, hp, 0, 0, 8, 2, None, None, 0, None) == N.IRIS_EINVAL
    assert lib.iris_b200_concurrent_gemm_collective(None, None, None, 0, 0, 0, 0, 2, hp, 0, 0, 12, 2, None, None, 0, None) == N.IRIS_EALIGN
    # query_status needs a workspace
    assert lib.iris_b200_query_status(None, None, None, None, None) == N.IRIS_EINVAL
    # the SM partition needs somewhere to put its streams
    assert lib.iris_b200_sm_partition_streams(80, None, None, None, None) == N.IRIS_EINVAL


def test_config_builder_rejects_unknown_keys():
    c = gct.make_config(tile_n=128, gemm_ctas=-1, wait_ns=10**6)
    assert c.tile_n == 128 and c.gemm_ctas == -1 and c.wait_ns == 10**6
    with pytest.raises(KeyError):
        gct.make_config(bogus=1)


def test_ctypes_structs_match_the_c_header(tmp_path):
    """Compile a probe against the header with the host C compiler and compare
    every field offset and the struct sizes with the ctypes mirrors."""
    fields = [f[0] for f in N.iris_b200_config._fields_]
    src = ['#include <stdio.h>', '#include <stddef.h>', '#include "gemm_collective_tiles.h"', 'int main(void) {',
           'printf("cfg %zu\\n", sizeof(iris_b200_config));', 'printf("heap %zu\\n", sizeof(iris_b200_heap));']
    for f in fields:
        src.append(f'printf("{f} %zu\\n", offsetof(iris_b200_config, {f}));')
    for f in ("base", "rank_stride", "world"):
        src.append(f'printf("heap.{f} %zu\\n", offsetof(iris_b200_heap, {f}));')
    # every numeric constant the binding mirrors, as the C compiler sees it
    consts = [n for n in dir(N) if n.startswith("IRIS_") and isinstance(getattr(N, n), int)]
    for n in consts:
        src.append(f'printf("const.{n} %lld\\n", (long long)({n}));')
    src.append("return 0; }")
    c = tmp_path / "probe.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "probe"
    cuda_inc = "/usr/local/cuda/include"
    r = subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(c), "-o", str(exe)],
                       capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("no host C compiler with the CUDA headers: " + r.stderr[:200])
    out = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True).stdout.splitlines())
    assert int(out["cfg"]) == ctypes.sizeof(N.iris_b200_config)
    assert int(out["heap"]) == ctypes.sizeof(N.iris_b200_heap)
    for f in fields:
        assert int(out[f]) == getattr(N.iris_b200_config, f).offset, f
    for f in ("base", "rank_stride", "world"):
        assert int(out["heap." + f]) == getattr(N.iris_b200_heap, f).offset, f
    for n in consts:
        want = getattr(N, n)
        got = int(out["const." + n])
        assert got == want or got == want - (1 << 64), n


def test_split_k_workspace():
    """all_gather_matmul above K = 32768 splits K by default (chunks of about
    16384) and its workspace then holds one 8-byte chained-reduce counter per
    tile after the gather counters, and an M x N fp32 running sum; k_split 1
    (or one-CTA tiles) leaves the workspace as without the split."""
    lib = N.load()
    out = ctypes.c_size_t(0)
    W, M, Nn, K = 8, 16384, 16384, 131072
    mb, nb = M // 128, Nn // 256
    assert lib.iris_b200_workspace_size(N.IRIS_OP_ALL_GATHER_MATMUL, M, Nn, K, W, N.IRIS_BF16, None,
                                        ctypes.byref(out)) == 0
    flags = (2 * W * mb + 2 * mb * nb) * 4
    assert out.value == 256 + ((flags + 255) // 256) * 256 + M * Nn * 4
    for cfg in (gct.make_config(k_split=1), gct.make_config(tile_m=128)):
        assert lib.iris_b200_workspace_size(N.IRIS_OP_ALL_GATHER_MATMUL, M, Nn, K, W, N.IRIS_BF16,
                                            ctypes.byref(cfg), ctypes.byref(out)) == 0
        assert out.value == 256 + ((2 * W * mb * 4 + 255) // 256) * 256
    # K = 32768: no split by default; an explicit k_split asks for it
    assert lib.iris_b200_workspace_size(N.IRIS_OP_ALL_GATHER_MATMUL, 256, 256, 32768, W, N.IRIS_BF16, None,
                                        ctypes.byref(out)) == 0
    assert out.value == 256 + 256
    cfg = gct.make_config(k_split=4)
    assert lib.iris_b200_workspace_size(N.IRIS_OP_ALL_GATHER_MATMUL, 256, 256, 32768, W, N.IRIS_BF16,
                                        ctypes.byref(cfg), ctypes.byref(out)) == 0
    assert out.value == 256 + 256 + 256 * 256 * 4
    # N not a multiple of 32: the chained reduce does not apply, no split
    assert lib.iris_b200_workspace_size(N.IRIS_OP_ALL_GATHER_MATMUL, 256, 264, 131072, W, N.IRIS_BF16, None,
                                        ctypes.byref(out)) == 0
    assert out.value == 256 + 256
    bad = gct.make_config(k_split=-1)
    assert lib.iris_b200_workspace_size(N.IRIS_OP_ALL_GATHER_MATMUL, 256, 256, 65536, W, N.IRIS_BF16,
                                        ctypes.byref(bad), ctypes.byref(out)) == N.IRIS_EINVAL


def test_split_k_workspace_matmul_all_gather():
    """matmul_all_gather needs no workspace beyond the header unless it
    splits K; then one 8-byte counter per (rank, 128-row block, tile column)
    and a running sum of all W x M_l rows."""
    lib = N.load()
    out = ctypes.c_size_t(0)
    W, M, Nn, K = 4, 4 * 1024, 1024, 65536
    assert lib.iris_b200_workspace_size(N.IRIS_OP_MATMUL_ALL_GATHER, M, Nn, K, W, N.IRIS_BF16, None,
                                        ctypes.byref(out)) == 0
    flags = 2 * W * (1024 // 128) * (Nn // 256) * 4
    assert out.value == ((256 + flags + 255) // 256) * 256 + M * Nn * 4
    cfg = gct.make_config(k_split=1)
    assert lib.iris_b200_workspace_size(N.IRIS_OP_MATMUL_ALL_GATHER, M, Nn, K, W, N.IRIS_BF16, ctypes.byref(cfg),
                                        ctypes.byref(out)) == 0
    assert out.value == 256
