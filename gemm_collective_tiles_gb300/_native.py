"""ctypes binding of the C ABI in include/gemm_collective_tiles.h.

Argument marshalling only: every entry point here forwards to the shared
library built from ``csrc/`` (``build.py``).  Importing this module builds the
library when its sources are newer than it and raises if it cannot be built
or loaded -- there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

IRIS_OK = 0
IRIS_EINVAL = -1
IRIS_EALIGN = -2
IRIS_ENOWS = -3
IRIS_ECUDA = -4
IRIS_ETIMEOUT = -5
IRIS_EUNSUPPORTED = -6
IRIS_NO_BIAS = ctypes.c_size_t(-1).value
IRIS_MAX_WORLD = 16
IRIS_NOALLOC_MAX_FLAGS = 16384
IRIS_NOALLOC_SCRATCH_BYTES = 256 + 8 * IRIS_NOALLOC_MAX_FLAGS

IRIS_F16, IRIS_BF16, IRIS_F32 = 0, 1, 2
IRIS_COLL_ALL_GATHER, IRIS_COLL_ALL_REDUCE, IRIS_COLL_REDUCE_SCATTER = 0, 1, 2
IRIS_COLL_ALL_TO_ALL, IRIS_COLL_BROADCAST = 3, 4
(IRIS_OP_ALL_GATHER_MATMUL, IRIS_OP_MATMUL_REDUCE_SCATTER, IRIS_OP_MATMUL_ALL_GATHER,
 IRIS_OP_MATMUL_ALL_REDUCE, IRIS_OP_CONCURRENT) = range(5)

# every function the header declares (checked by the CPU export test)
EXPORTS = (
    "iris_b200_workspace_size",
    "iris_b200_all_gather_matmul",
    "iris_b200_all_gather_matmul_noalloc",
    "iris_b200_matmul_reduce_scatter",
    "iris_b200_matmul_all_gather",
    "iris_b200_matmul_all_reduce",
    "iris_b200_concurrent_gemm_collective",
    "iris_b200_concurrent_two_stream",
    "iris_b200_sm_partition_streams",
    "iris_b200_sm_partition_release",
    "iris_b200_query_status",
    "iris_b200_strerror",
    "iris_b200_num_sms",
)


class iris_b200_config(ctypes.Structure):
    _fields_ = [
        ("tile_m", ctypes.c_int),
        ("tile_n", ctypes.c_int),
        ("tile_k", ctypes.c_int),
        ("group_m", ctypes.c_int),
        ("gemm_ctas", ctypes.c_int),
        ("stages", ctypes.c_int),
        ("comm_block", ctypes.c_int),
        ("replicate_outputs", ctypes.c_int),
        ("bias_on_m", ctypes.c_int),
        ("grid", ctypes.c_int),
        ("wait_ns", ctypes.c_ulonglong),
        ("debug_skip_flag", ctypes.c_int),
        ("trace_buf", ctypes.c_ulonglong),
        ("trace_cap", ctypes.c_int),
        ("reduce_mode", ctypes.c_int),
        ("root", ctypes.c_int),
        ("rank_inner", ctypes.c_int),
        ("coll_ring", ctypes.c_int),
        ("coll_l2_hint", ctypes.c_int),
        ("coll_path", ctypes.c_int),
        ("gather_parts", ctypes.c_int),
        ("startup_gather", ctypes.c_int),
        ("gemm_l2_hint", ctypes.c_int),
        ("out_l2_hint", ctypes.c_int),
        ("sum_l2_hint", ctypes.c_int),
        ("k_split", ctypes.c_int),
        ("coll_out_stage", ctypes.c_int),
    ]


class iris_b200_heap(ctypes.Structure):
    _fields_ = [
        ("base", ctypes.c_void_p),
        ("rank_stride", ctypes.c_size_t),
        ("world", ctypes.c_int),
    ]


_lib = None


def _declare(lib):
    P = ctypes.POINTER
    i64, sz, vp, ci = ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int
    cfgp, heapp = P(iris_b200_config), P(iris_b200_heap)
    sig = {
        "iris_b200_workspace_size": (ci, [ci, i64, i64, i64, ci, ci, cfgp, P(sz)]),
        "iris_b200_all_gather_matmul": (ci, [heapp, sz, sz, sz, sz, sz, i64, i64, i64, ci, cfgp, vp, sz, vp]),
        "iris_b200_all_gather_matmul_noalloc": (ci, [heapp, sz, sz, sz, sz, sz, i64, i64, i64, ci, cfgp, vp]),
        "iris_b200_matmul_reduce_scatter": (ci, [heapp, sz, sz, sz, sz, i64, i64, i64, ci, cfgp, vp, sz, vp]),
        "iris_b200_matmul_all_gather": (ci, [heapp, sz, sz, sz, sz, i64, i64, i64, ci, cfgp, vp, sz, vp]),
        "iris_b200_matmul_all_reduce": (ci, [heapp, sz, sz, sz, sz, i64, i64, i64, ci, cfgp, vp, sz, vp]),
        "iris_b200_concurrent_gemm_collective": (
            ci, [vp, vp, vp, i64, i64, i64, ci, ci, heapp, sz, sz, i64, ci, cfgp, vp, sz, vp]),
        "iris_b200_concurrent_two_stream": (
            ci, [vp, vp, vp, i64, i64, i64, ci, ci, heapp, sz, sz, i64, ci, cfgp, vp, sz, vp, sz, vp, vp]),
        "iris_b200_sm_partition_streams": (ci, [ci, P(vp), P(vp), P(ci), P(ci)]),
        "iris_b200_sm_partition_release": (ci, []),
        "iris_b200_query_status": (ci, [vp, vp, P(ci), P(ci), P(ci)]),
        "iris_b200_strerror": (ctypes.c_char_p, [ci]),
        "iris_b200_num_sms": (ci, [P(ci)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def lib_path() -> str:
    return _build.lib_path()


def load():
    """Build (if stale) and load the shared library; cached."""
    global _lib
    if _lib is None:
        path = _build.build()
        if not os.path.exists(path):
            raise ImportError(f"native library missing: {path}")
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib = lib
    return _lib


def strerror(code: int) -> str:
    return load().iris_b200_strerror(int(code)).decode()


class IrisError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")
        self.code = code


def check(fn: str, code: int) -> int:
    if code != IRIS_OK:
        raise IrisError(fn, code)
    return code


# Same-name thin wrappers (raw codes returned, no checking).
def iris_b200_workspace_size(op, M, N, K, world, dtype, cfg, bytes_out):
    return load().iris_b200_workspace_size(op, M, N, K, world, dtype, cfg, bytes_out)


def iris_b200_all_gather_matmul(*args):
    return load().iris_b200_all_gather_matmul(*args)


def iris_b200_all_gather_matmul_noalloc(*args):
    return load().iris_b200_all_gather_matmul_noalloc(*args)


def iris_b200_matmul_reduce_scatter(*args):
    return load().iris_b200_matmul_reduce_scatter(*args)


def iris_b200_matmul_all_gather(*args):
    return load().iris_b200_matmul_all_gather(*args)


def iris_b200_matmul_all_reduce(*args):
    return load().iris_b200_matmul_all_reduce(*args)


def iris_b200_concurrent_gemm_collective(*args):
    return load().iris_b200_concurrent_gemm_collective(*args)


def iris_b200_concurrent_two_stream(*args):
    return load().iris_b200_concurrent_two_stream(*args)


def iris_b200_query_status(*args):
    return load().iris_b200_query_status(*args)


def iris_b200_strerror(code):
    return load().iris_b200_strerror(code)


def iris_b200_num_sms(n_out):
    return load().iris_b200_num_sms(n_out)
