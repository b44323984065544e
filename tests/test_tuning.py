"""Config selection: JSON cache round trip, atomic writes, stable keys, and
tuning that always measures the static default and never ends worse.  CPU."""
import json
import os

import pytest

from gemm_collective_tiles_gb300 import tuning


def test_keys_are_stable_strings():
    a = tuning.arch_key("NVIDIA GB300 ", 152, (10, 3))
    assert a == "NVIDIA GB300|sm_103|152sm"
    assert tuning.shape_key("matmul_reduce_scatter", 4, 4096, 4096, 4096, "f16") == \
        "matmul_reduce_scatter|W4|4096x4096x4096|f16"


def test_cache_round_trip_and_atomic_write(tmp_path):
    path = str(tmp_path / "sub" / "tuning.json")
    assert tuning.lookup("a", "k", path) is None
    assert tuning.record("a", "k", {"group_m": 16, "not_a_knob": 1}, 1.0, 2.0, path)
    assert tuning.lookup("a", "k", path) == {"group_m": 16}
    # no temporary files left behind, valid JSON on disk
    assert sorted(os.listdir(tmp_path / "sub")) == ["tuning.json"]
    json.load(open(path))
    # a second key keeps the first
    tuning.record("a", "k2", {"tile_n": 128}, 1.0, 1.0, path)
    assert tuning.lookup("a", "k", path) == {"group_m": 16}
    assert tuning.lookup("b", "k", path) is None


def test_corrupt_cache_reads_as_empty(tmp_path):
    path = tmp_path / "tuning.json"
    path.write_text("{not json")
    assert tuning.load_db(str(path)) == {}
    assert tuning.select("a", "k", None, str(path)) == {}


def test_tune_measures_default_and_never_loses(tmp_path):
    path = str(tmp_path / "t.json")
    times = {json.dumps({}): 5.0, json.dumps({"group_m": 16}): 4.0, json.dumps({"tile_n": 128}): 6.0}
    seen = []

    def measure(cfg):
        seen.append(cfg)
        if cfg == {"group_m": 64}:
            raise RuntimeError("rejected by the library")
        return times[json.dumps(cfg, sort_keys=True)]

    res = tuning.tune(measure, [{"group_m": 16}, {"tile_n": 128}, {"group_m": 64}], "a", "k", path)
    assert {} in seen                       # the static default is always measured
    assert res["config"] == {"group_m": 16} and res["ms"] == 4.0 and res["default_ms"] == 5.0
    assert res["tried"] == 3
    assert tuning.select("a", "k", None, path) == {"group_m": 16}
    # when nothing beats the default, the default wins
    res = tuning.tune(lambda c: 1.0 if c == {} else 2.0, [{"group_m": 8}], "a", "k3", path)
    assert res["config"] == {} and tuning.select("a", "k3", None, path) == {}
    # explicit configs win over the cache
    assert tuning.select("a", "k", {"tile_n": 128}, path) == {"tile_n": 128}


def test_candidates():
    c = tuning.candidates("concurrent", 8, 8192, 8192, 8192, 152, top_k=50)
    assert c[0] == {}
    assert any("gemm_ctas" in x for x in c)
    assert len({json.dumps(x, sort_keys=True) for x in c}) == len(c)
    r = tuning.candidates("matmul_reduce_scatter", 4, 4096, 4096, 4096, 152, top_k=50)
    assert {"reduce_mode": 1} in r and {"reduce_mode": 2} in r
    assert len(tuning.candidates("all_gather_matmul", 8, 4096, 14336, 4096, 152, top_k=3)) == 3
    # the CTA-pair pipeline the default does not pick for the K one item runs
    # is tried early: every fused op splits K above 32768 into chunks of
    # ~16384 (so the three-stage default) when N is a multiple of 32
    short_k = tuning.candidates("all_gather_matmul", 8, 4096, 14336, 4096, 152, top_k=3)
    split_k = tuning.candidates("all_gather_matmul", 8, 16384, 16384, 131072, 152, top_k=3)
    for op in ("matmul_all_reduce", "matmul_reduce_scatter", "matmul_all_gather"):
        assert tuning.candidates(op, 8, 4096, 4096, 131072, 152, top_k=3)[1] == {"k_split": 1}
    long_k = tuning.candidates("matmul_all_gather", 8, 4096, 4104, 131072, 152, top_k=3)
    assert {"stages": 6} in short_k and {"stages": 3} not in short_k
    assert {"k_split": 1} in split_k and {"stages": 6} in split_k and {"stages": 3} not in split_k
    assert {"stages": 3} in long_k and {"stages": 6} not in long_k
    # unsplit all_gather_matmul with a long K (N not a multiple of 32)
    odd_n = tuning.candidates("all_gather_matmul", 8, 4096, 4104, 131072, 152, top_k=3)
    assert {"stages": 3} in odd_n and not any("k_split" in c for c in odd_n)
    # start-up gathers by the worker threads (the default up to 16384 rows is
    # the TMA producer): tried where the default differs
    assert {"startup_gather": 1} in tuning.candidates("all_gather_matmul", 8, 4096, 4096, 4096, 152)
    assert {"startup_gather": 1} in tuning.candidates("all_gather_matmul", 8, 16384, 16384, 131072, 152)
    assert not any("startup_gather" in c for c in tuning.candidates("all_gather_matmul", 8, 131072, 16384, 16384, 152))
    assert not any("startup_gather" in c for c in tuning.candidates("matmul_all_gather", 8, 4096, 4096, 4096, 152))
    # unsplit long K (N not a multiple of 32): the workers are the default there
    assert not any("startup_gather" in c for c in tuning.candidates("all_gather_matmul", 8, 4096, 4104, 131072, 152))


def test_all_tuned_knobs_exist_in_the_config_struct():
    from gemm_collective_tiles_gb300 import _native
    names = {f[0] for f in _native.iris_b200_config._fields_}
    assert set(tuning.TUNABLE) <= names


def test_concurrent_key_names_the_collective_and_its_size():
    k1 = tuning.shape_key("concurrent", 8, 8192, 8192, 8192, "bf16", "all_reduce", 64 << 20, "f32")
    k2 = tuning.shape_key("concurrent", 8, 8192, 8192, 8192, "bf16", "all_gather", 1 << 20, "f32")
    k3 = tuning.shape_key("concurrent", 8, 8192, 8192, 8192, "bf16", "all_reduce", 1 << 20, "f32")
    assert k1 == "concurrent|W8|8192x8192x8192|bf16|all_reduce|count67108864|f32"
    assert len({k1, k2, k3}) == 3
    # the fused ops' keys are unchanged
    assert tuning.shape_key("all_gather_matmul", 8, 4096, 14336, 4096, "bf16") == \
        "all_gather_matmul|W8|4096x14336x4096|bf16"


def _rec(path, op, M, N, K, cfg, ms, dms, W=8, dtype="bf16", **kw):
    shape = tuning.shape_info(op, W, M, N, K, dtype, **kw)
    key = tuning.shape_key(op, W, M, N, K, dtype, **kw)
    assert tuning.record("a", key, cfg, ms, dms, path, shape)


def test_nearest_shape_exact_nearest_and_none(tmp_path):
    path = str(tmp_path / "t.json")
    _rec(path, "all_gather_matmul", 4096, 14336, 4096, {"group_m": 16}, 1.0, 1.2)   # beat its default
    _rec(path, "all_gather_matmul", 8192, 8192, 8192, {"group_m": 64}, 2.0, 2.0)    # default won: no info
    _rec(path, "all_gather_matmul", 65536, 16384, 16384, {"stages": 6}, 30.0, 31.0)

    def sel(M, N, K, W=8, dtype="bf16", op="all_gather_matmul"):
        return tuning.select("a", tuning.shape_key(op, W, M, N, K, dtype), path=path,
                             shape=tuning.shape_info(op, W, M, N, K, dtype))

    assert sel(4096, 14336, 4096) == {"group_m": 16}                # exact
    assert sel(4096, 11008, 4096) == {"group_m": 16}                # 0.38 log2 away
    assert sel(131072, 16384, 16384) == {"stages": 6}               # one size x2
    assert sel(8192, 8192, 8192) == {"group_m": 64}                 # exact match is not filtered
    assert sel(8192, 8192, 16384) == {}                             # nearest lost to its default
    assert sel(1024, 1024, 1024) == {}                              # nothing close
    assert sel(4096, 14336, 4096, W=4) == {}                        # other world size
    assert sel(4096, 14336, 4096, dtype="f16") == {}                # other dtype
    assert sel(4096, 14336, 4096, op="matmul_all_gather") == {}     # other op
    # explicit wins over everything
    assert tuning.select("a", "x", {"tile_n": 128}, path, tuning.shape_info("all_gather_matmul", 8, 4096,
                                                                            14336, 4096, "bf16")) == {"tile_n": 128}


def test_nearest_shape_concurrent_needs_the_same_collective(tmp_path):
    path = str(tmp_path / "t.json")
    _rec(path, "concurrent", 8192, 8192, 8192, {"gemm_ctas": 90}, 1.0, 1.1, coll="all_reduce", count=64 << 20,
         coll_dtype="f32")
    info = tuning.shape_info("concurrent", 8, 8192, 8192, 8192, "bf16", "all_reduce", 48 << 20, "f32")
    assert tuning.lookup_nearest("a", info, path) == {"gemm_ctas": 90}
    info = tuning.shape_info("concurrent", 8, 8192, 8192, 8192, "bf16", "all_gather", 64 << 20, "f32")
    assert tuning.lookup_nearest("a", info, path) is None
    assert tuning.shape_distance(tuning.shape_info("concurrent", 8, 1, 1, 1, "bf16", "all_reduce", 4, "f32"),
                                 tuning.shape_info("concurrent", 8, 2, 1, 1, "bf16", "all_reduce", 8, "f32")) == \
        pytest.approx(2 ** 0.5)


def test_concurrent_candidates_rank_tiles_and_splits():
    c = tuning.concurrent_candidates(8192, 8192, 8192, "all_reduce", 8, 64 << 20, 152, top_k=6)
    assert c[0] == {} and len(c) == 6
    # the default split with smaller and larger collective items, then the
    # predictor's (tile, split) ranking
    assert c[1] == {"comm_block": 65536} and c[2] == {"comm_block": 196608}
    assert all("gemm_ctas" in x and "tile_m" in x for x in c[3:])
    # a collective with few items keeps its item size
    small = tuning.concurrent_candidates(8192, 8192, 8192, "all_reduce", 8, 1 << 19, 152, top_k=6)
    assert all("comm_block" not in x for x in small)
    assert len({json.dumps(x, sort_keys=True) for x in c}) == len(c)
    # the fused-op candidate helper hands the concurrent mode to it
    assert tuning.candidates("concurrent", 8, 8192, 8192, 8192, 152, top_k=6, coll="all_reduce",
                             count=64 << 20) == c
