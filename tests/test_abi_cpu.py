"""C-ABI checks that need no GPU: the library builds and loads, exports every
entry point include/lkv.h declares, rejects bad configurations with status
codes before touching the device, and the binding fails loudly without it."""
import ctypes as C
import os
import re

import pytest

import cluster_indexed_kv_gb300 as lkv
from cluster_indexed_kv_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def libpath():
    return lkv.build()


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(lkv_[a-z0-9_]+)\s*\(", src))
    return names


def test_every_declared_entry_point_is_exported(libpath):
    lib = C.CDLL(libpath)
    declared = _declared()
    assert {"lkv_create", "lkv_build_index", "lkv_decode_step"} <= declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(_lib.EXPORTED) <= declared


@pytest.mark.parametrize("field,value", [
    ("head_dim", 64), ("group", 3), ("n_kv_heads", 0), ("n_kv_heads", 17), ("batch", 0),
    ("dtype", 7), ("local_buf", 0), ("max_clusters", 0), ("max_prefill", 1 << 19),
    ("max_steps", 0), ("max_budget", -1),
])
def test_create_rejects_bad_config_without_device(libpath, field, value):
    _lib.load(libpath)
    good = dict(batch=1, n_layers=1, n_kv_heads=8, group=4, head_dim=128, dtype=1, local_buf=16,
                max_clusters=64, max_prefill=4096, max_steps=16, max_budget=128, offload=0,
                stream=None)
    good[field] = value
    cfg = _lib.lkv_config(**good)
    with pytest.raises(_lib.LKVError) as e:
        _lib.lkv_create(cfg)
    assert e.value.status == _lib.LKV_EINVAL
    assert _lib.lkv_last_error(None)


def test_null_arguments_are_rejected(libpath):
    L = _lib.load(libpath)
    assert L.lkv_create(None, None) == _lib.LKV_EINVAL
    assert L.lkv_sync(None) == _lib.LKV_EINVAL
    assert L.lkv_build_index(None, 0, None, None, 1, 1, 1, 0) == _lib.LKV_EINVAL
    assert L.lkv_decode_step(None, 0, 1, None, None, None, 0.7, 1, 1, None, None, None, None,
                             None) == _lib.LKV_EINVAL
    assert L.lkv_set_kmeans_filter(None, _lib.LKV_FILTER_SIMT) == _lib.LKV_EINVAL


def test_injected_allocation_failure_without_device(libpath, monkeypatch):
    """LKV_FAIL_ALLOC_AFTER=0 fails the first allocation of lkv_create, before
    any CUDA call, so the status path is checked here without a GPU."""
    _lib.load(libpath)
    monkeypatch.setenv("LKV_FAIL_ALLOC_AFTER", "0")
    cfg = _lib.lkv_config(batch=1, n_layers=1, n_kv_heads=8, group=4, head_dim=128, dtype=1,
                          local_buf=16, max_clusters=64, max_prefill=4096, max_steps=16,
                          max_budget=128, offload=0, stream=None)
    with pytest.raises(_lib.LKVError) as e:
        _lib.lkv_create(cfg)
    assert e.value.status == _lib.LKV_ENOMEM and "injected" in str(e.value)


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        _lib._lib = None
        try:
            _lib.load(str(tmp_path / "missing.so"))
        finally:
            _lib._lib = None


def test_paris_prior_tables_match_the_oracle(libpath):
    """lkv_paris_levels is host-only: the library's closed-form tables equal
    the oracle's Simpson/bisection tables bit for bit (both are the float
    roundings of the same prior quantiles and bin means)."""
    import numpy as np
    import oracle
    thr, lev = _lib.lkv_paris_levels()
    othr, olev = oracle.paris_levels(8)
    assert np.array_equal(np.array(thr, np.float32).view(np.uint32), othr.view(np.uint32))
    assert np.array_equal(np.array(lev, np.float32).view(np.uint32), olev.view(np.uint32))
