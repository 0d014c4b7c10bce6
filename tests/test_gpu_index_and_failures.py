"""Teacher-forced index loading and the failure paths, on the GPU.

* lkv_load_index with the oracle's own K-means index (the direction in which
  the oracle's index drives the GPU decode): the loaded index reads back
  unchanged, and the decode from it matches the oracle decode from the same
  index bit for bit on every decision.
* Host-side allocation failure (LKV_FAIL_ALLOC_AFTER) returns LKV_ENOMEM and
  leaks nothing; a device-side bounded wait that runs out is reported as
  LKV_ETIMEOUT by lkv_sync with the context still usable; an out-of-range
  teacher-forced assignment is reported by lkv_sync. No test here faults,
  traps or hangs the GPU: every failure is made on the host, or is a wait
  on a barrier that nothing completes, bounded to a millisecond."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from cluster_indexed_kv_gb300 import _lib
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import cluster_indexed_kv_gb300 as lkv
    lkv.build()
    oracle.build()


def _small():
    return synth.WORKLOADS["long_out"].replace(batch=2, n_prefill=2048, n_components=64,
                                               n_clusters=64, iters=6, n_steps=400,
                                               local_buf=64, budget=256)


def test_load_index_from_oracle_kmeans():
    w = _small()
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    B, Hkv, N, C = w.batch, w.n_kv_heads, w.n_prefill, w.n_clusters
    km = [[oracle.kmeans(synth.to_oracle(K[b, h]), C, w.iters, 40 + 8 * b + h) for h in range(Hkv)]
          for b in range(B)]
    assign = torch.tensor(np.stack([[k["assign"] for k in row] for row in km]), device="cuda")
    cent = torch.tensor(np.stack([[k["cent"] for k in row] for row in km]), device="cuda")
    ctx = H.make_ctx(w)
    ctx.load_index(0, K, V, C, assign, cent)
    ctx.sync()
    for b in range(B):
        for h in range(Hkv):
            ix = ctx.get_index(0, b, h, N)
            k = km[b][h]
            assert np.array_equal(ix["assign"], k["assign"])
            assert np.array_equal(ix["centroids"][:C].view(np.uint32), k["cent"].view(np.uint32))
            assert np.array_equal(ix["unit_len"][:C], k["count"])
            assert np.array_equal(ix["perm"], np.argsort(k["assign"], kind="stable"))
    g = H.run_decode(ctx, w, q, kn, vn)
    for b in range(B):
        idx = [dict(assign=km[b][h]["assign"], centroids=km[b][h]["cent"]) for h in range(Hkv)]
        o = H.oracle_decode(w, K, V, idx, q, kn, vn, b, 0)
        rep = H.compare_decode(g, o, w, b, 0)
        H.compare_segments(ctx, w, o, b, 0, 0)
        assert rep["n_boundary"] >= 3 and rep["n_evicted"] >= 1
    ctx.close()


def test_load_index_rejects_out_of_range_assignment():
    w = _small().replace(batch=1)
    K, V = synth.prefill(w, 0, "cuda")
    ctx = H.make_ctx(w)
    assign = torch.zeros(1, w.n_kv_heads, w.n_prefill, dtype=torch.int32, device="cuda")
    assign[0, 1, 17] = w.n_clusters  # one id past the last cluster
    cent = torch.zeros(1, w.n_kv_heads, w.n_clusters, 128, device="cuda")
    ctx.load_index(0, K, V, w.n_clusters, assign, cent)
    with pytest.raises(_lib.LKVError) as e:
        ctx.sync()
    assert e.value.status == _lib.LKV_ECUDA and "invariant" in str(e.value)
    ctx.sync()  # reported once; the context stays usable
    ctx.build_index(0, K, V, w.n_clusters, 2, 1)
    ctx.sync()
    ctx.close()


def _create_fails(w, fail_at, monkeypatch):
    monkeypatch.setenv("LKV_FAIL_ALLOC_AFTER", str(fail_at))
    try:
        ctx = H.make_ctx(w)
    except _lib.LKVError as e:
        assert e.status == _lib.LKV_ENOMEM and "injected" in str(e)
        return True
    finally:
        monkeypatch.delenv("LKV_FAIL_ALLOC_AFTER")
    ctx.close()
    return False


def test_injected_allocation_failure(monkeypatch):
    """Failing the first, some middle and the last of lkv_create's
    allocations (device and pinned host) returns LKV_ENOMEM and frees the
    rest; past the last one the injection has nothing to fail."""
    w = _small()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for k in (0, 5, 20):
        assert _create_fails(w, k, monkeypatch)
    n = 21
    while _create_fails(w, n, monkeypatch):
        n += 1
        assert n < 200
    assert n > 25  # the context's arrays (pool, index, plans, scratch) are many
    assert _create_fails(w, n - 1, monkeypatch)
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info()[0] - free0) < (64 << 20), "allocations leaked"
    ctx = H.make_ctx(w)  # a normal create still works
    ctx.close()


def test_device_wait_timeout_is_reported():
    w = _small().replace(batch=1)
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=4)
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, w.n_clusters, 2, 1)
    ctx.diag_wait_timeout(1_000_000)  # 1 ms
    with pytest.raises(_lib.LKVError) as e:
        ctx.sync()
    assert e.value.status == _lib.LKV_ETIMEOUT
    ctx.sync()  # cleared once reported
    out = torch.empty(1, 1, w.n_heads, 128, device="cuda")
    ctx.decode_step(0, q[0], kn[0], vn[0], w.tau, w.budget, out)
    ctx.sync()
    assert torch.isfinite(out).all()
    with pytest.raises(_lib.LKVError) as e:
        _lib.lkv_diag_wait_timeout(ctx._ctx, 2_000_000_000)
    assert e.value.status == _lib.LKV_EINVAL
    ctx.close()


def test_uva_read_copies_pinned_host_memory():
    n = (3 << 20) + 48  # not a multiple of the grid's 8-deep stride
    host = torch.randint(0, 255, (n,), dtype=torch.uint8).pin_memory()
    dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
    _lib.lkv_uva_read(host.data_ptr(), dst.data_ptr(), n, None)
    torch.cuda.synchronize()
    assert torch.equal(dst.cpu(), host)
    pageable = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(_lib.LKVError) as e:
        _lib.lkv_uva_read(pageable.data_ptr(), dst.data_ptr(), 64, None)
    assert e.value.status == _lib.LKV_EINVAL


def test_read_ceiling_reads_device_memory_and_checks_arguments():
    n = (5 << 20) + 32  # not a multiple of the grid's 8-deep stride
    src = torch.randint(0, 255, (n,), dtype=torch.uint8, device="cuda")
    _lib.lkv_read_ceiling(src.data_ptr(), n, None)
    torch.cuda.synchronize()
    host = torch.zeros(64, dtype=torch.uint8)
    for args in ((host.data_ptr(), 64), (src.data_ptr(), 24), (src.data_ptr() + 8, 64)):
        with pytest.raises(_lib.LKVError) as e:
            _lib.lkv_read_ceiling(args[0], args[1], None)
        assert e.value.status == _lib.LKV_EINVAL
