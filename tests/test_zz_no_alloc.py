"""lkv_kmeans_static: the K-means entry point that allocates nothing.

Some callers cannot allocate GPU memory: their process's device memory is
owned by another allocator (a serving engine or framework that reserves the
whole GPU at start-up), or they must avoid the implicit device
synchronisation of cudaMalloc/cudaFree. For them lkv_kmeans_static runs the
index build's K-means for one (sequence, KV head) slice with all scratch in a
fixed array inside the library. This file checks, through the C ABI, that two
calls in a row give exactly what lkv_build_index gives and what the oracle's
K-means gives (bit-exact centroids and assignments, the tolerance the other
K-means tests use), which also shows that the shared array's leftovers from
one call do not leak into the next; that slice h of a multi-head build is
reproduced with the build's seed + h; and that lkv_kmeans_static_status
reports a clean run. It is collected last on purpose."""
import numpy as np
import pytest
import torch

import oracle
import synth
from cluster_indexed_kv_gb300 import _lib
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _reference(w, K, V, seed, head=0):
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, seed)
    ix = ctx.get_index(0, 0, head, w.n_prefill)
    ctx.close()
    return ix["centroids"][: w.n_clusters], ix["assign"]


def _static(w, K, seed, head=0):
    import cluster_indexed_kv_gb300 as lkv
    lkv.build()
    keys = K[0, head].contiguous()
    cent = torch.full((w.n_clusters, 128), float("nan"), dtype=torch.float32, device="cuda")
    assign = torch.full((w.n_prefill,), -1, dtype=torch.int32, device="cuda")
    dt = _lib.LKV_DTYPE_BF16 if w.dtype == "bf16" else _lib.LKV_DTYPE_FP32
    stream = torch.cuda.current_stream().cuda_stream
    _lib.lkv_kmeans_static(keys.data_ptr(), dt, w.n_prefill, w.n_clusters, w.iters, seed,
                           cent.data_ptr(), assign.data_ptr(), stream)
    _lib.lkv_kmeans_static_status(stream)  # waits for the stream; raises on a device anomaly
    return cent.cpu().numpy(), assign.cpu().numpy()


def _oracle(w, K, seed, head=0):
    o = oracle.kmeans(synth.to_oracle(K[0, head]), w.n_clusters, w.iters, seed)
    return o["cent"], o["assign"]


def test_two_calls_in_a_row_match_build_index_and_oracle():
    cases = [
        (synth.WORKLOADS["long_in"].replace(batch=1, n_kv_heads=1, n_prefill=4099,
                                            n_components=120, n_clusters=100, iters=6), 21),
        (synth.WORKLOADS["long_in"].replace(batch=1, n_kv_heads=1, n_prefill=2000,
                                            n_components=40, n_clusters=37, iters=4, seed=9), 5),
    ]
    for w, seed in cases:
        K, V = synth.prefill(w, 0, "cuda")
        c_ref, a_ref = _reference(w, K, V, seed)
        c_or, a_or = _oracle(w, K, seed)
        c_got, a_got = _static(w, K, seed)
        for c, a in ((c_ref, a_ref), (c_or, a_or)):
            assert np.array_equal(a_got, a)
            assert np.array_equal(c_got.view(np.uint32), c.view(np.uint32))


def test_head_h_of_a_build_needs_seed_plus_h():
    w = synth.WORKLOADS["long_in"].replace(batch=1, n_kv_heads=3, n_prefill=1500,
                                           n_components=48, n_clusters=40, iters=3, seed=13)
    K, V = synth.prefill(w, 0, "cuda")
    seed, h = 100, 2
    c_ref, a_ref = _reference(w, K, V, seed, head=h)
    c_got, a_got = _static(w, K, seed + h, head=h)
    assert np.array_equal(a_got, a_ref)
    assert np.array_equal(c_got.view(np.uint32), c_ref.view(np.uint32))


def test_fp32_keys_and_limits():
    w = synth.WORKLOADS["tiny"].replace(n_prefill=1500, n_components=24, n_clusters=24, iters=5)
    K, V = synth.prefill(w, 0, "cuda")
    c_ref, a_ref = _reference(w, K, V, 3)
    c_or, a_or = _oracle(w, K, 3)
    c_got, a_got = _static(w, K, 3)
    for c, a in ((c_ref, a_ref), (c_or, a_or)):
        assert np.array_equal(a_got, a)
        assert np.array_equal(c_got.view(np.uint32), c.view(np.uint32))
    keys = torch.zeros(40000, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(16, 128, device="cuda")
    asg = torch.zeros(40000, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.LKVError) as e:
        _lib.lkv_kmeans_static(keys.data_ptr(), _lib.LKV_DTYPE_BF16, 40000, 16, 2, 1,
                               out.data_ptr(), asg.data_ptr(), None)
    assert e.value.status == _lib.LKV_EINVAL and "32768" in str(e.value)
    _lib.lkv_kmeans_static_status(None)
