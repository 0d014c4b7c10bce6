"""GPU parity of the tensor-core K-means filter (tcgen05 distance tiles).

The filter only screens candidates: every key whose fp32 tensor-core margin
is not certified goes to the exact double-precision settlement, so the
assignment and centroids must equal the oracle's bit for bit at any size.
Small cases compare whole slices against the oracle's full K-means; the
full-size case (32768 keys x 2048 clusters per head, eight heads) checks
sampled keys against the oracle's assignment to the seeded initial centroids
and whole slices against the oracle's member means, and checks that both
filters give identical indexes after 20 rounds."""
import numpy as np
import pytest
import torch

import oracle
import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import cluster_indexed_kv_gb300 as lkv
    lkv.build()


def _launches(ctx):
    stats, _ = ctx.profile()
    return stats.get("kmeans_assign_tc", (0, 0.0))[0], stats.get("kmeans_assign", (0, 0.0))[0]


def _build(w, K, V, iters, seed, tensor_cores=True):
    ctx = H.make_ctx(w)
    ctx.set_kmeans_filter(tensor_cores)
    ctx.build_index(0, K, V, w.n_clusters, iters, seed)
    ctx.sync()
    return ctx


@pytest.mark.parametrize("n,c", [(3001, 50), (4096, 300), (257, 1), (130, 7), (1000, 513),
                                 (256, 256)])
def test_tc_filter_matches_oracle(n, c):
    """Several 128-key tiles with a ragged tail, centroid chunks of 256 with a
    ragged last chunk, one and two slices per tile boundary."""
    w = synth.WORKLOADS["long_in"].replace(n_kv_heads=2, batch=2, n_prefill=n,
                                           n_components=max(c, 4), n_clusters=c, iters=4)
    K, V = synth.prefill(w, 0, "cuda")
    seed = 29
    ctx = _build(w, K, V, w.iters, seed)
    n_tc, n_simt = _launches(ctx)
    assert n_tc == w.iters and n_simt == 0
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            s = b * w.n_kv_heads + h
            o = oracle.kmeans(synth.to_oracle(K[b, h]), c, w.iters, seed + s)
            g = ctx.get_index(0, b, h, n)
            assert np.array_equal(g["assign"], o["assign"]), \
                f"slice {s}: {np.sum(g['assign'] != o['assign'])} assignments differ"
            assert np.array_equal(g["centroids"].view(np.uint32), o["cent"].view(np.uint32))
            assert np.array_equal(g["unit_len"], o["count"])
    ctx.close()


def test_tc_filter_duplicate_and_equidistant_keys():
    """Exact ties (duplicated keys, duplicated initial centroids) go to the
    lowest cluster id through the exact settlement."""
    w = synth.WORKLOADS["long_in"].replace(n_kv_heads=1, batch=1, n_prefill=512, n_clusters=40,
                                           iters=3)
    K, V = synth.prefill(w, 0, "cuda")
    K[0, 0, 256:] = K[0, 0, :256]
    ctx = _build(w, K, V, 3, 11)
    assert _launches(ctx)[0] == 3
    g = ctx.get_index(0, 0, 0, 512)
    o = oracle.kmeans(synth.to_oracle(K[0, 0]), 40, 3, 11)
    assert np.array_equal(g["assign"], o["assign"])
    assert np.array_equal(g["centroids"].view(np.uint32), o["cent"].view(np.uint32))
    ctx.close()


def test_tc_filter_full_size_sampled():
    """32768 keys x 2048 clusters x 8 heads, one Lloyd round: the assignment of
    sampled keys equals the oracle's argmin against the seeded initial
    centroids, and every centroid of two whole heads equals the oracle's
    member mean of the GPU assignment."""
    w = synth.WORKLOADS["long_in"]
    K, V = synth.prefill(w, 0, "cuda")
    seed = 5
    ctx = _build(w, K, V, 1, seed)
    assert _launches(ctx)[0] == 1
    rng = np.random.default_rng(1)
    for h in (0, 5):
        keys = synth.to_oracle(K[0, h])
        init = keys[oracle.init_indices(w.n_prefill, w.n_clusters, seed + h)]
        cent0 = oracle.bf16_bits_to_f32(init) if init.dtype == np.uint16 else init
        g = ctx.get_index(0, 0, h, w.n_prefill)
        rows = np.sort(rng.choice(w.n_prefill, 384, replace=False))
        a = oracle.assign(keys[rows], oracle.operand(cent0, 1))
        assert np.array_equal(g["assign"][rows], a)
        cent, cnt, _ = oracle.update(keys, g["assign"], cent0)
        assert np.array_equal(g["unit_len"], cnt)
        assert np.array_equal(g["centroids"][:w.n_clusters].view(np.uint32), cent.view(np.uint32))
    ctx.close()


def test_tc_and_simt_filters_identical_full_size():
    """Both filters certify their choices against the same exact distance, so
    20 rounds at full size give identical indexes."""
    w = synth.WORKLOADS["long_in"]
    K, V = synth.prefill(w, 0, "cuda")
    out = []
    for tc in (True, False):
        ctx = _build(w, K, V, w.iters, 7, tensor_cores=tc)
        n_tc, n_simt = _launches(ctx)
        assert (n_tc, n_simt) == ((w.iters, 0) if tc else (0, w.iters))
        out.append([ctx.get_index(0, 0, h, w.n_prefill) for h in range(w.n_kv_heads)])
        ctx.close()
    for a, b in zip(*out):
        assert np.array_equal(a["assign"], b["assign"])
        assert np.array_equal(a["centroids"].view(np.uint32), b["centroids"].view(np.uint32))
        assert np.array_equal(a["perm"], b["perm"])


def test_fp32_keys_ignore_tensor_filter():
    w = synth.WORKLOADS["tiny"]
    K, V = synth.prefill(w, 0, "cuda")
    ctx = _build(w, K, V, 2, 3, tensor_cores=True)
    assert _launches(ctx) == (0, 2)
    ctx.close()
