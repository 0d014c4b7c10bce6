"""Full-size GPU parity of two selection variants on the benchmarked shape
(the 32K-input, batch-8 workload, through the pipelined decode graph):

* per-query-head selection ("LouisKV ... Long Input-Output Sequences",
  消融实验: the baseline of group-consistent selection), 1200 steps so that
  the local buffer fills and segments are evicted;
* the ParisKV-style token selector (ParisKV technical summary, 核心算法创新
  1-2), 700 steps.

Sequence 0 is compared with the oracle run with the same variant: flags, r_t
and selection sizes at every step, every selected set, and the attention
outputs at sampled steps. Decisions bit-exact, attention within 2e-3 abs +
1e-2 rel; oracle work in a spawn process pool."""
import numpy as np
import pytest

import oracle
import synth
from tests import _harness as H
from tests import _oracle_jobs as J

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import cluster_indexed_kv_gb300 as lkv
    lkv.build()
    oracle.build()


def _steps(T, L):
    s = set(range(0, T, 48)) | set(range(max(0, L - 4), min(T, L + 8))) | set(range(T - 8, T))
    return np.array(sorted(s), dtype=np.int64)


def test_b8_32k_per_head_selection(tmp_path):
    T = 1200
    w = synth.WORKLOADS["b8_32k"].replace(n_steps=T)
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, 1)
    ctx.set_policy(per_head=True)
    idx = [ctx.get_index(0, 0, h, w.n_prefill) for h in range(w.n_kv_heads)]
    g = H.run_graph(ctx, w, q, kn, vn, seqs=(0,), chunk=128, per_head=True)
    steps = _steps(T, w.local_buf)
    kw = dict(n_clusters=w.n_clusters, local_buf=w.local_buf, tau=w.tau, budget=w.budget,
              per_head=True, max_sel=512)
    with H.spawn_pool(1) as pool:
        o = pool.submit(J.decode_run, H.oracle_inputs(tmp_path, "ph", w, K, V, idx, q, kn, vn, 0),
                        kw, steps).result()
    rep = H.compare_graph_run(g, o, w, 0, label="per-head")
    assert rep["n_boundary"] > 10 and rep["n_evicted"] > 5
    assert o["n_sel"].shape[1] == w.n_heads
    ctx.close()


def test_b8_32k_paris_selector(tmp_path):
    T = 700
    w = synth.WORKLOADS["b8_32k"].replace(n_steps=T)
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    ctx = H.make_ctx(w)          # max_prefill = N: a decode token's pool row is N + t
    prm = dict(rho=4, n_cand=2560, seed=1)
    ctx.build_paris(0, K, V, **prm)
    g = H.run_graph(ctx, w, q, kn, vn, seqs=(0,), chunk=128)
    idx = [dict(assign=np.zeros(w.n_prefill, np.int32),
                centroids=np.zeros((w.n_clusters, 128), np.float32)) for _ in range(w.n_kv_heads)]
    steps = _steps(T, w.local_buf)
    kw = dict(n_clusters=0, local_buf=w.local_buf, tau=w.tau, budget=w.budget, paris=prm)
    with H.spawn_pool(1) as pool:
        o = pool.submit(J.decode_run, H.oracle_inputs(tmp_path, "px", w, K, V, idx, q, kn, vn, 0),
                        kw, steps).result()
    rep = H.compare_graph_run(g, o, w, 0, label="paris")
    assert rep["n_boundary"] > 10
    ctx.close()
