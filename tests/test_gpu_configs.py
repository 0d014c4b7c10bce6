"""GPU parity at the sizes of the evaluation configurations.

Each test runs one configuration at its full size on the GPU and checks it
against the oracle on the same seeded inputs, where the oracle can follow in
seconds: whole runs for the long-output configuration, every step for the
long-input one and sampled layers for the 36-layer host-offload
configuration (the batch-32 sweep and the benchmarked workload are in
test_gpu_fullsize.py). Decisions (flags, r_t, selections, evicted segments,
cluster assignments) must be bit-exact and
attention outputs within 2e-3 abs + 1e-2 rel; the indexes are teacher-forced
into the oracle from the GPU once K-means itself has been checked."""
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


def _index(ctx, w, layer, b):
    return [ctx.get_index(layer, b, h, w.n_prefill) for h in range(w.n_kv_heads)]


def _oracle_run(w, K, V, idx, q, kn, vn, b, li, **kw):
    C = w.n_clusters
    assign = np.stack([ix["assign"] for ix in idx])
    cent = np.stack([ix["centroids"][:C] for ix in idx])
    return oracle.decode(synth.to_oracle(K), synth.to_oracle(V), assign, cent,
                         synth.to_oracle(q[:, b, li]), synth.to_oracle(kn[:, b, li]),
                         synth.to_oracle(vn[:, b, li]), n_clusters=C, local_buf=w.local_buf,
                         **kw)


def test_long_output_full_run():
    """B = 8, N = 2048, C = 128, T = 16384 with eviction: K-means of one
    sequence against the oracle's full 20 rounds; the first 2048 steps of
    sequences 0 and 7 step by step; then the remaining steps through the
    pipelined graph, with sequence 0's flags, evicted segments and the last
    steps' attention checked against one oracle run over all 16384 steps."""
    w = synth.WORKLOADS["long_out"]
    T, T1 = w.n_steps, 2048
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    ctx = H.make_ctx(w)
    seed = 3
    ctx.build_index(0, K, V, w.n_clusters, w.iters, seed)
    ctx.sync()
    for h in range(w.n_kv_heads):
        o = oracle.kmeans(synth.to_oracle(K[0, h]), w.n_clusters, w.iters, seed + h)
        g = ctx.get_index(0, 0, h, w.n_prefill)
        assert np.array_equal(g["assign"], o["assign"])
        assert np.array_equal(g["centroids"][:w.n_clusters].view(np.uint32), o["cent"].view(np.uint32))
    idx = {b: _index(ctx, w, 0, b) for b in (0, 7)}

    # phase 1: single steps, every selection recorded
    g1 = H.run_decode(ctx, w, q[:T1], kn[:T1], vn[:T1])
    mask1 = np.zeros(T1, np.uint8)
    mask1[::8] = 1
    for b in (0, 7):
        o = _oracle_run(w, K[b], V[b], idx[b], q[:T1], kn[:T1], vn[:T1], b, 0, tau=w.tau,
                        budget=w.budget, attn_mask=mask1)
        H.compare_decode(g1, o, w, b, 0, attn_mask=mask1)
    # phase 2: the rest through the pipelined multi-step graph
    out = torch.empty(T - T1, w.batch, 1, w.n_heads, 128, device="cuda")
    bnd = torch.zeros(T - T1, w.batch, 1, dtype=torch.uint8, device="cuda")
    r = torch.zeros(T - T1, w.batch, 1, device="cuda")
    ctx.decode_steps(0, q[T1:], kn[T1:], vn[T1:], w.tau, w.budget, out, boundary=bnd, r_out=r)
    ctx.sync()
    last = 32
    mask = np.zeros(T, np.uint8)
    mask[-last:] = 1
    o = _oracle_run(w, K[0], V[0], idx[0], q, kn, vn, 0, 0, tau=w.tau, budget=w.budget,
                    attn_mask=mask, want_sel=False, want_seg_cent=True)
    flags = np.concatenate([g1["boundary"][:, 0, 0], bnd[:, 0, 0].cpu().numpy()])
    assert np.array_equal(flags, o["flag"])
    rr = np.concatenate([g1["r"][:, 0, 0], r[:, 0, 0].cpu().numpy()])
    assert np.array_equal(rr.view(np.uint32), o["r32"].view(np.uint32))
    assert o["n_evicted"] > 100
    H.compare_segments(ctx, w, o, 0, 0, 0)
    got = out[-last:, 0, 0].double().cpu().numpy()
    want = o["out"][-last:]
    assert (np.abs(got - want) <= H.ATOL + H.RTOL * np.abs(want)).all()
    ctx.close()


def test_long_input_every_step():
    """B = 1, N = 32768, C = 2048, T = 256: all steps of every KV head,
    attention at every step, teacher-forced from the GPU index (the
    full-size K-means itself is checked in the tensor-core filter tests)."""
    w = synth.WORKLOADS["long_in"]
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, 1)
    idx = _index(ctx, w, 0, 0)
    g = H.run_decode(ctx, w, q, kn, vn)
    o = _oracle_run(w, K[0], V[0], idx, q, kn, vn, 0, 0, tau=w.tau, budget=w.budget)
    rep = H.compare_decode(g, o, w, 0, 0)
    assert rep["n_boundary"] >= 5
    ctx.close()


def test_host_offload_36_layers():
    """36 layers x 8 KV heads x 131072 keys, C = 8192, K/V pool in pinned
    host memory read over UVA. Layer 0's first Lloyd round is checked on
    sampled keys and all centroids; then all layers are built with 20 rounds
    and decoded for 512 steps, and layers 0 and 35 are compared step by step
    with the oracle (attention at every fourth step)."""
    w = synth.WORKLOADS["offload"]
    C, N = w.n_clusters, w.n_prefill
    ctx = H.make_ctx(w)
    # one Lloyd round of layer 0, head 3: sampled assignments and all centroids
    K0, V0 = synth.prefill(w, 0, "cuda")
    ctx.build_index(0, K0, V0, C, 1, 11)
    keys = synth.to_oracle(K0[0, 3])
    init = oracle.bf16_bits_to_f32(keys[oracle.init_indices(N, C, 11 + 3)])
    g = ctx.get_index(0, 0, 3, N)
    rows = np.sort(np.random.default_rng(4).choice(N, 256, replace=False))
    assert np.array_equal(g["assign"][rows], oracle.assign(keys[rows], oracle.operand(init, 1)))
    cent, cnt, _ = oracle.update(keys, g["assign"], init)
    assert np.array_equal(g["unit_len"][:C], cnt)
    assert np.array_equal(g["centroids"][:C].view(np.uint32), cent.view(np.uint32))
    del keys
    # the full build, keeping the checked layers' tensors for the oracle
    keep = {}
    for layer in range(w.n_layers):
        K, V = (K0, V0) if layer == 0 else synth.prefill(w, layer, "cuda")
        ctx.build_index(layer, K, V, C, w.iters, 100 + layer)
        if layer in (0, w.n_layers - 1):
            keep[layer] = (K.cpu(), V.cpu())
        del K, V
    K0 = V0 = None
    torch.cuda.empty_cache()
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    ctx.set_profiling(True)
    ctx.profile(reset=True)
    g = H.run_decode(ctx, w, q, kn, vn)
    kern, ctr = ctx.profile(reset=True)
    ctx.set_profiling(False)
    assert kern["lkv_gather_offload"][0] == w.n_steps and ctr["gather_rows"] > 0
    mask = np.zeros(w.n_steps, np.uint8)
    mask[::4] = 1
    for layer, (K, V) in keep.items():
        idx = _index(ctx, w, layer, 0)
        o = _oracle_run(w, K[0], V[0], idx, q, kn, vn, 0, layer, tau=w.tau, budget=w.budget,
                        attn_mask=mask)
        H.compare_decode(g, o, w, 0, layer, attn_mask=mask)
    ctx.close()
