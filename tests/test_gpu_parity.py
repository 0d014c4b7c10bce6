"""GPU parity: liblkv (through its C ABI) against the CPU oracle on the same
seeded inputs. Decisions (cluster assignments, boundary flags, segment
boundaries, selected unit sets) must be bit-exact; centroids bit-exact;
attention outputs within 2e-3 abs + 1e-2 rel."""
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


def _kmeans_check(w, layer=0, iters=None, seed=17):
    iters = iters or w.iters
    dev = "cuda"
    K, V = synth.prefill(w, layer, dev)
    ctx = H.make_ctx(w)
    ctx.build_index(layer, K, V, w.n_clusters, iters, seed)
    ctx.sync()
    S = w.batch * w.n_kv_heads
    refined = 0
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            s = b * w.n_kv_heads + h
            keys = synth.to_oracle(K[b, h])
            o = oracle.kmeans(keys, w.n_clusters, iters, seed + s)
            g = ctx.get_index(layer, b, h, w.n_prefill)
            assert g["n_units"] == w.n_clusters
            assert np.array_equal(g["assign"], o["assign"]), \
                f"slice {s}: {np.sum(g['assign'] != o['assign'])} assignments differ"
            assert np.array_equal(g["centroids"].view(np.uint32), o["cent"].view(np.uint32))
            assert np.array_equal(g["unit_len"], o["count"])
            # pool rows grouped by cluster, token order inside a cluster
            assert np.array_equal(g["perm"], np.argsort(o["assign"], kind="stable"))
            starts = np.concatenate([[0], np.cumsum(o["count"])[:-1]])
            assert np.array_equal(g["unit_row"], starts)
    st = ctx.decode_state(layer, 0)
    ctx.close()
    return st


def test_kmeans_tiny_fp32():
    st = _kmeans_check(synth.WORKLOADS["tiny"])
    assert st["n_units"] == 32


@pytest.mark.parametrize("n,c", [(3001, 50), (64, 64), (200, 1), (130, 7)])
def test_kmeans_bf16_ragged(n, c):
    w = synth.WORKLOADS["long_in"].replace(n_kv_heads=2, batch=2, n_prefill=n, n_components=max(c, 4),
                                           n_clusters=c, iters=6)
    _kmeans_check(w)


def test_kmeans_duplicate_keys_tie_to_lowest():
    w = synth.WORKLOADS["long_in"].replace(n_kv_heads=1, batch=1, n_prefill=256, n_clusters=16,
                                           iters=4)
    K, V = synth.prefill(w, 0, "cuda")
    K[0, 0, 128:] = K[0, 0, :128]          # every key appears twice
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, 16, 4, 5)
    g = ctx.get_index(0, 0, 0, 256)
    o = oracle.kmeans(synth.to_oracle(K[0, 0]), 16, 4, 5)
    assert np.array_equal(g["assign"], o["assign"])
    assert np.array_equal(g["centroids"].view(np.uint32), o["cent"].view(np.uint32))
    ctx.close()


def test_kmeans_update_sums_in_token_order_past_2_13():
    """A cluster of 512 members whose dimension-0 partial sums pass 2^13 and
    whose small members fall below the double-precision ulp there: the
    token-order double sum rounds, the exact fixed-point sum does not, and
    the two means differ in their last float bit. The update must give the
    token-order result (here 16.0), bit for bit with the oracle."""
    keys, seed = H.rounding_update_keys()
    w = synth.WORKLOADS["long_in"].replace(n_kv_heads=1, batch=1, n_prefill=1024, n_clusters=2,
                                           iters=3)
    K = torch.from_numpy(keys).to(torch.bfloat16).reshape(1, 1, 1024, 128).cuda()
    V = torch.zeros_like(K)
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, 2, 3, seed)
    g = ctx.get_index(0, 0, 0, 1024)
    o = oracle.kmeans(synth.to_oracle(K[0, 0]), 2, 3, seed)
    st = ctx.decode_state(0, 0)
    ctx.close()
    assert np.array_equal(g["assign"], o["assign"])
    assert np.array_equal(g["centroids"].view(np.uint32), o["cent"].view(np.uint32))
    a = int(o["assign"][0])
    assert o["cent"][a, 0] == np.float32(16.0)
    assert st["n_inexact"] >= 1  # the cluster left the fixed-point path


def _decode_check(w, *, tau=None, budget=None, T=None, seqs=None, teacher=True, build_seed=3,
                  key_scale=1.0):
    T = T or w.n_steps
    dev = "cuda"
    K, V = synth.prefill(w, 0, dev)
    q, kn, vn, _ = synth.decode_inputs(w, dev, n_steps=T)
    if key_scale != 1.0:
        kn = (kn.float() * key_scale).to(kn.dtype)
    ctx = H.make_ctx(w, max_steps=T, max_budget=max(budget or w.budget, 1))
    ctx.build_index(0, K, V, w.n_clusters, w.iters, build_seed)
    ctx.sync()
    idx = {(b, h): ctx.get_index(0, b, h, w.n_prefill) for b in range(w.batch)
           for h in range(w.n_kv_heads)}
    if not teacher:
        for (b, h), ix in idx.items():
            o = oracle.kmeans(synth.to_oracle(K[b, h]), w.n_clusters, w.iters,
                              build_seed + b * w.n_kv_heads + h)
            ix["assign"], ix["centroids"] = o["assign"], o["cent"]
    g = H.run_decode(ctx, w, q, kn, vn, tau=tau, budget=budget)
    reports = []
    for b in (seqs if seqs is not None else range(w.batch)):
        o = H.oracle_decode(w, K, V, [idx[(b, h)] for h in range(w.n_kv_heads)], q, kn, vn, b, 0,
                            tau=tau, budget=budget)
        reports.append(H.compare_decode(g, o, w, b, 0))
        H.compare_segments(ctx, w, o, b, 0, 0)
    ctx.close()
    return reports


def test_decode_tiny_fp32_full():
    rep = _decode_check(synth.WORKLOADS["tiny"], teacher=False)
    assert rep[0]["n_boundary"] >= 1


def test_kmeans_update_tiny_and_zero_members():
    """Members below the fast path's range: |v| < 2^-28 sends a cluster of at
    most 256 members to the 2^-40 sums, |v| < 2^-33 to the double-precision
    token-order sums, and signed zeros add nothing. Centroids stay bit-exact
    with the oracle on every path."""
    w = synth.WORKLOADS["long_in"].replace(n_kv_heads=1, batch=1, n_prefill=1024, n_components=16,
                                           n_clusters=16, iters=3)
    K, V = synth.prefill(w, 0, "cuda")
    Kf = K.float()
    idx = torch.arange(1024, device="cuda")
    Kf[0, 0, idx % 7 == 0, 0] = 2.0 ** -30
    Kf[0, 0, idx % 11 == 0, 1] = -(2.0 ** -36)
    Kf[0, 0, idx % 5 == 0, 2] = 0.0
    Kf[0, 0, idx % 13 == 0, 3] = -0.0
    K = Kf.to(torch.bfloat16)
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, 16, 3, 9)
    g = ctx.get_index(0, 0, 0, 1024)
    st = ctx.decode_state(0, 0)
    ctx.close()
    o = oracle.kmeans(synth.to_oracle(K[0, 0]), 16, 3, 9)
    assert int(g["unit_len"].max()) <= 256  # every cluster takes the fast path first
    assert np.array_equal(g["assign"], o["assign"])
    assert np.array_equal(g["centroids"].view(np.uint32), o["cent"].view(np.uint32))
    assert st["n_inexact"] > 0  # the 2^-36 members took the double-precision path


def test_decode_segment_means_with_large_keys():
    """Decode keys scaled so that some reach 16..32: with L = 512 a segment
    that holds one leaves the fixed-point sum for the token-order double sum
    (the exponent bound that keeps every partial sum exact). The segment
    means stay bit-exact with the oracle either way."""
    w = synth.WORKLOADS["long_out"].replace(batch=2, n_kv_heads=2, n_prefill=700, n_components=30,
                                            n_clusters=30, iters=5, local_buf=512, budget=200,
                                            jump_p=0.08)
    rep = _decode_check(w, tau=0.9, T=640, key_scale=12.0)
    assert all(r["n_evicted"] >= 1 for r in rep)


def test_decode_bf16_evictions_and_forced_cuts():
    w = synth.WORKLOADS["long_out"].replace(batch=2, n_kv_heads=2, n_prefill=700, n_components=30,
                                            n_clusters=30, iters=5, local_buf=16, budget=200,
                                            jump_p=0.08)
    rep = _decode_check(w, tau=0.9, T=300)
    assert all(r["n_evicted"] > 5 for r in rep)


@pytest.mark.parametrize("group", [1, 2, 8])
def test_decode_query_group_sizes(group):
    """GQA groups other than 4 query heads per KV head: 8 takes the
    tensor-core attention with two products per row block, 1 and 2 the scalar
    one; decisions bit-exact, outputs within tolerance, ragged last chunks."""
    w = synth.WORKLOADS["long_out"].replace(batch=2, n_kv_heads=2, group=group, n_prefill=700,
                                            n_components=30, n_clusters=30, iters=4, local_buf=40,
                                            budget=150, jump_p=0.08)
    rep = _decode_check(w, tau=0.9, T=120)
    assert sum(r["n_boundary"] for r in rep) >= 2


def test_decode_never_triggering_forces_cuts():
    w = synth.WORKLOADS["long_in"].replace(batch=1, n_kv_heads=2, n_prefill=500, n_components=20,
                                           n_clusters=20, iters=3, local_buf=8, budget=64)
    rep = _decode_check(w, tau=-2.0, T=60)
    assert rep[0]["n_forced"] == rep[0]["n_evicted"] > 0


@pytest.mark.parametrize("budget", [0, 1, 10 ** 6])
def test_decode_budget_edges(budget):
    w = synth.WORKLOADS["long_in"].replace(batch=2, n_kv_heads=2, n_prefill=400, n_components=16,
                                           n_clusters=16, iters=3, local_buf=4, budget=budget)
    _decode_check(w, tau=0.95, T=40, budget=budget)


def test_decode_local_buf_one():
    w = synth.WORKLOADS["tiny"].replace(n_prefill=300, n_components=8, n_clusters=8, iters=3,
                                        local_buf=1, budget=40)
    _decode_check(w, tau=0.98, T=50)


def test_decode_fullcache_equals_full_attention():
    """tau > 1 (retrieve every step) and a budget covering every token:
    liblkv's output is full softmax attention over all tokens so far."""
    w = synth.WORKLOADS["long_in"].replace(batch=2, n_kv_heads=2, n_prefill=333, n_components=9,
                                           n_clusters=9, iters=3, local_buf=5)
    T = 30
    budget = w.n_prefill + T
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    ctx = H.make_ctx(w, max_steps=T, max_budget=budget)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, 1)
    g = H.run_decode(ctx, w, q, kn, vn, tau=1.5, budget=budget, keep_sel=False)
    Kf, Vf = K.double().cpu(), V.double().cpu()
    qf, knf, vnf = q.double().cpu(), kn.double().cpu(), vn.double().cpu()
    for t in range(T):
        for b in range(w.batch):
            for h in range(w.n_kv_heads):
                kk = torch.cat([Kf[b, h], knf[: t + 1, b, 0, h]])
                vv = torch.cat([Vf[b, h], vnf[: t + 1, b, 0, h]])
                qq = qf[t, b, 0, h * w.group:(h + 1) * w.group]
                want = torch.softmax(qq @ kk.T / np.sqrt(128), -1) @ vv
                got = torch.from_numpy(g["out"][t, b, 0, h * w.group:(h + 1) * w.group]).double()
                assert torch.allclose(got, want, atol=H.ATOL, rtol=H.RTOL)
    ctx.close()


def test_decode_two_layers_one_call():
    w = synth.WORKLOADS["long_in"].replace(batch=2, n_layers=2, n_kv_heads=2, n_prefill=300,
                                           n_components=12, n_clusters=12, iters=3, local_buf=8,
                                           budget=80)
    T = 40
    ctx = H.make_ctx(w, max_steps=T)
    Ks = [synth.prefill(w, l, "cuda") for l in range(2)]
    for l in range(2):
        ctx.build_index(l, Ks[l][0], Ks[l][1], w.n_clusters, w.iters, 7 + l)
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    g = H.run_decode(ctx, w, q, kn, vn, tau=0.95)
    for l in range(2):
        idx = [ctx.get_index(l, 1, h, w.n_prefill) for h in range(w.n_kv_heads)]
        o = H.oracle_decode(w, Ks[l][0], Ks[l][1], idx, q, kn, vn, 1, l, tau=0.95)
        H.compare_decode(g, o, w, 1, l)
        H.compare_segments(ctx, w, o, 1, l, l)
    ctx.close()


def test_errors_are_status_codes():
    import cluster_indexed_kv_gb300 as lkv
    w = synth.WORKLOADS["tiny"].replace(n_prefill=256, n_clusters=8)
    ctx = H.make_ctx(w, max_steps=2)
    q = torch.zeros(1, 1, 4, 128, device="cuda")
    kv = torch.zeros(1, 1, 1, 128, device="cuda")
    out = torch.zeros(1, 1, 4, 128, device="cuda")
    with pytest.raises(lkv.LKVError) as e:      # decode before an index
        ctx.decode_step(0, q, kv, kv, 0.7, 10, out)
    assert e.value.status == 5
    K, V = synth.prefill(w, 0, "cuda")
    with pytest.raises(lkv.LKVError) as e:      # more clusters than tokens allowed
        ctx.build_index(0, K, V, 9, 2, 1)
    assert e.value.status == 1
    ctx.build_index(0, K, V, 8, 2, 1)
    with pytest.raises(lkv.LKVError) as e:      # budget above max_budget
        ctx.decode_step(0, q, kv, kv, 0.7, 10 ** 6, out)
    assert e.value.status == 1
    ctx.decode_step(0, q, kv, kv, 0.7, 10, out)
    ctx.decode_step(0, q, kv, kv, 0.7, 10, out)
    with pytest.raises(lkv.LKVError) as e:      # max_steps reached
        ctx.decode_step(0, q, kv, kv, 0.7, 10, out)
    assert e.value.status == 4
    ctx.sync()
    ctx.close()


def test_decode_steps_graph_matches_single_steps():
    """lkv_decode_steps (64-step CUDA graphs + tail, chunked over one set of
    full-length buffers) takes bit-identical decisions (flags, selection
    sizes and sets) to single steps; the attention outputs agree within fp32
    rounding (the two paths split a slice's rows over different warp groups,
    which changes the order of the partial softmax sums)."""
    w = synth.WORKLOADS["long_out"].replace(batch=2, n_kv_heads=2, n_prefill=600, n_components=20,
                                            n_clusters=20, iters=3, local_buf=16, budget=120,
                                            jump_p=0.1)
    T = 300
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    outs = []
    for mode in ("single", "chunks"):
        ctx = H.make_ctx(w, max_steps=T)
        ctx.build_index(0, K, V, w.n_clusters, w.iters, 9)
        out = torch.zeros(T, w.batch, 1, w.n_heads, 128, device="cuda")
        bnd = torch.zeros(T, w.batch, 1, dtype=torch.uint8, device="cuda")
        nsel = torch.zeros(T, w.batch, 1, w.n_kv_heads, dtype=torch.int32, device="cuda")
        sel = torch.full((T, w.batch, 1, w.n_kv_heads, ctx.u_cap), -1, dtype=torch.int32,
                         device="cuda")
        if mode == "single":
            for t in range(T):
                ctx.decode_step(0, q[t], kn[t], vn[t], 0.9, w.budget, out[t], boundary=bnd[t],
                                n_selected=nsel[t], selected_units=sel[t])
        else:
            for c0, c1 in ((0, 140), (140, 280), (280, 300)):
                ctx.decode_steps(0, q[c0:c1], kn[c0:c1], vn[c0:c1], 0.9, w.budget, out[c0:c1],
                                 boundary=bnd[c0:c1], n_selected=nsel[c0:c1],
                                 selected_units=sel[c0:c1])
        ctx.sync()
        outs.append((out.cpu(), bnd.cpu(), nsel.cpu(), sel.cpu()))
        ctx.close()
    for a, b in zip(outs[0][1:], outs[1][1:]):
        assert torch.equal(a, b)
    o1, o2 = outs[0][0], outs[1][0]
    assert torch.allclose(o1, o2, rtol=1e-5, atol=1e-6), (o1 - o2).abs().max()
    assert outs[0][1].sum() > 3


def test_graph_with_every_step_retrieving():
    """tau > 1: every step retrieves, so the pipelined graph advances the
    selection-plan slot at every step and the ring of in-flight attentions
    is always full of distinct plans; the result must still equal the
    oracle step for step."""
    w = synth.WORKLOADS["long_out"].replace(batch=2, n_kv_heads=2, n_prefill=900, n_components=30,
                                            n_clusters=30, iters=3, local_buf=24, budget=160,
                                            jump_p=0.05)
    T = 300
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    ctx = H.make_ctx(w, max_steps=T)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, 4)
    idx = {b: [ctx.get_index(0, b, h, w.n_prefill) for h in range(w.n_kv_heads)] for b in range(w.batch)}
    out = torch.zeros(T, w.batch, 1, w.n_heads, 128, device="cuda")
    bnd = torch.zeros(T, w.batch, 1, dtype=torch.uint8, device="cuda")
    nsel = torch.zeros(T, w.batch, 1, w.n_kv_heads, dtype=torch.int32, device="cuda")
    sel = torch.full((T, w.batch, 1, w.n_kv_heads, ctx.u_cap), -1, dtype=torch.int32, device="cuda")
    ctx.decode_steps(0, q, kn, vn, 2.0, w.budget, out, boundary=bnd, n_selected=nsel,
                     selected_units=sel)
    ctx.sync()
    g = dict(out=out.cpu().numpy(), boundary=bnd.cpu().numpy(), r=np.zeros((T, w.batch, 1), np.float32),
             n_sel=nsel.cpu().numpy(), sel={})
    sel_h = sel.cpu().numpy()
    assert g["boundary"].all()
    for b in range(w.batch):
        o = H.oracle_decode(w, K, V, idx[b], q, kn, vn, b, 0, tau=2.0)
        assert np.array_equal(g["boundary"][:, b, 0], o["flag"])
        assert np.array_equal(g["n_sel"][:, b, 0], o["n_sel"])
        for t in range(T):
            for h in range(w.n_kv_heads):
                k = o["n_sel"][t, h]
                assert np.array_equal(np.sort(sel_h[t, b, 0, h, :k]), np.sort(o["sel"][t, h, :k]))
        err = np.abs(g["out"][:, b, 0].astype(np.float64) - o["out"])
        assert (err <= H.ATOL + H.RTOL * np.abs(o["out"])).all(), err.max()
    ctx.close()


def test_profile_counters_and_launch_counts():
    w = synth.WORKLOADS["long_in"].replace(batch=2, n_kv_heads=2, n_prefill=500, n_components=20,
                                           n_clusters=20, iters=2, local_buf=8, budget=100)
    T = 70
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    ctx = H.make_ctx(w, max_steps=T)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, 1)
    ctx.set_profiling(True)
    ctx.profile(reset=True)
    out = torch.zeros(T, w.batch, 1, w.n_heads, 128, device="cuda")
    ctx.decode_steps(0, q, kn, vn, 0.9, w.budget, out)
    kern, ctr = ctx.profile(reset=True)
    assert kern["lkv_attn"][0] == T and kern["lkv_attn"][1] > 0
    assert ctr["attn_slices"] == T * w.batch * w.n_kv_heads
    # every attended row is a selected token (<= budget) or a buffer token (<= L)
    assert ctr["attn_rows"] <= ctr["attn_slices"] * (w.budget + w.local_buf)
    ctx.close()
