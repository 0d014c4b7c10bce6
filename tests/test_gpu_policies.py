"""GPU parity of the retrieval-policy variants (lkv_set_policy) and of the
page-unit index (lkv_build_pages) against the oracle run with the same
policy: the baselines the pages compare the method with ("LouisKV ... Long
Input-Output Sequences", 研究背景与动机 and 消融实验: retrieval at every token or
at a fixed step, page-granular units) and the skip-and-continue budget fill.
Decisions (flags, r_t, selections, segments) bit-exact, attention within the
tolerance of the other parity tests, through the pipelined graph path."""
import numpy as np
import pytest
import torch

import oracle
import synth
from cluster_indexed_kv_gb300 import _lib
from tests import _harness as H

pytestmark = pytest.mark.gpu

_TRIG = {"adaptive": oracle.TRIGGER_ADAPTIVE, "every": oracle.TRIGGER_EVERY,
         "interval": oracle.TRIGGER_INTERVAL}
_FILL = {"prefix": oracle.FILL_PREFIX, "skip": oracle.FILL_SKIP}


def _workload(**kw):
    base = dict(batch=2, n_kv_heads=2, n_prefill=1500, n_components=40, n_clusters=48, iters=3,
                local_buf=40, budget=180, jump_p=0.06)
    base.update(kw)
    return synth.WORKLOADS["long_out"].replace(**base)


def _run(w, T, policy, *, pages=0, graph=True, seed=4):
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    ctx = H.make_ctx(w, max_steps=T)
    if pages:
        ctx.build_pages(0, K, V, pages)
    else:
        ctx.build_index(0, K, V, w.n_clusters, w.iters, seed)
    ctx.set_policy(**policy)
    C = ctx.get_index(0, 0, 0, w.n_prefill)["n_units"]
    idx = {b: [ctx.get_index(0, b, h, w.n_prefill) for h in range(w.n_kv_heads)] for b in range(w.batch)}
    out = torch.zeros(T, w.batch, 1, w.n_heads, 128, device="cuda")
    bnd = torch.zeros(T, w.batch, 1, dtype=torch.uint8, device="cuda")
    r = torch.zeros(T, w.batch, 1, dtype=torch.float32, device="cuda")
    hs = w.n_heads if policy.get("per_head") else w.n_kv_heads   # selection records per head
    nsel = torch.zeros(T, w.batch, 1, hs, dtype=torch.int32, device="cuda")
    sel = torch.full((T, w.batch, 1, hs, ctx.u_cap), -1, dtype=torch.int32, device="cuda")
    if graph:
        ctx.decode_steps(0, q, kn, vn, w.tau, w.budget, out, boundary=bnd, n_selected=nsel,
                         selected_units=sel, r_out=r)
    else:
        for t in range(T):
            ctx.decode_step(0, q[t], kn[t], vn[t], w.tau, w.budget, out[t], boundary=bnd[t],
                            n_selected=nsel[t], selected_units=sel[t], r_out=r[t])
    ctx.sync()
    g = dict(out=out.cpu().numpy(), bnd=bnd.cpu().numpy(), r=r.cpu().numpy(),
             nsel=nsel.cpu().numpy(), sel=sel.cpu().numpy())
    states = [ctx.decode_state(0, b) for b in range(w.batch)]
    segs = {b: [ctx.get_index(0, b, h, w.n_prefill) for h in range(w.n_kv_heads)] for b in range(w.batch)}
    ctx.close()
    return K, V, q, kn, vn, C, idx, g, states, segs


def _check(w, T, policy, *, pages=0, graph=True):
    K, V, q, kn, vn, C, idx, g, states, segs = _run(w, T, policy, pages=pages, graph=graph)
    kw = dict(trigger=_TRIG[policy.get("trigger", "adaptive")], interval=policy.get("interval", 1),
              fill=_FILL[policy.get("fill", "prefix")], page=policy.get("page", 0),
              per_head=policy.get("per_head", False))
    hs = w.n_heads if kw["per_head"] else w.n_kv_heads
    report = []
    for b in range(w.batch):
        assign = np.stack([idx[b][h]["assign"] for h in range(w.n_kv_heads)])
        cent = np.stack([idx[b][h]["centroids"][:C] for h in range(w.n_kv_heads)])
        o = oracle.decode(synth.to_oracle(K[b]), synth.to_oracle(V[b]), assign, cent,
                          synth.to_oracle(q[:, b, 0]), synth.to_oracle(kn[:, b, 0]),
                          synth.to_oracle(vn[:, b, 0]), n_clusters=C, local_buf=w.local_buf,
                          tau=w.tau, budget=w.budget, want_seg_cent=True, **kw)
        assert np.array_equal(g["bnd"][:, b, 0], o["flag"]), np.flatnonzero(g["bnd"][:, b, 0] != o["flag"])[:8]
        assert np.array_equal(g["r"][:, b, 0].view(np.uint32), o["r32"].view(np.uint32))
        assert np.array_equal(g["nsel"][:, b, 0], o["n_sel"])
        for t in range(T):
            for h in range(hs):
                k = o["n_sel"][t, h]
                assert np.array_equal(np.sort(g["sel"][t, b, 0, h, :k]), np.sort(o["sel"][t, h, :k])), (t, h)
        err = np.abs(g["out"][:, b, 0].astype(np.float64) - o["out"])
        assert (err <= H.ATOL + H.RTOL * np.abs(o["out"])).all(), err.max()
        assert states[b]["n_evicted"] == o["n_evicted"] and states[b]["n_forced"] == o["n_forced"]
        for h in range(w.n_kv_heads):
            ix = segs[b][h]
            assert np.array_equal(ix["unit_row"][C:ix["n_units"]] - w.n_prefill, o["seg_start"])
            assert np.array_equal(ix["unit_len"][C:ix["n_units"]], o["seg_len"])
            assert np.array_equal(ix["centroids"][C:ix["n_units"]].view(np.uint32),
                                  o["seg_cent"][:, h].view(np.uint32))
        report.append((int(o["flag"].sum()), o["n_evicted"], o["n_forced"]))
    return report


def test_every_token_retrieval():
    rep = _check(_workload(), 300, dict(trigger="every"))
    assert all(n == 300 for n, _, _ in rep)


@pytest.mark.parametrize("interval", [1, 7, 64])
def test_fixed_interval_retrieval(interval):
    rep = _check(_workload(), 300, dict(trigger="interval", interval=interval))
    assert all(n == len(range(0, 300, interval)) for n, _, _ in rep)


@pytest.mark.parametrize("graph", [True, False])
def test_skip_and_continue_fill(graph):
    # many units of uneven length near the cut: budget not a multiple of the sizes
    rep = _check(_workload(budget=173), 300, dict(fill="skip"), graph=graph)
    assert sum(n for n, _, _ in rep) > 2


def test_skip_fill_differs_from_prefix_somewhere():
    """The variant is not vacuous on this workload: some retrieval takes more
    tokens with skip-and-continue than with the stop-at-first-misfit rule."""
    w = _workload(budget=173)
    _, _, _, _, _, _, _, g_skip, _, _ = _run(w, 200, dict(fill="skip"))
    _, _, _, _, _, _, _, g_pre, _, _ = _run(w, 200, dict(fill="prefix"))
    assert (g_skip["nsel"] >= g_pre["nsel"]).all() and (g_skip["nsel"] > g_pre["nsel"]).any()


def test_output_pages():
    rep = _check(_workload(), 300, dict(page=16))
    assert all(f == 0 for _, _, f in rep)


def test_page_units_every_token():
    """The page-granular, every-token baseline: prefill page-mean units,
    16-token output pages, a retrieval at every step."""
    w = _workload(n_clusters=94)   # ceil(1500 / 16) units
    _check(w, 300, dict(trigger="every", page=16), pages=16)


def test_combined_policy_single_steps():
    _check(_workload(budget=173), 160, dict(trigger="interval", interval=5, fill="skip", page=8),
           graph=False)


def test_build_pages_matches_oracle():
    w = _workload(n_prefill=1000, n_clusters=63)
    K, V = synth.prefill(w, 0, "cuda")
    ctx = H.make_ctx(w)
    for page in (16, 1000, 17):
        ctx.build_pages(0, K, V, page)
        for b in range(w.batch):
            for h in range(w.n_kv_heads):
                ix = ctx.get_index(0, b, h, w.n_prefill)
                a, cent = oracle.page_index(synth.to_oracle(K[b, h]), page)
                c = len(cent)
                assert ix["n_units"] == c
                assert np.array_equal(ix["assign"], a)
                assert np.array_equal(ix["perm"], np.arange(w.n_prefill))
                assert np.array_equal(ix["centroids"][:c].view(np.uint32), cent.view(np.uint32))
                assert np.array_equal(ix["unit_len"][:c], np.bincount(a))
    with pytest.raises(_lib.LKVError) as e:
        ctx.build_pages(0, K, V, 15)            # 67 pages > max_clusters 63
    assert e.value.status == _lib.LKV_EINVAL
    ctx.close()


def test_policy_argument_checks():
    w = _workload(n_prefill=300, n_clusters=10)
    ctx = H.make_ctx(w)
    for bad in (dict(trigger=3, interval=1, fill=0, page=0), dict(trigger=2, interval=0, fill=0, page=0),
                dict(trigger=0, interval=1, fill=2, page=0), dict(trigger=0, interval=1, fill=0, page=-1),
                dict(trigger=0, interval=1, fill=0, page=0, per_head=2)):
        with pytest.raises(_lib.LKVError) as e:
            _lib.lkv_set_policy(ctx._ctx, **bad)
        assert e.value.status == _lib.LKV_EINVAL
    ctx.close()


def test_skip_fill_above_smem_units_reports_capacity():
    w = _workload(batch=1, n_kv_heads=1, n_prefill=4200, n_clusters=4200, iters=1, budget=50)
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=2)
    ctx = H.make_ctx(w, max_steps=2)
    ctx.build_index(0, K, V, w.n_clusters, 1, 1)
    ctx.set_policy(fill="skip")
    out = torch.zeros(1, 1, w.n_heads, 128, device="cuda")
    ctx.decode_step(0, q[0], kn[0], vn[0], w.tau, w.budget, out)
    with pytest.raises(_lib.LKVError) as e:
        ctx.sync()
    assert e.value.status == _lib.LKV_ECAPACITY
    ctx.close()


@pytest.mark.parametrize("graph", [True, False])
def test_per_head_selection(graph):
    """A selection per query head: every head's set bit-exact, each head's
    attention over its own set (the kernel reads the group's union once and
    masks each head to its own rows)."""
    rep = _check(_workload(budget=150), 300, dict(per_head=True), graph=graph)
    assert sum(n for n, _, _ in rep) > 2


def test_per_head_with_skip_fill_and_every_step():
    _check(_workload(budget=173, n_kv_heads=1, group=8), 200,
           dict(per_head=True, fill="skip", trigger="every"))


def test_per_head_rejected_without_streaming_attention():
    w = _workload(n_prefill=300, n_clusters=10, dtype="fp32")
    ctx = H.make_ctx(w)
    with pytest.raises(_lib.LKVError) as e:
        ctx.set_policy(per_head=True)
    assert e.value.status == _lib.LKV_EINVAL
    ctx.close()


def test_graph_of_2048_steps_matches_oracle():
    """One call of 2100 steps replays a 2048-step graph (32 chunks, so the
    selection of chunk j waits for the attentions of chunk j - 2) and runs
    the last 52 steps singly; every decision and output matches the oracle."""
    _check(_workload(local_buf=24, jump_p=0.08), 2100, dict())
