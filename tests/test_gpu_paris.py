"""GPU parity of the ParisKV-style token selector (lkv_build_paris) against
the oracle's restatement of the same pipeline (ParisKV technical summary,
核心算法创新 1-2): the same tokens at every retrieval step (bit-exact: the
metadata is computed from exact integer rotations and the same
floating-point operation order on both sides), the same flags and segments,
and the attention over the selected tokens and the local buffer within the
tolerance of the other parity tests."""
import numpy as np
import pytest
import torch

import oracle
import synth
from cluster_indexed_kv_gb300 import _lib
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _workload(**kw):
    base = dict(batch=2, n_kv_heads=2, n_prefill=1500, n_components=40, n_clusters=64, iters=1,
                local_buf=40, budget=150, jump_p=0.06, n_steps=300)
    base.update(kw)
    return synth.WORKLOADS["long_out"].replace(**base)


def _run_and_check(w, prm, *, graph=True, policy=None, T=None):
    T = T or w.n_steps
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    ctx = H.make_ctx(w, max_steps=T)
    ctx.build_paris(0, K, V, **prm)
    if policy:
        ctx.set_policy(**policy)
    out = torch.zeros(T, w.batch, 1, w.n_heads, 128, device="cuda")
    bnd = torch.zeros(T, w.batch, 1, dtype=torch.uint8, device="cuda")
    r = torch.zeros(T, w.batch, 1, dtype=torch.float32, device="cuda")
    nsel = torch.zeros(T, w.batch, 1, w.n_kv_heads, dtype=torch.int32, device="cuda")
    sel = torch.full((T, w.batch, 1, w.n_kv_heads, ctx.u_cap), -1, dtype=torch.int32, device="cuda")
    if graph:
        ctx.decode_steps(0, q, kn, vn, w.tau, w.budget, out, boundary=bnd, n_selected=nsel,
                         selected_units=sel, r_out=r)
    else:
        for t in range(T):
            ctx.decode_step(0, q[t], kn[t], vn[t], w.tau, w.budget, out[t], boundary=bnd[t],
                            n_selected=nsel[t], selected_units=sel[t], r_out=r[t])
    ctx.sync()
    g = dict(out=out.cpu().numpy(), bnd=bnd.cpu().numpy(), r=r.cpu().numpy(), nsel=nsel.cpu().numpy(),
             sel=sel.cpu().numpy())
    states = [ctx.decode_state(0, b) for b in range(w.batch)]
    ctx.close()
    trig = {"every": oracle.TRIGGER_EVERY, "interval": oracle.TRIGGER_INTERVAL}.get(
        (policy or {}).get("trigger"), oracle.TRIGGER_ADAPTIVE)
    N, n_cap = w.n_prefill, w.n_prefill   # the test contexts have max_prefill = n_prefill
    for b in range(w.batch):
        o = oracle.decode(synth.to_oracle(K[b]), synth.to_oracle(V[b]), None, None,
                          synth.to_oracle(q[:, b, 0]), synth.to_oracle(kn[:, b, 0]),
                          synth.to_oracle(vn[:, b, 0]), n_clusters=0, local_buf=w.local_buf,
                          tau=w.tau, budget=w.budget, paris=prm, trigger=trig,
                          interval=(policy or {}).get("interval", 1))
        assert np.array_equal(g["bnd"][:, b, 0], o["flag"])
        assert np.array_equal(g["r"][:, b, 0].view(np.uint32), o["r32"].view(np.uint32))
        assert np.array_equal(g["nsel"][:, b, 0], o["n_sel"])
        for t in range(T):
            for h in range(w.n_kv_heads):
                k = o["n_sel"][t, h]
                rows = g["sel"][t, b, 0, h, :k].astype(np.int64)
                ids = np.where(rows < n_cap, rows, N + (rows - n_cap))  # decode t at row n_cap + t
                assert np.array_equal(np.sort(ids), np.sort(o["sel"][t, h, :k])), (b, t, h)
        err = np.abs(g["out"][:, b, 0].astype(np.float64) - o["out"])
        assert (err <= H.ATOL + H.RTOL * np.abs(o["out"])).all(), err.max()
        assert states[b]["n_evicted"] == o["n_evicted"] and states[b]["n_forced"] == o["n_forced"]
    return g


@pytest.mark.parametrize("graph", [True, False])
def test_paris_selector_parity(graph):
    g = _run_and_check(_workload(), dict(rho=4, n_cand=400, seed=7), graph=graph)
    assert g["bnd"].sum() > 4


def test_paris_every_step_with_wide_vote():
    """Every step retrieves; rho 15 and few candidates (ties at the cut)."""
    _run_and_check(_workload(budget=100, n_kv_heads=1, group=8), dict(rho=15, n_cand=130, seed=3),
                   policy=dict(trigger="every"), T=200)


def test_paris_all_tokens_is_full_attention():
    """Budget and candidates above every token: every prefill and evicted
    token is attended (the FullCache configuration)."""
    w = _workload(n_prefill=600, budget=1000, local_buf=16, n_clusters=900)  # u_cap >= budget
    _run_and_check(w, dict(rho=2, n_cand=1000, seed=1), policy=dict(trigger="every"), T=140)


def test_paris_argument_checks():
    w = _workload(n_prefill=300)
    K, V = synth.prefill(w, 0, "cuda")
    ctx = H.make_ctx(w)
    for bad in (dict(rho=0, n_cand=10, seed=1), dict(rho=16, n_cand=10, seed=1),
                dict(rho=4, n_cand=0, seed=1), dict(rho=4, n_cand=5000, seed=1)):
        with pytest.raises(_lib.LKVError) as e:
            ctx.build_paris(0, K, V, **bad)
        assert e.value.status == _lib.LKV_EINVAL
    ctx.build_paris(0, K, V, rho=4, n_cand=100, seed=1)
    with pytest.raises(_lib.LKVError):
        ctx.build_paris(0, K, V, rho=4, n_cand=100, seed=2)     # params fixed by the first build
    with pytest.raises(_lib.LKVError):
        ctx.build_index(0, K, V, 16, 1, 1)                      # no clusters on this context
    with pytest.raises(_lib.LKVError):
        ctx.set_policy(per_head=True)
    ctx.close()
    ctx = H.make_ctx(w)
    ctx.build_index(0, K, V, 16, 1, 1)
    with pytest.raises(_lib.LKVError):
        ctx.build_paris(0, K, V, rho=4, n_cand=100, seed=1)     # a layer has clusters
    ctx.close()
