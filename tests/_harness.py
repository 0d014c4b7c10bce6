"""Shared helpers of the GPU parity tests: drive liblkv through its C ABI on
seeded synthetic inputs and run the oracle on the very same tensors."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

ATOL, RTOL = 2e-3, 1e-2   # attention outputs: bf16 in, fp32 accumulate


def rounding_update_keys():
    """1024 bf16 keys in two far-apart groups of 512 (all dimensions 16, and
    all -16). In token order, dimension 0 of the first group holds 497 x 16,
    10 x 24 and 2^-11 (partial sums reach 2^13 = 8192 + 2^-11), then
    -2^-33, 2^-33 + 2^-40, -2^-33, 2^-33 + 2^-40. A double-precision sum in
    token order rounds each 2^-40 away (a tie to even at 2^13) and ends at
    8192 + 2^-11, whose mean 16 + 2^-20 is a float midpoint that rounds to
    16. The exact sum carries 2^-39 more, and its mean rounds to 16 + 2^-19.
    Returns (keys [1024, 128] float32, an init seed that draws one key from
    each group)."""
    keys = np.full((1024, 128), 16.0, np.float32)
    keys[512:] = -16.0
    col = [16.0] * 497 + [24.0] * 10 + [2.0 ** -11] + [-2.0 ** -33, 2.0 ** -33 + 2.0 ** -40] * 2
    keys[:512, 0] = np.array(col, np.float64).astype(np.float32)
    return keys, 8


def make_ctx(w: synth.Workload, max_steps=None, max_budget=None):
    import cluster_indexed_kv_gb300 as lkv
    return lkv.Context(batch=w.batch, n_layers=w.n_layers, n_kv_heads=w.n_kv_heads,
                       group=w.group, dtype=w.torch_dtype, local_buf=w.local_buf,
                       max_clusters=w.n_clusters, max_prefill=w.n_prefill,
                       max_steps=max_steps or w.n_steps, max_budget=max_budget or w.budget,
                       offload=w.offload)


def gpu_index(ctx, layer, b, h, n):
    return ctx.get_index(layer, b, h, n)


def run_decode(ctx, w, q, kn, vn, *, tau=None, budget=None, keep_sel=True, layers=None):
    """Drive T decode steps (all sequences, the given layers in one call each
    step). Returns host arrays: out [T,B,nl,H,d], boundary [T,B,nl], r [T,B,nl],
    n_sel [T,B,nl,Hkv] and, with keep_sel, sel: dict (t, b, li, h) -> sorted ids
    for boundary steps and t = 0."""
    tau = w.tau if tau is None else tau
    budget = w.budget if budget is None else budget
    T, B, nl = q.shape[0], q.shape[1], q.shape[2]
    l0 = 0 if layers is None else layers[0]
    dev = q.device
    H, Hkv = w.n_heads, w.n_kv_heads
    out = torch.empty(T, B, nl, H, 128, dtype=torch.float32, device=dev)
    bnd = torch.zeros(T, B, nl, dtype=torch.uint8, device=dev)
    r = torch.zeros(T, B, nl, dtype=torch.float32, device=dev)
    nsel = torch.zeros(T, B, nl, Hkv, dtype=torch.int32, device=dev)
    K = 32
    ring = torch.full((K, B, nl, Hkv, ctx.u_cap), -1, dtype=torch.int32, device=dev)
    sel = {}

    def drain(t0, t1):
        b_h = bnd[t0:t1].cpu().numpy()
        n_h = nsel[t0:t1].cpu().numpy()
        rg = ring.cpu().numpy()
        for t in range(t0, t1):
            for b in range(B):
                for li in range(nl):
                    if b_h[t - t0, b, li]:
                        for h in range(Hkv):
                            k = n_h[t - t0, b, li, h]
                            sel[(t, b, li, h)] = np.sort(rg[t % K, b, li, h, :k])

    for t in range(T):
        ctx.decode_step(l0, q[t], kn[t], vn[t], tau, budget, out[t], n_layers=nl,
                        selected_units=ring[t % K] if keep_sel else None,
                        n_selected=nsel[t], boundary=bnd[t], r_out=r[t])
        if keep_sel and (t % K == K - 1 or t == T - 1):
            drain(t - (t % K), t + 1)
    ctx.sync()
    return dict(out=out.cpu().numpy(), boundary=bnd.cpu().numpy(), r=r.cpu().numpy(),
                n_sel=nsel.cpu().numpy(), sel=sel)


def oracle_decode(w, K, V, idx, q, kn, vn, b, li, *, layer=None, tau=None, budget=None,
                  attn_mask=None):
    """Oracle run of sequence b, call-layer li, teacher-forced from idx: a list
    over kv heads of dicts with 'assign' and 'centroids' (fp32, clusters first)."""
    tau = w.tau if tau is None else tau
    budget = w.budget if budget is None else budget
    C = w.n_clusters
    assign = np.stack([idx[h]["assign"] for h in range(w.n_kv_heads)])
    cent = np.stack([idx[h]["centroids"][:C] for h in range(w.n_kv_heads)])
    return oracle.decode(synth.to_oracle(K[b]), synth.to_oracle(V[b]), assign, cent,
                         synth.to_oracle(q[:, b, li]), synth.to_oracle(kn[:, b, li]),
                         synth.to_oracle(vn[:, b, li]), n_clusters=C, local_buf=w.local_buf,
                         tau=tau, budget=budget, attn_mask=attn_mask, want_seg_cent=True)


def compare_decode(g, o, w, b, li, *, attn_mask=None, check_sel=True):
    """Bit-exact decisions, tolerance on attention. Returns a short report."""
    T = o["flag"].shape[0]
    Hkv = w.n_kv_heads
    bnd = g["boundary"][:, b, li]
    assert np.array_equal(bnd, o["flag"]), f"boundary flags differ at {np.flatnonzero(bnd != o['flag'])[:10]}"
    rg = g["r"][:, b, li]
    assert np.array_equal(rg.view(np.uint32), o["r32"].view(np.uint32)), "r_t differs"
    assert np.array_equal(g["n_sel"][:, b, li], o["n_sel"]), "n_selected differs"
    if check_sel:
        for t in np.flatnonzero(o["flag"]):
            for h in range(Hkv):
                k = o["n_sel"][t, h]
                want = np.sort(o["sel"][t, h, :k])
                assert np.array_equal(g["sel"][(t, b, li, h)], want), f"selection differs t={t} h={h}"
    steps = np.arange(T) if attn_mask is None else np.flatnonzero(attn_mask)
    got = g["out"][steps, b, li].astype(np.float64)
    want = o["out"][steps]
    err = np.abs(got - want)
    ok = err <= ATOL + RTOL * np.abs(want)
    assert ok.all(), f"attention mismatch: max abs err {err.max():.3e}"
    return dict(max_abs_err=float(err.max()), n_boundary=int(o["flag"].sum()),
                n_evicted=o["n_evicted"], n_forced=o["n_forced"])


def compare_segments(ctx, w, o, b, li, layer):
    """Evicted segments: same order, start, length and index vector."""
    st = ctx.decode_state(layer, b)
    assert st["n_evicted"] == o["n_evicted"], (st["n_evicted"], o["n_evicted"])
    assert st["n_forced"] == o["n_forced"]
    C = w.n_clusters
    for h in range(w.n_kv_heads):
        ix = ctx.get_index(layer, b, h, w.n_prefill)
        assert ix["n_units"] == C + o["n_evicted"]
        seg_row = ix["unit_row"][C:] - w.n_prefill
        assert np.array_equal(seg_row, o["seg_start"])
        assert np.array_equal(ix["unit_len"][C:], o["seg_len"])
        assert np.array_equal(ix["centroids"][C:].view(np.uint32),
                              o["seg_cent"][:, h].view(np.uint32))


# ---------------------------------------------------------------- graph path at full size

def run_graph(ctx, w, q, kn, vn, *, seqs, tau=None, budget=None, chunk=512, keep_out=True,
              per_head=False):
    """A whole run through lkv_decode_steps (the pipelined CUDA graph that the
    benchmark times), in chunks of `chunk` steps. Returns host arrays:
    boundary [T,B], r [T,B], n_sel [T,B,Hs] for every sequence (Hs = Hkv, or
    H with per-head selection records); for the sequences in `seqs`, out
    {b: [T,H,d]} and the selections at retrieval steps sel {(t, b, h):
    ascending ids}."""
    tau = w.tau if tau is None else tau
    budget = w.budget if budget is None else budget
    T, B = q.shape[0], q.shape[1]
    H = w.n_heads
    Hkv = H if per_head else w.n_kv_heads
    dev = q.device
    out = torch.empty(T, B, 1, H, 128, dtype=torch.float32, device=dev)
    bnd = torch.zeros(T, B, 1, dtype=torch.uint8, device=dev)
    r = torch.zeros(T, B, 1, dtype=torch.float32, device=dev)
    nsel = torch.zeros(T, B, 1, Hkv, dtype=torch.int32, device=dev)
    selbuf = torch.full((chunk, B, 1, Hkv, ctx.u_cap), -1, dtype=torch.int32, device=dev)
    sel = {}
    sidx = torch.tensor(list(seqs), dtype=torch.long, device=dev)
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        ctx.decode_steps(0, q[c0:c1], kn[c0:c1], vn[c0:c1], tau, budget, out[c0:c1],
                         selected_units=selbuf[:c1 - c0], n_selected=nsel[c0:c1],
                         boundary=bnd[c0:c1], r_out=r[c0:c1])
        ctx.sync()
        fl = bnd[c0:c1, :, 0].index_select(1, sidx).cpu().numpy()
        ns = nsel[c0:c1, :, 0].index_select(1, sidx).cpu().numpy()
        kmax = int(ns.max()) if ns.size else 0
        steps = np.flatnonzero(fl.any(axis=1))
        if len(steps) and kmax:
            st = torch.as_tensor(steps, device=dev)
            got = selbuf[:, :, 0, :, :kmax].index_select(0, st).index_select(1, sidx).cpu().numpy()
            for i, t in enumerate(steps):
                for j, b in enumerate(seqs):
                    if fl[t, j]:
                        for h in range(Hkv):
                            sel[(c0 + int(t), b, h)] = np.sort(got[i, j, h, :ns[t, j, h]])
    res = dict(boundary=bnd[:, :, 0].cpu().numpy(), r=r[:, :, 0].cpu().numpy(),
               n_sel=nsel[:, :, 0].cpu().numpy(), sel=sel)
    if keep_out:
        res["out"] = {b: out[:, b, 0].cpu().numpy() for b in seqs}
    return res


def spawn_pool(workers):
    """Process pool for oracle work (spawn: safe after the parent used the GPU)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    return cf.ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))


def oracle_inputs(tmpdir, tag, w, K, V, idx, q, kn, vn, b, li=0):
    """Write one sequence's oracle inputs (teacher-forced index `idx`: a list
    over KV heads of dicts with 'assign' and 'centroids') as .npy files."""
    import os
    C = w.n_clusters
    arrays = dict(keys=synth.to_oracle(K[b]), values=synth.to_oracle(V[b]),
                  assign=np.stack([ix["assign"] for ix in idx]).astype(np.int32),
                  cent=np.stack([ix["centroids"][:C] for ix in idx]).astype(np.float32),
                  q=synth.to_oracle(q[:, b, li]), k_new=synth.to_oracle(kn[:, b, li]),
                  v_new=synth.to_oracle(vn[:, b, li]))
    paths = {}
    for k, a in arrays.items():
        p = os.path.join(str(tmpdir), f"{tag}_{k}.npy")
        np.save(p, a)
        paths[k] = p
    return paths


def compare_graph_run(g, o, w, b, *, label=""):
    """Bit-exact flags, r_t, selection sizes and selections; tolerance on the
    attention outputs at the oracle's sampled steps."""
    bnd = g["boundary"][:, b]
    assert np.array_equal(bnd, o["flag"]), \
        f"{label} flags differ at {np.flatnonzero(bnd != o['flag'])[:10]}"
    assert np.array_equal(g["r"][:, b].view(np.uint32), o["r32"].view(np.uint32)), f"{label} r_t differs"
    assert np.array_equal(g["n_sel"][:, b], o["n_sel"]), f"{label} n_selected differs"
    n_checked = 0
    for (t, h), want in o["sel"].items():
        assert np.array_equal(g["sel"][(t, b, h)], want), f"{label} selection differs t={t} h={h}"
        n_checked += 1
    steps = o["attn_steps"]
    got = g["out"][b][steps].astype(np.float64)
    err = np.abs(got - o["out"])
    ok = err <= ATOL + RTOL * np.abs(o["out"])
    assert ok.all(), f"{label} attention mismatch: max abs err {err.max():.3e}"
    return dict(n_sel_checked=n_checked, n_attn_steps=len(steps), max_abs_err=float(err.max()),
                n_boundary=int(o["flag"].sum()), n_evicted=o["n_evicted"])
