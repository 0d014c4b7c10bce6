"""Pins of the CPU oracle against facts fixed outside the oracle itself:
published generator outputs, closed forms, textbook properties of Lloyd's
K-means and softmax attention, brute force on tiny inputs, and the FullCache
special case (every step retrieves with a budget covering every token, so the
sparse attention must equal full attention). No GPU needed."""
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(12345)


def bf16(x):
    return oracle.f32_to_bf16_bits(np.asarray(x, np.float32))


def unbf16(b):
    return oracle.bf16_bits_to_f32(b)


# ------------------------------------------------------------------ splitmix64

def test_splitmix64_published_vectors():
    with open(os.path.join(GOLDEN, "splitmix64.txt")) as f:
        lines = [l for l in f if l.strip() and not l.startswith("#")]
    assert len(lines) == 2
    for line in lines:
        seed_s, outs = line.split(":")
        seed = int(seed_s, 0)
        want = [int(x, 0) for x in outs.split()]
        got = [int(x) for x in oracle.splitmix64(seed, len(want))]
        assert got == want


def test_init_indices_distinct_and_full_shuffle_is_permutation():
    for n, c, seed in [(10, 10, 7), (2048, 32, 1), (5, 1, 99), (131072, 8192, 3)]:
        idx = oracle.init_indices(n, c, seed)
        assert idx.min() >= 0 and idx.max() < n
        assert len(set(idx.tolist())) == c
    full = oracle.init_indices(1000, 1000, 5)
    assert sorted(full.tolist()) == list(range(1000))
    with pytest.raises(ValueError):
        oracle.init_indices(4, 5, 1)


def test_init_indices_first_draw_matches_generator():
    # the first index is (first splitmix64 output) mod n
    for seed in (1, 2, 0xDEADBEEF):
        first = int(oracle.splitmix64(seed, 1)[0])
        assert oracle.init_indices(1000, 3, seed)[0] == first % 1000


# ------------------------------------------------------------------ bf16

def test_bf16_rounding_matches_torch():
    import torch
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0, 65504.0, 1e-30, 3.4e38, -2.5e-8],
                                 np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16(x), want)
    # ties to even: 1 + 2^-8 is halfway between two bf16 values
    assert unbf16(bf16(np.float32(1.0 + 2 ** -8)))[()] == 1.0
    assert unbf16(bf16(np.float32(1.0 + 3 * 2 ** -8)))[()] == 1.0 + 2 ** -6


# ------------------------------------------------------------------ K-means

def test_sqdist_closed_form():
    k = np.zeros(128, np.float32); k[0] = 3
    c = np.zeros(128, np.float32); c[1] = 4
    assert oracle.sqdist(k, c) == 25.0
    kb = bf16(k)
    assert oracle.sqdist(kb, c) == 25.0


def test_assign_brute_force_and_ties():
    d = 8
    keys = rng.standard_normal((50, d)).astype(np.float32)
    cent = rng.standard_normal((7, d)).astype(np.float32)
    a = oracle.assign(keys, cent)
    dist = ((keys[:, None, :].astype(np.float64) - cent[None].astype(np.float64)) ** 2).sum(-1)
    assert np.array_equal(a, dist.argmin(1))
    # exact tie between centroid 0 and 1 -> lowest id; 2 and 3 -> 2
    k = np.zeros((2, d), np.float32)
    k[1, 0] = 10
    c = np.zeros((4, d), np.float32)
    c[0, 1], c[1, 1] = 1, -1
    c[2, 0], c[3, 0] = 11, 11
    c[2, 2], c[3, 2] = 1, -1
    assert oracle.assign(k, c).tolist() == [0, 2]


def test_update_is_member_mean_and_empty_keeps_centroid():
    d = 16
    keys = rng.standard_normal((200, d)).astype(np.float32)
    a = rng.integers(0, 5, 200).astype(np.int32)
    a[a == 3] = 4  # cluster 3 empty
    old = rng.standard_normal((5, d)).astype(np.float32)
    cent, cnt, inexact = oracle.update(keys, a, old)
    for j in range(5):
        m = a == j
        assert cnt[j] == m.sum()
        if m.any():
            want = keys[m].astype(np.float64).mean(0)
            assert np.allclose(cent[j], want, atol=1e-6, rtol=0)
        else:
            assert np.array_equal(cent[j], old[j])
    # bf16 keys: member sums are exact in double, so the centroid is the
    # correctly rounded mean of the exact sum
    kb = bf16(keys)
    centb, _, inexact_b = oracle.update(kb, a, old)
    assert inexact_b == 0
    kf = unbf16(kb).astype(np.float64)
    for j in (0, 1, 2, 4):
        want = (kf[a == j].sum(0) / (a == j).sum()).astype(np.float32)
        assert np.array_equal(centb[j], want)


def test_update_sums_in_token_order_not_exactly():
    """The member sums are double-precision sums in token order, rounded at
    every step (the plain reading of "fp64 member sums"), not the exact sum
    rounded once. On this construction the two give means one float ulp
    apart: 16.0 from the token-order sum, 16 + 2^-19 from the exact one."""
    from fractions import Fraction
    from tests import _harness as H
    keys, _ = H.rounding_update_keys()
    kb = bf16(keys)
    assert np.array_equal(unbf16(kb), keys)  # every value is a bf16
    a = np.repeat(np.arange(2, dtype=np.int32), 512)
    cent, cnt, inexact = oracle.update(kb, a, np.zeros((2, 128), np.float32))
    assert cnt.tolist() == [512, 512]
    assert inexact == 2  # the two additions of 2^-33 + 2^-40 round (ties to even)
    assert cent[0, 0] == np.float32(16.0)
    exact = sum(Fraction(float(x)) for x in keys[:512, 0]) / 512
    assert np.float32(float(exact)) == np.float32(16.0 + 2.0 ** -19)
    assert np.all(cent[0, 1:] == 16.0) and np.all(cent[1] == -16.0)


def test_well_separated_mixture_recovers_partition():
    # textbook case: components far apart, one initial centroid per component
    # -> one Lloyd round returns the generating partition and its means
    d, C, per = 32, 6, 40
    means = np.zeros((C, d), np.float32)
    for j in range(C):
        means[j, j] = 100.0
    lab = np.repeat(np.arange(C), per)
    rng.shuffle(lab)
    keys = (means[lab] + rng.standard_normal((C * per, d)).astype(np.float32)).astype(np.float32)
    init = np.stack([keys[np.flatnonzero(lab == j)[0]] for j in range(C)])
    a = oracle.assign(keys, init)
    assert np.array_equal(a, lab)
    cent, cnt, _ = oracle.update(keys, a, init)
    assert np.array_equal(cnt, np.full(C, per))
    for j in range(C):
        assert np.allclose(cent[j], keys[lab == j].astype(np.float64).mean(0), atol=1e-5)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_kmeans_objective_monotone_and_composition(dtype):
    n, d, c, iters = 600, 16, 12, 8
    keys = (rng.standard_normal((c, d))[rng.integers(0, c, n)] * 1.0
            + 0.4 * rng.standard_normal((n, d))).astype(np.float32)
    if dtype == "bf16":
        keys = bf16(keys)
    dt = oracle.dtype_of(keys)
    r = oracle.kmeans(keys, c, iters, seed=11, trace=True)
    tc, ta = r["trace_cent"], r["trace_assign"]
    # the run is init + (assign with operand, update) repeated
    idx = oracle.init_indices(n, c, 11)
    kf = unbf16(keys) if dtype == "bf16" else keys
    assert np.array_equal(tc[0], kf[idx])
    cent = tc[0].copy()
    for it in range(iters):
        op = oracle.operand(cent, dt)
        a = oracle.assign(keys, op)
        assert np.array_equal(a, ta[it])
        cent, cnt, _ = oracle.update(keys, a, cent)
        assert np.array_equal(cent, tc[it + 1])
    assert np.array_equal(r["assign"], ta[-1]) and np.array_equal(r["cent"], tc[-1])
    # argmin step can only lower J for fixed centroids; mean step can only lower
    # J for a fixed assignment (exact for the unrounded centroid up to the
    # float rounding of the mean)
    for it in range(1, iters):
        op = oracle.operand(tc[it], dt)
        j_new = oracle.objective(keys, op, ta[it])
        j_old = oracle.objective(keys, op, ta[it - 1])
        assert j_new <= j_old
        j_mean = oracle.objective(keys, tc[it + 1], ta[it])
        j_prev = oracle.objective(keys, tc[it], ta[it])
        assert j_mean <= j_prev * (1 + 1e-9)
    # end-to-end objective (with operand centroids) non-increasing
    js = [oracle.objective(keys, oracle.operand(tc[it + 1], dt), ta[it]) for it in range(iters)]
    tol = 1e-9 if dtype == "fp32" else 1e-3
    for a_, b_ in zip(js, js[1:]):
        assert b_ <= a_ * (1 + tol)


def test_kmeans_centroids_are_member_means():
    n, d, c = 500, 128, 20
    keys = bf16(rng.standard_normal((n, d)))
    r = oracle.kmeans(keys, c, 5, seed=3)
    kf = unbf16(keys).astype(np.float64)
    for j in range(c):
        m = r["assign"] == j
        assert r["count"][j] == m.sum()
        if m.any():
            assert np.array_equal(r["cent"][j], (kf[m].sum(0) / m.sum()).astype(np.float32))


# ------------------------------------------------------------------ boundary

def _boundary_case(rel, h, d=128):
    qp = rng.standard_normal((h, d)).astype(np.float32)
    qc = np.empty_like(qp)
    for i, r in enumerate(rel):
        if r == "same":
            qc[i] = qp[i]
        elif r == "neg":
            qc[i] = -qp[i]
        elif r == "scaled":
            qc[i] = 3 * qp[i]
        elif r == "orth":
            # exactly orthogonal in float arithmetic: disjoint supports
            qp[i, d // 2:] = 0
            qc[i] = 0
            qc[i, d // 2:] = rng.standard_normal(d - d // 2)
    return qp, qc


def test_boundary_golden_cases():
    with open(os.path.join(GOLDEN, "boundary_cases.txt")) as f:
        rows = [l for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 7
    for row in rows:
        name, h, rel, want, tau, trig = (x.strip() for x in row.split("|"))
        qp, qc = _boundary_case(rel.split(), int(h))
        r32, r64 = oracle.boundary_r(qp, qc)
        assert abs(r32 - float(want)) <= 2e-7, name
        assert abs(r64 - float(want)) <= 1e-12, name
        assert int(r32 < float(tau)) == int(trig), name


def test_boundary_matches_mean_cosine_and_is_head_symmetric():
    for dtype in ("fp32", "bf16"):
        qp = rng.standard_normal((32, 128)).astype(np.float32)
        qc = (qp + 0.3 * rng.standard_normal((32, 128))).astype(np.float32)
        if dtype == "bf16":
            qp, qc = bf16(qp), bf16(qc)
        a = (unbf16(qp) if dtype == "bf16" else qp).astype(np.float64)
        b = (unbf16(qc) if dtype == "bf16" else qc).astype(np.float64)
        want = np.mean((a * b).sum(1) / np.linalg.norm(a, axis=1) / np.linalg.norm(b, axis=1))
        r32, r64 = oracle.boundary_r(qp, qc)
        assert abs(r64 - want) < 1e-12
        assert abs(r32 - want) < 2e-6
        perm = rng.permutation(32)
        r32p, r64p = oracle.boundary_r(qp[perm], qc[perm])
        assert abs(r64p - r64) < 1e-12 and abs(r32p - r32) < 2e-6
    z = np.zeros((2, 128), np.float32)
    o = rng.standard_normal((2, 128)).astype(np.float32)
    assert oracle.boundary_r(z, o) == (0.0, 0.0)


# ------------------------------------------------------------------ scoring + selection

def test_group_scores_are_group_sum_dot_products():
    G, d, U = 4, 128, 300
    q = rng.standard_normal((G, d)).astype(np.float32)
    cent = rng.standard_normal((U, d)).astype(np.float32)
    s = oracle.group_scores(q, cent)
    exact = cent.astype(np.float64) @ q.astype(np.float64).sum(0)
    bound = 2 * (d + G) * 2.0 ** -24 * (np.abs(cent) @ np.abs(q).sum(0))
    assert np.all(np.abs(s - exact) <= bound)
    # single head, small integers: every intermediate is exact
    qi = rng.integers(-8, 8, (1, d)).astype(np.float32)
    ci = rng.integers(-8, 8, (U, d)).astype(np.float32)
    assert np.array_equal(oracle.group_scores(qi, ci),
                          (ci.astype(np.int64) @ qi[0].astype(np.int64)).astype(np.float32))


def _selection_properties(s, ln, budget, sel, ntok):
    order = sorted(range(len(s)), key=lambda u: (-float(s[u]), u))
    k = len(sel)
    assert list(sel) == order[:k]                      # a prefix of the order
    assert ntok == sum(int(ln[u]) for u in sel) <= budget
    if k < len(s):
        assert ntok + int(ln[order[k]]) > budget       # stopped at first misfit


def test_select_brute_force_unique_prefix():
    for trial in range(300):
        u = int(rng.integers(1, 8))
        s = rng.integers(-3, 4, u).astype(np.float32)   # many score ties
        ln = rng.integers(0, 6, u).astype(np.int32)
        budget = int(rng.integers(0, 20))
        sel, ntok = oracle.select(s, ln, budget)
        _selection_properties(s, ln, budget, sel, ntok)
        # brute force: exactly one (ordering, prefix) pair satisfies the rule
        valid = []
        for perm in itertools.permutations(range(u)):
            if any((-s[a], a) > (-s[b], b) for a, b in zip(perm, perm[1:])):
                continue
            tok, take = 0, []
            for x in perm:
                if tok + ln[x] > budget:
                    break
                tok += ln[x]
                take.append(x)
            valid.append(take)
        assert len(valid) == 1 and valid[0] == list(sel)


def test_select_budget_covers_all_and_zero_budget():
    s = rng.standard_normal(50).astype(np.float32)
    ln = rng.integers(1, 30, 50).astype(np.int32)
    sel, ntok = oracle.select(s, ln, int(ln.sum()))
    assert sorted(sel.tolist()) == list(range(50)) and ntok == ln.sum()
    sel0, ntok0 = oracle.select(s, ln, 0)
    assert len(sel0) == 0 and ntok0 == 0
    big = ln.copy(); big[int(np.argmax(s))] = 10 ** 6   # best unit never fits
    selb, _ = oracle.select(s, big, 100)
    assert len(selb) == 0


# ------------------------------------------------------------------ attention

def _softmax_attn(q, k, v):
    q, k, v = (x.astype(np.float64) for x in (q, k, v))
    lg = q @ k.T / math.sqrt(q.shape[1])
    w = np.exp(lg - lg.max(1, keepdims=True))
    return (w / w.sum(1, keepdims=True)) @ v


def test_attention_closed_forms():
    d = 128
    q = rng.standard_normal((4, d)).astype(np.float32)
    v1 = rng.standard_normal((1, d)).astype(np.float32)
    k1 = rng.standard_normal((1, d)).astype(np.float32)
    assert np.allclose(oracle.attention(q, k1, v1), np.repeat(v1, 4, 0), atol=1e-12)
    kk = np.repeat(k1, 9, 0)
    vv = rng.standard_normal((9, d)).astype(np.float32)
    assert np.allclose(oracle.attention(q, kk, vv), np.repeat(vv.astype(np.float64).mean(0, keepdims=True), 4, 0), atol=1e-12)
    k = rng.standard_normal((70, d)).astype(np.float32)
    v = rng.standard_normal((70, d)).astype(np.float32)
    assert np.allclose(oracle.attention(q, k, v), _softmax_attn(q, k, v), atol=1e-12)


# ------------------------------------------------------------------ decode

def _decode_inputs(dtype, hkv=2, g=4, d=128, n=300, c=10, T=60, jump=0.1, seed=0):
    r = np.random.default_rng(seed)
    comps = r.standard_normal((c, d))
    keys = (comps[r.integers(0, c, (hkv, n))] + 0.3 * r.standard_normal((hkv, n, d))).astype(np.float32)
    values = r.standard_normal((hkv, n, d)).astype(np.float32)
    q = np.empty((T, hkv * g, d), np.float32)
    cur = r.standard_normal((hkv * g, d))
    for t in range(T):
        if t and r.random() < jump:
            cur = r.standard_normal((hkv * g, d))
        elif t:
            cur = cur + 0.2 * r.standard_normal(cur.shape)
            cur = math.sqrt(d) * cur / np.linalg.norm(cur, axis=1, keepdims=True)
        q[t] = cur
    kn = r.standard_normal((T, hkv, d)).astype(np.float32)
    vn = r.standard_normal((T, hkv, d)).astype(np.float32)
    if dtype == "bf16":
        keys, values, q, kn, vn = (bf16(x) for x in (keys, values, q, kn, vn))
    assign = np.zeros((hkv, n), np.int32)
    cent = np.zeros((hkv, c, d), np.float32)
    for h in range(hkv):
        km = oracle.kmeans(np.ascontiguousarray(keys[h]), c, 4, seed=h)
        assign[h], cent[h] = km["assign"], km["cent"]
    return keys, values, assign, cent, q, kn, vn


def _f(x):
    return unbf16(x).astype(np.float64) if x.dtype == np.uint16 else x.astype(np.float64)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_fullcache_special_case(dtype):
    """tau > 1 makes every step retrieve; a budget >= every token selects every
    unit; the local buffer holds the rest: the output is full attention over
    all prefill and decode tokens so far (the FullCache configuration)."""
    hkv, g, n, c, T, L = 2, 4, 300, 10, 60, 8
    keys, values, assign, cent, q, kn, vn = _decode_inputs(dtype, hkv, g, n=n, c=c, T=T)
    res = oracle.decode(keys, values, assign, cent, q, kn, vn, n_clusters=c, local_buf=L,
                        tau=1.5, budget=n + T, want_seg_cent=True)
    assert res["flag"].all()
    K, Vv, Q, KN, VN = (_f(x) for x in (keys, values, q, kn, vn))
    for t in range(T):
        for kh in range(hkv):
            kk = np.concatenate([K[kh], KN[: t + 1, kh]])
            vv = np.concatenate([Vv[kh], VN[: t + 1, kh]])
            want = _softmax_attn(Q[t, kh * g:(kh + 1) * g], kk, vv)
            assert np.allclose(res["out"][t, kh * g:(kh + 1) * g], want, atol=1e-10)
    # every boundary closes a segment: all evicted segments have length 1 here
    assert res["n_evicted"] == T - L and (res["seg_len"] == 1).all()


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_decode_invariants(dtype):
    hkv, g, n, c, T, L, budget = 2, 4, 300, 10, 200, 16, 90
    keys, values, assign, cent, q, kn, vn = _decode_inputs(dtype, hkv, g, n=n, c=c, T=T,
                                                           jump=0.15, seed=4)
    tau = 0.9
    res = oracle.decode(keys, values, assign, cent, q, kn, vn, n_clusters=c, local_buf=L,
                        tau=tau, budget=budget, want_seg_cent=True)
    flag, ws, nu = res["flag"], res["win_start"], res["n_units"]
    assert flag[0] == 1
    assert np.array_equal(flag[1:], (res["r32"][1:] < tau).astype(np.uint8))
    assert 0 < flag[1:].sum() < T - 1
    # the local buffer never exceeds L and always holds the current token
    t = np.arange(T)
    assert np.all(t - ws + 1 <= L) and np.all(ws <= t)
    # evicted segments + buffer tile the decode tokens [0, t] in time order
    ss, sl = res["seg_start"], res["seg_len"]
    assert ss[0] == 0 and np.all(ss[1:] == ss[:-1] + sl[:-1])
    assert ss[-1] + sl[-1] == ws[-1]
    assert nu[-1] == c + res["n_evicted"]
    # segment boundaries are boundary steps, except forced cuts
    starts = set((ss + sl).tolist())
    cuts_not_flagged = [s for s in starts if s < T and flag[s] == 0]
    assert len(cuts_not_flagged) <= res["n_forced"]
    # a segment's index vector is the mean of its keys
    KN = _f(kn)
    for e in range(res["n_evicted"]):
        seg = KN[ss[e]: ss[e] + sl[e]]
        for kh in range(hkv):
            assert np.allclose(res["seg_cent"][e, kh], seg[:, kh].mean(0), atol=1e-6)
    # selections: within budget, reused verbatim between boundaries
    assert np.all(res["n_tok"] <= budget)
    for step in range(1, T):
        if not flag[step]:
            assert np.array_equal(res["n_sel"][step], res["n_sel"][step - 1])
            assert np.array_equal(res["sel"][step], res["sel"][step - 1])


def test_decode_never_triggering_forces_cuts():
    hkv, g, n, c, T, L = 1, 4, 200, 8, 100, 16
    keys, values, assign, cent, q, kn, vn = _decode_inputs("fp32", hkv, g, n=n, c=c, T=T)
    res = oracle.decode(keys, values, assign, cent, q, kn, vn, n_clusters=c, local_buf=L,
                        tau=-2.0, budget=64)
    assert res["flag"].sum() == 1
    assert res["n_forced"] == res["n_evicted"] == (T - 1) // L
    assert (res["seg_len"] == L).all()


def test_decode_selection_is_group_scored_budget_prefix():
    hkv, g, n, c, T, L, budget = 2, 4, 300, 10, 30, 8, 70
    keys, values, assign, cent, q, kn, vn = _decode_inputs("bf16", hkv, g, n=n, c=c, T=T)
    res = oracle.decode(keys, values, assign, cent, q, kn, vn, n_clusters=c, local_buf=L,
                        tau=0.95, budget=budget)
    step = 0  # only clusters exist at t = 0
    for kh in range(hkv):
        op = oracle.operand(cent[kh], oracle.BF16)
        s = oracle.group_scores(q[step, kh * g:(kh + 1) * g], op)
        ln = np.bincount(assign[kh], minlength=c).astype(np.int32)
        k = res["n_sel"][step, kh]
        _selection_properties(s, ln, budget, res["sel"][step, kh, :k], res["n_tok"][step, kh])


# ------------------------------------------------------------------ policy variants

def test_select_skip_is_lexicographic_max_feasible_subset():
    """Skip-and-continue fill: among all subsets whose length fits the budget,
    the one whose membership vector, read in (score desc, id asc) order, is
    lexicographically largest (take the best unit whenever it still fits).
    Brute force over every subset of <= 8 units."""
    for trial in range(300):
        u = int(rng.integers(1, 9))
        s = rng.integers(-3, 4, u).astype(np.float32)
        ln = rng.integers(0, 7, u).astype(np.int32)
        budget = int(rng.integers(0, 20))
        sel, ntok = oracle.select(s, ln, budget, oracle.FILL_SKIP)
        order = sorted(range(u), key=lambda x: (-float(s[x]), x))
        best = None
        for bits in itertools.product((1, 0), repeat=u):   # lexicographically descending
            if sum(int(ln[order[i]]) for i in range(u) if bits[i]) <= budget:
                best = [order[i] for i in range(u) if bits[i]]
                break
        assert list(sel) == best
        assert ntok == sum(int(ln[x]) for x in sel) <= budget
        pre, _ = oracle.select(s, ln, budget)
        assert list(sel[: len(pre)]) == list(pre)           # extends the stop-at-misfit prefix


def test_select_skip_special_cases():
    s = rng.standard_normal(40).astype(np.float32)
    ones = np.ones(40, np.int32)
    sel, ntok = oracle.select(s, ones, 13, oracle.FILL_SKIP)   # unit lengths: the 13 best
    assert list(sel) == list(np.argsort(-s, kind="stable")[:13]) and ntok == 13
    ln = rng.integers(1, 9, 40).astype(np.int32)
    sel, ntok = oracle.select(s, ln, int(ln.sum()), oracle.FILL_SKIP)
    assert sorted(sel.tolist()) == list(range(40)) and ntok == ln.sum()
    big = ln.copy(); big[int(np.argmax(s))] = 10 ** 6           # best never fits: the rest still do
    sel, ntok = oracle.select(s, big, int(ln.sum()), oracle.FILL_SKIP)
    assert int(np.argmax(s)) not in sel.tolist() and len(sel) == 39


def _dec(keys, values, assign, cent, q, kn, vn, c, L, **kw):
    return oracle.decode(keys, values, assign, cent, q, kn, vn, n_clusters=c, local_buf=L, **kw)


def test_decode_trigger_policies():
    hkv, g, n, c, T, L = 2, 4, 300, 10, 90, 12
    args = _decode_inputs("bf16", hkv, g, n=n, c=c, T=T, jump=0.1, seed=7)
    every = _dec(*args, c, L, tau=-5.0, budget=60, trigger=oracle.TRIGGER_EVERY)
    forced = _dec(*args, c, L, tau=1.5, budget=60)                 # r_t < 1.5 at every step
    assert every["flag"].all()
    for k in ("flag", "n_sel", "n_tok", "sel", "seg_start", "seg_len"):
        assert np.array_equal(every[k], forced[k]), k
    assert np.array_equal(every["out"], forced["out"])
    assert np.array_equal(every["r32"], forced["r32"])             # r_t still recorded
    for k_int in (1, 7, 16):
        fx = _dec(*args, c, L, tau=0.0, budget=60, trigger=oracle.TRIGGER_INTERVAL, interval=k_int)
        assert np.array_equal(np.nonzero(fx["flag"])[0], np.arange(0, T, k_int))
        # segments close exactly at the retrieval steps (or are cut by a full buffer)
        ends = (fx["seg_start"] + fx["seg_len"]).tolist()
        assert all(e % k_int == 0 for e in ends) or fx["n_forced"] > 0
    one = _dec(*args, c, L, tau=0.0, budget=60, trigger=oracle.TRIGGER_INTERVAL, interval=1)
    assert np.array_equal(one["sel"], every["sel"]) and np.array_equal(one["out"], every["out"])


def test_decode_page_segments():
    hkv, g, n, c, T, L, P = 2, 4, 300, 10, 120, 32, 8
    args = _decode_inputs("fp32", hkv, g, n=n, c=c, T=T, jump=0.2, seed=3)
    res = _dec(*args, c, L, tau=0.9, budget=60, page=P, want_seg_cent=True)
    assert res["n_forced"] == 0
    ne = res["n_evicted"]
    assert ne >= (T - L) // P
    assert np.array_equal(res["seg_start"], np.arange(ne) * P)     # fixed pages from token 0
    assert (res["seg_len"] == P).all()
    KN = _f(args[5])
    for e in range(ne):
        for kh in range(hkv):
            assert np.allclose(res["seg_cent"][e, kh], KN[e * P:(e + 1) * P, kh].mean(0), atol=1e-6)
    # pages do not depend on the retrieval steps
    other = _dec(*args, c, L, tau=-1.0, budget=60, page=P)
    assert np.array_equal(other["seg_start"], res["seg_start"])


def test_page_index_closed_forms():
    keys = rng.standard_normal((50, 128)).astype(np.float32)
    a, cent = oracle.page_index(keys, 1)
    assert np.array_equal(a, np.arange(50)) and np.array_equal(cent, keys)
    a, cent = oracle.page_index(keys, 50)
    want = np.array([math.fsum(keys[:, j].astype(np.float64)) / 50 for j in range(128)])
    assert np.array_equal(cent[0], want.astype(np.float32))
    a, cent = oracle.page_index(keys, 16)                          # 16, 16, 16, 2
    assert np.array_equal(np.bincount(a), [16, 16, 16, 2])
    assert np.allclose(cent[3], keys[48:].astype(np.float64).mean(0), atol=1e-7)


def test_decode_per_head_reduces_to_group_cases():
    """Per-query-head selection with g = 1 is the group selection; with the g
    heads of every group carrying the same query, the group sum scales every
    score by g (a power of two: exact) and each head selects what the group
    does."""
    hkv, n, c, T, L = 2, 300, 10, 40, 8
    a1 = _decode_inputs("bf16", hkv, 1, n=n, c=c, T=T, seed=5)
    r_grp = _dec(*a1, c, L, tau=0.95, budget=70)
    r_ph = _dec(*a1, c, L, tau=0.95, budget=70, per_head=True)
    for k in ("flag", "n_sel", "n_tok", "sel", "out"):
        assert np.array_equal(r_grp[k], r_ph[k]), k
    g = 4
    keys, values, assign, cent, q, kn, vn = _decode_inputs("bf16", hkv, g, n=n, c=c, T=T, seed=5)
    q = np.repeat(q[:, ::g], g, axis=1)                            # heads of a group share the query
    r_grp = _dec(keys, values, assign, cent, q, kn, vn, c, L, tau=0.95, budget=70)
    r_ph = _dec(keys, values, assign, cent, q, kn, vn, c, L, tau=0.95, budget=70, per_head=True)
    assert r_ph["n_sel"].shape == (T, hkv * g)
    for h in range(hkv * g):
        assert np.array_equal(r_ph["sel"][:, h], r_grp["sel"][:, h // g])
        assert np.array_equal(r_ph["n_tok"][:, h], r_grp["n_tok"][:, h // g])
    assert np.allclose(r_ph["out"], r_grp["out"], atol=1e-12)


def test_decode_per_head_selection_uses_own_query():
    hkv, g, n, c, T, L, budget = 2, 4, 300, 10, 20, 8, 70
    keys, values, assign, cent, q, kn, vn = _decode_inputs("bf16", hkv, g, n=n, c=c, T=T, seed=9)
    res = _dec(keys, values, assign, cent, q, kn, vn, c, L, tau=0.95, budget=budget, per_head=True)
    for h in range(hkv * g):
        kh = h // g
        op = oracle.operand(cent[kh], oracle.BF16)
        s = oracle.group_scores(q[0, h:h + 1], op)
        ln = np.bincount(assign[kh], minlength=c).astype(np.int32)
        k = res["n_sel"][0, h]
        _selection_properties(s, ln, budget, res["sel"][0, h, :k], res["n_tok"][0, h])
    # heads of one group disagree somewhere (otherwise the variant measures nothing)
    assert any(res["n_tok"][0, h] != res["n_tok"][0, h + 1] or
               not np.array_equal(res["sel"][0, h], res["sel"][0, h + 1]) for h in range(g - 1))


# ------------------------------------------------------------------ ParisKV-style selector

def test_paris_levels_are_beta_prior_quantiles_and_bin_means():
    """The rotation makes each coordinate x of a subspace direction in R^8
    behave like one of a uniform unit vector: x^2 ~ Beta(1/2, 7/2). The
    thresholds are its quantiles at l/8, the levels the bin means of |x|."""
    stats = pytest.importorskip("scipy.stats")
    integrate = pytest.importorskip("scipy.integrate")
    thr, lev = oracle.paris_levels(8)
    want = stats.beta.ppf(np.arange(1, 8) / 8, 0.5, 3.5)
    assert np.allclose(thr, want, rtol=2e-7, atol=0)
    t = np.concatenate([[0.0], np.sqrt(want), [1.0]])
    dens = lambda x: (1 - x * x) ** 2.5
    for l in range(8):
        num = integrate.quad(lambda x: x * dens(x), t[l], t[l + 1], epsabs=1e-14)[0]
        den = integrate.quad(dens, t[l], t[l + 1], epsabs=1e-14)[0]
        assert abs(lev[l] - num / den) <= 2e-7 * num / den
    assert np.all(np.diff(lev) > 0) and lev[0] > 0 and lev[-1] < 1


def test_paris_signs_follow_splitmix64_bits():
    s = oracle.paris_signs(77, 128)
    words = oracle.splitmix64(77, 2)
    for j in range(128):
        bit = (int(words[j // 64]) >> (j % 64)) & 1
        assert s[j] == (-1 if bit else 1)


def _paris_keys(n=64, seed=3):
    r = np.random.default_rng(seed)
    return bf16(r.standard_normal((n, 128)).astype(np.float32))


def test_paris_encode_against_hadamard_and_nearest_sign_centroid():
    linalg = pytest.importorskip("scipy.linalg")
    seed = 11
    keys = _paris_keys()
    bk, lv, w = oracle.paris_encode(keys, seed)
    Hm = linalg.hadamard(128).astype(np.float64)
    D = oracle.paris_signs(seed).astype(np.float64)
    thr, lev = oracle.paris_levels(8)
    for i in range(len(keys)):
        k = unbf16(keys[i]).astype(np.float64)
        y = Hm @ (D * k)                                  # exact: bf16 values, +-1 weights
        yb = y.reshape(16, 8)
        # the bucket is the nearest of the 256 analytic centroids s / sqrt(8)
        pats = np.array([[-1.0 if (p >> j) & 1 else 1.0 for j in range(8)] for p in range(256)])
        for b in range(16):
            u = yb[b] / np.linalg.norm(yb[b])
            assert int(np.argmax(pats @ u)) == bk[i, b]
            mag = (u * u)[:, None] >= thr[None, :].astype(np.float64)
            assert np.array_equal(lv[i, 8 * b:8 * b + 8], mag.sum(1))
            v = np.where(pats[bk[i, b]] < 0, -1.0, 1.0) * lev[lv[i, 8 * b:8 * b + 8]]
            ws = (yb[b] @ v) / (v @ v) / math.sqrt(128)
            assert abs(w[i, b] - ws) <= 1e-6 * abs(ws)


def test_paris_query_rotation_is_hadamard_of_signed_group_sum():
    linalg = pytest.importorskip("scipy.linalg")
    r = np.random.default_rng(5)
    q = bf16(r.standard_normal((4, 128)).astype(np.float32))
    got = oracle.paris_rotate_query(q, 9)
    qbar = unbf16(q).astype(np.float64).sum(0)
    want = linalg.hadamard(128) @ (oracle.paris_signs(9).astype(np.float64) * qbar)
    assert np.allclose(got, want, rtol=1e-5, atol=1e-4)


def test_paris_estimate_tracks_the_inner_product():
    """est_i ~ sqrt(d) <k_i, qbar> (the rotation scale): strong correlation
    and the right scale, from 3-bit magnitudes."""
    seed = 4
    keys = _paris_keys(400, seed=8)
    r = np.random.default_rng(6)
    q = bf16(r.standard_normal((4, 128)).astype(np.float32))
    bk, lv, w = oracle.paris_encode(keys, seed)
    qr = oracle.paris_rotate_query(q, seed)
    _, coarse, est = oracle.paris_select(qr, bk, lv, w, rho=4, n_cand=400, budget=10)
    true = unbf16(keys).astype(np.float64) @ unbf16(q).astype(np.float64).sum(0)
    assert np.corrcoef(est, true)[0, 1] > 0.97
    slope = (est @ true) / (true @ true)
    assert abs(slope / math.sqrt(128) - 1) < 0.05
    assert coarse.max() <= 16 * 4 and coarse.min() >= 0


def test_paris_select_definition_on_small_sets():
    """Brute force: candidates are the n_cand best (coarse desc, id asc), the
    selection the budget best of those by (estimate desc, id asc); a key with
    the query's own direction collects every subspace's top vote."""
    seed = 2
    for trial in range(20):
        r = np.random.default_rng(100 + trial)
        n = int(r.integers(5, 60))
        keys = _paris_keys(n, seed=200 + trial)
        q = bf16(r.standard_normal((2, 128)).astype(np.float32))
        bk, lv, w = oracle.paris_encode(keys, seed)
        qr = oracle.paris_rotate_query(q, seed)
        rho, n_cand, budget = int(r.integers(1, 9)), int(r.integers(1, n + 3)), int(r.integers(0, n + 3))
        sel, coarse, est = oracle.paris_select(qr, bk, lv, w, rho=rho, n_cand=n_cand, budget=budget)
        cand = sorted(range(n), key=lambda i: (-int(coarse[i]), i))[:n_cand]
        want = sorted(cand, key=lambda i: (-float(est[i]), i))[:budget]
        assert list(sel) == want
    # the query's own direction: its sign pattern is the top centroid everywhere
    k = bf16(np.random.default_rng(1).standard_normal((1, 128)).astype(np.float32))
    bk, lv, w = oracle.paris_encode(np.concatenate([k, _paris_keys(30)]), seed)
    qr = oracle.paris_rotate_query(k, seed)
    _, coarse, _ = oracle.paris_select(qr, bk, lv, w, rho=3, n_cand=31, budget=1)
    assert coarse[0] == 16 * 3


def test_decode_paris_fullcache_special_case():
    """Budget and candidate count above every token: the ParisKV-style
    selection takes every prefill and evicted token, so the output is full
    attention over all tokens so far."""
    hkv, g, n, T, L = 2, 4, 120, 40, 8
    keys, values, _, _, q, kn, vn = _decode_inputs("bf16", hkv, g, n=n, c=4, T=T)
    res = oracle.decode(keys, values, None, None, q, kn, vn, n_clusters=0, local_buf=L, tau=1.5,
                        budget=n + T, paris=dict(rho=4, n_cand=n + T, seed=3))
    K, Vv, Q, KN, VN = (_f(x) for x in (keys, values, q, kn, vn))
    for t in range(T):
        assert res["n_sel"][t, 0] == n + res["win_start"][t]
        for kh in range(hkv):
            kk = np.concatenate([K[kh], KN[: t + 1, kh]])
            vv = np.concatenate([Vv[kh], VN[: t + 1, kh]])
            want = _softmax_attn(Q[t, kh * g:(kh + 1) * g], kk, vv)
            assert np.allclose(res["out"][t, kh * g:(kh + 1) * g], want, atol=1e-10)


def test_decode_paris_selection_matches_select_over_region():
    hkv, g, n, T, L, budget = 1, 4, 200, 60, 8, 40
    keys, values, _, _, q, kn, vn = _decode_inputs("bf16", hkv, g, n=n, c=4, T=T, jump=0.2, seed=12)
    pr = dict(rho=4, n_cand=80, seed=5)
    res = oracle.decode(keys, values, None, None, q, kn, vn, n_clusters=0, local_buf=L, tau=0.9,
                        budget=budget, paris=pr)
    allk = np.concatenate([keys[0], kn[:, 0]])
    bk, lv, w = oracle.paris_encode(allk, pr["seed"])
    for t in np.flatnonzero(res["flag"]):
        reg = n + res["win_start"][t]
        qr = oracle.paris_rotate_query(q[t, 0:g], pr["seed"])
        sel, _, _ = oracle.paris_select(qr, bk[:reg], lv[:reg], w[:reg], rho=4, n_cand=80, budget=budget)
        k = res["n_sel"][t, 0]
        assert k == len(sel) == min(budget, 80, reg)
        assert np.array_equal(res["sel"][t, 0, :k], sel)
