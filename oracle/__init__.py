"""Python access to the plain CPU oracle (``lkv_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use this module; the product package never
imports it. The oracle is single-threaded C built with
``-O2 -ffp-contract=off`` (no FMA contraction; the fused multiply-adds the
decision values need are explicit ``fmaf`` calls).

Arrays cross as numpy buffers: bf16 tensors as ``uint16`` bit patterns, fp32 as
``float32``. See ``lkv_oracle.h`` for each function's definition and the page
passages it follows.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

FP32, BF16 = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lkv_oracle.c")
_HDR = os.path.join(_HERE, "lkv_oracle.h")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblkv_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (if missing or older than its sources)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or force or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB_PATH) for p in (_SRC, _HDR))
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class DecodeArgs(C.Structure):
    _fields_ = [
        ("dtype", C.c_int32), ("n_kv_heads", C.c_int32), ("group", C.c_int32),
        ("head_dim", C.c_int32), ("n_prefill", C.c_int64),
        ("n_clusters", C.c_int32), ("local_buf", C.c_int32),
        ("n_steps", C.c_int32), ("tau", C.c_float), ("budget", C.c_int32),
        ("keys", C.c_void_p), ("values", C.c_void_p), ("assign", C.c_void_p),
        ("cent", C.c_void_p), ("q", C.c_void_p), ("k_new", C.c_void_p),
        ("v_new", C.c_void_p), ("attn_mask", C.c_void_p),
        ("trigger", C.c_int32), ("interval", C.c_int32), ("fill", C.c_int32),
        ("page", C.c_int32), ("per_head", C.c_int32),
        ("selector", C.c_int32), ("paris_rho", C.c_int32), ("paris_n_cand", C.c_int32),
        ("paris_seed", C.c_uint64),
    ]


SELECT_CLUSTERS, SELECT_PARIS = 0, 1


TRIGGER_ADAPTIVE, TRIGGER_EVERY, TRIGGER_INTERVAL = 0, 1, 2
FILL_PREFIX, FILL_SKIP = 0, 1


class DecodeResult(C.Structure):
    _fields_ = [
        ("max_sel", C.c_int32), ("max_segs", C.c_int32), ("out", C.c_void_p),
        ("flag", C.c_void_p), ("r32", C.c_void_p), ("r64", C.c_void_p),
        ("n_sel", C.c_void_p), ("n_tok", C.c_void_p), ("sel", C.c_void_p),
        ("win_start", C.c_void_p), ("n_units", C.c_void_p),
        ("seg_start", C.c_void_p), ("seg_len", C.c_void_p),
        ("seg_cent", C.c_void_p), ("n_evicted", C.c_int32),
        ("n_forced", C.c_int32),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            vp, i32, i64, u64 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64
            L.lkvo_init_indices.argtypes = [i64, i32, u64, vp]
            L.lkvo_init_indices.restype = C.c_int
            L.lkvo_splitmix64.argtypes = [u64, i32, vp]
            L.lkvo_sqdist.argtypes = [vp, C.c_int, vp, i32]
            L.lkvo_sqdist.restype = C.c_double
            L.lkvo_assign.argtypes = [vp, C.c_int, i64, i32, vp, i32, vp, vp]
            L.lkvo_update.argtypes = [vp, C.c_int, i64, i32, vp, i32, vp, vp, vp]
            L.lkvo_operand.argtypes = [vp, i64, C.c_int, vp]
            L.lkvo_objective.argtypes = [vp, C.c_int, i64, i32, vp, vp]
            L.lkvo_objective.restype = C.c_double
            L.lkvo_kmeans.argtypes = [vp, C.c_int, i64, i32, i32, i32, u64, vp, vp,
                                      vp, vp, vp, vp]
            L.lkvo_kmeans.restype = C.c_int
            L.lkvo_boundary_r32.argtypes = [vp, vp, C.c_int, i32, i32]
            L.lkvo_boundary_r32.restype = C.c_float
            L.lkvo_boundary_r64.argtypes = [vp, vp, C.c_int, i32, i32]
            L.lkvo_boundary_r64.restype = C.c_double
            L.lkvo_group_scores.argtypes = [vp, C.c_int, i32, i32, vp, i32, vp]
            L.lkvo_select.argtypes = [vp, vp, i32, i32, vp, vp]
            L.lkvo_select.restype = i32
            L.lkvo_select_skip.argtypes = [vp, vp, i32, i32, vp, vp]
            L.lkvo_select_skip.restype = i32
            L.lkvo_paris_signs.argtypes = [u64, i32, vp]
            L.lkvo_paris_levels.argtypes = [i32, vp, vp]
            L.lkvo_paris_levels.restype = C.c_int
            L.lkvo_paris_encode.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp]
            L.lkvo_paris_rotate_query.argtypes = [vp, C.c_int, i32, i32, vp, vp]
            L.lkvo_paris_select.argtypes = [vp, i32, i32, i32, i64, i32, i64, vp, vp, vp, vp,
                                            vp, vp, vp]
            L.lkvo_paris_select.restype = i64
            L.lkvo_attention.argtypes = [vp, C.c_int, i32, i32, vp, vp, i64, vp]
            L.lkvo_decode.argtypes = [C.POINTER(DecodeArgs), C.POINTER(DecodeResult)]
            L.lkvo_decode.restype = C.c_int
            L.lkvo_f32_to_bf16.argtypes = [C.c_float]
            L.lkvo_f32_to_bf16.restype = C.c_uint16
            _lib = L
    return _lib


# ---------------------------------------------------------------- helpers

def _arr(x, dtype):
    return np.ascontiguousarray(x, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


def dtype_of(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return FP32
    raise TypeError(f"oracle takes uint16 (bf16 bits) or float32, got {a.dtype}")


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit patterns (same rule as the C)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def splitmix64(seed: int, count: int) -> np.ndarray:
    out = np.zeros(count, np.uint64)
    lib().lkvo_splitmix64(seed, count, _p(out))
    return out


def init_indices(n: int, c: int, seed: int) -> np.ndarray:
    idx = np.zeros(c, np.int64)
    if lib().lkvo_init_indices(n, c, seed, _p(idx)) != 0:
        raise ValueError("bad init arguments")
    return idx


def operand(cent: np.ndarray, dtype: int) -> np.ndarray:
    cent = _arr(cent, np.float32)
    out = np.empty_like(cent)
    lib().lkvo_operand(_p(cent), cent.size, dtype, _p(out))
    return out


def sqdist(key: np.ndarray, cent_row: np.ndarray) -> float:
    key = np.ascontiguousarray(key)
    c = _arr(cent_row, np.float32)
    return lib().lkvo_sqdist(_p(key), dtype_of(key), _p(c), key.shape[-1])


def assign(keys: np.ndarray, cent_op: np.ndarray, with_gap: bool = False):
    keys = np.ascontiguousarray(keys)
    cent_op = _arr(cent_op, np.float32)
    n, d = keys.shape
    a = np.zeros(n, np.int32)
    gap = np.zeros(n, np.float64) if with_gap else None
    lib().lkvo_assign(_p(keys), dtype_of(keys), n, d, _p(cent_op), cent_op.shape[0],
                      _p(a), _p(gap))
    return (a, gap) if with_gap else a


def update(keys: np.ndarray, assign_: np.ndarray, cent: np.ndarray):
    keys = np.ascontiguousarray(keys)
    n, d = keys.shape
    cent = _arr(cent, np.float32).copy()
    a = _arr(assign_, np.int32)
    cnt = np.zeros(cent.shape[0], np.int32)
    inexact = C.c_int64(0)
    lib().lkvo_update(_p(keys), dtype_of(keys), n, d, _p(a), cent.shape[0], _p(cent),
                      _p(cnt), C.addressof(inexact))
    return cent, cnt, inexact.value


def objective(keys: np.ndarray, cent_op: np.ndarray, assign_: np.ndarray) -> float:
    keys = np.ascontiguousarray(keys)
    n, d = keys.shape
    return lib().lkvo_objective(_p(keys), dtype_of(keys), n, d,
                                _p(_arr(cent_op, np.float32)), _p(_arr(assign_, np.int32)))


def kmeans(keys: np.ndarray, c: int, iters: int, seed: int, trace: bool = False):
    """Returns dict(cent [c,d] fp32, assign [n], count [c], inexact, and with
    trace: trace_cent [iters+1,c,d], trace_assign [iters,n])."""
    keys = np.ascontiguousarray(keys)
    n, d = keys.shape
    cent = np.zeros((c, d), np.float32)
    a = np.zeros(n, np.int32)
    cnt = np.zeros(c, np.int32)
    tc = np.zeros((iters + 1, c, d), np.float32) if trace else None
    ta = np.zeros((iters, n), np.int32) if trace else None
    inexact = C.c_int64(0)
    rc = lib().lkvo_kmeans(_p(keys), dtype_of(keys), n, d, c, iters, seed, _p(cent),
                           _p(a), _p(cnt), _p(tc), _p(ta), C.addressof(inexact))
    if rc != 0:
        raise ValueError("bad k-means arguments")
    out = dict(cent=cent, assign=a, count=cnt, inexact=inexact.value)
    if trace:
        out.update(trace_cent=tc, trace_assign=ta)
    return out


def boundary_r(q_prev: np.ndarray, q_cur: np.ndarray):
    """(r32 decision value, r64) for q of shape [H, d]."""
    qp, qc = np.ascontiguousarray(q_prev), np.ascontiguousarray(q_cur)
    h, d = qc.shape
    dt = dtype_of(qc)
    L = lib()
    return (L.lkvo_boundary_r32(_p(qp), _p(qc), dt, h, d),
            L.lkvo_boundary_r64(_p(qp), _p(qc), dt, h, d))


def group_scores(q_group: np.ndarray, cent_op: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q_group)
    g, d = q.shape
    cent_op = _arr(cent_op, np.float32)
    s = np.zeros(cent_op.shape[0], np.float32)
    lib().lkvo_group_scores(_p(q), dtype_of(q), g, d, _p(cent_op), cent_op.shape[0], _p(s))
    return s


def select(scores: np.ndarray, lens: np.ndarray, budget: int, fill: int = FILL_PREFIX):
    """(ids in selection order, tokens): lkvo_select, or lkvo_select_skip with
    fill=FILL_SKIP."""
    s = _arr(scores, np.float32)
    ln = _arr(lens, np.int32)
    sel = np.zeros(max(1, s.size), np.int32)
    ntok = C.c_int32(0)
    f = lib().lkvo_select_skip if fill == FILL_SKIP else lib().lkvo_select
    k = f(_p(s), _p(ln), s.size, budget, _p(sel), C.addressof(ntok))
    return sel[:k].copy(), ntok.value


def page_index(keys: np.ndarray, page: int):
    """Page-mean units of one slice [CTkvr, 1.1 (block-level indexes mean-pool
    runs of consecutive tokens)]: unit j holds tokens [j*page, (j+1)*page)
    (the last page may be short); its index vector is the mean of its keys,
    by the same update as a Lloyd round. Returns (assign [n], cent [c, d])."""
    keys = np.ascontiguousarray(keys)
    n, d = keys.shape
    c = -(-n // page)
    a = (np.arange(n) // page).astype(np.int32)
    cent, cnt, _ = update(keys, a, np.zeros((c, d), np.float32))
    assert (cnt > 0).all()
    return a, cent


def paris_signs(seed: int, d: int = 128) -> np.ndarray:
    out = np.zeros(d, np.int8)
    lib().lkvo_paris_signs(seed, d, _p(out))
    return out


def paris_levels(m: int = 8):
    """(thresholds T_l = t_l^2, l = 1..7, and bin means, 8) as float32."""
    thr = np.zeros(7, np.float32)
    lev = np.zeros(8, np.float32)
    if lib().lkvo_paris_levels(m, _p(thr), _p(lev)) != 0:
        raise ValueError("m must be >= 2")
    return thr, lev


def paris_encode(keys: np.ndarray, seed: int, m: int = 8):
    """Metadata of bf16 keys [n, d]: (buckets [n, d/m] u8, levels [n, d] u8,
    scales [n, d/m] f32)."""
    keys = _arr(keys, np.uint16)
    n, d = keys.shape
    sign = paris_signs(seed, d)
    thr, lev = paris_levels(m)
    bk = np.zeros((n, d // m), np.uint8)
    lv = np.zeros((n, d), np.uint8)
    w = np.zeros((n, d // m), np.float32)
    L = lib()
    for i in range(n):
        L.lkvo_paris_encode(_p(keys[i]), d, _p(sign), m, _p(thr), _p(lev), _p(bk[i]), _p(lv[i]),
                            _p(w[i]))
    return bk, lv, w


def paris_rotate_query(q_group: np.ndarray, seed: int) -> np.ndarray:
    q = np.ascontiguousarray(q_group)
    g, d = q.shape
    out = np.zeros(d, np.float32)
    lib().lkvo_paris_rotate_query(_p(q), dtype_of(q), g, d, _p(paris_signs(seed, d)), _p(out))
    return out


def paris_select(qrot, bucket, level, w, *, rho, n_cand, budget, m=8):
    """(selected ids best first, coarse scores [n], estimates [n])."""
    qrot = _arr(qrot, np.float32)
    bucket, level, w = _arr(bucket, np.uint8), _arr(level, np.uint8), _arr(w, np.float32)
    n, d = level.shape
    _, lev = paris_levels(m)
    sel = np.zeros(max(1, min(budget, n)), np.int64)
    coarse = np.zeros(max(1, n), np.int32)
    est = np.zeros(max(1, n), np.float32)
    k = lib().lkvo_paris_select(_p(qrot), d, m, rho, n_cand, budget, n, _p(bucket), _p(level),
                                _p(w), _p(lev), _p(sel), _p(coarse), _p(est))
    return sel[:k].copy(), coarse[:n], est[:n]


def attention(q_group: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q_group)
    k, v = np.ascontiguousarray(k_rows), np.ascontiguousarray(v_rows)
    g, d = q.shape
    out = np.zeros((g, d), np.float64)
    lib().lkvo_attention(_p(q), dtype_of(q), g, d, _p(k), _p(v), k.shape[0], _p(out))
    return out


def decode(keys, values, assign_, cent, q, k_new, v_new, *, n_clusters, local_buf,
           tau, budget, attn_mask=None, want_seg_cent=False, want_sel=True, max_sel=None,
           trigger=TRIGGER_ADAPTIVE, interval=1, fill=FILL_PREFIX, page=0, per_head=False,
           paris=None):
    """Run one (sequence, layer) decode through the oracle.

    keys/values [H_kv, N, d]; assign_ [H_kv, N]; cent [H_kv, C, d] fp32;
    q [T, H, d]; k_new/v_new [T, H_kv, d]. Returns a dict of numpy arrays.
    want_sel=False skips the per-step selection lists (n_sel and n_tok are
    still recorded); with lists, each holds at most budget + C ids (a unit
    that fits adds at least one token, except empty clusters). max_sel caps
    the recorded list length for long runs (the call fails if a selection is
    longer). trigger/interval/fill/page/per_head pick the retrieval policy
    (see lkvo_decode_args); with per_head the selection records are per
    query head ([T, H]) instead of per KV head. paris=dict(rho, n_cand, seed)
    selects tokens with the ParisKV-style pipeline instead (n_clusters 0;
    assign_ and cent unused; the records hold token ids, prefill i and decode
    t as N + t, best first).
    """
    keys, values = np.ascontiguousarray(keys), np.ascontiguousarray(values)
    q, k_new, v_new = (np.ascontiguousarray(x) for x in (q, k_new, v_new))
    hkv, n, d = keys.shape
    if paris is not None:
        assign_ = np.zeros((hkv, max(1, n)), np.int32)
        cent = np.zeros((hkv, 1, d), np.float32)
        n_clusters = 0
    assign_ = _arr(assign_, np.int32)
    cent = _arr(cent, np.float32)
    T, h_all, _ = q.shape
    g = h_all // hkv
    dt = dtype_of(q)
    c = n_clusters
    ucap = c + T
    max_sel = min(ucap, budget + c) if max_sel is None else min(ucap, budget + c, max_sel)
    if paris is not None:
        max_sel = max(1, budget)
    mask = None if attn_mask is None else _arr(attn_mask, np.uint8)
    pr = paris or {}
    args = DecodeArgs(dt, hkv, g, d, n, c, local_buf, T, tau, budget, _p(keys), _p(values),
                      _p(assign_), _p(cent), _p(q), _p(k_new), _p(v_new), _p(mask),
                      trigger, interval, fill, page, 1 if per_head else 0,
                      SELECT_PARIS if paris is not None else SELECT_CLUSTERS,
                      pr.get("rho", 0), pr.get("n_cand", 0), pr.get("seed", 0))
    hs = h_all if per_head else hkv
    res = dict(
        out=np.zeros((T, h_all, d), np.float64), flag=np.zeros(T, np.uint8),
        r32=np.zeros(T, np.float32), r64=np.zeros(T, np.float64),
        n_sel=np.zeros((T, hs), np.int32), n_tok=np.zeros((T, hs), np.int32),
        sel=np.full((T, hs, max_sel), -1, np.int32) if want_sel else None,
        win_start=np.zeros(T, np.int32),
        n_units=np.zeros(T, np.int32), seg_start=np.zeros(max(T, 1), np.int32),
        seg_len=np.zeros(max(T, 1), np.int32),
        seg_cent=np.zeros((max(T, 1), hkv, d), np.float32) if want_seg_cent else None)
    r = DecodeResult(max_sel, max(T, 1), *(_p(res[k]) for k in (
        "out", "flag", "r32", "r64", "n_sel", "n_tok", "sel", "win_start", "n_units",
        "seg_start", "seg_len", "seg_cent")), 0, 0)
    if lib().lkvo_decode(C.byref(args), C.byref(r)) != 0:
        raise ValueError("oracle decode rejected its arguments")
    ne = r.n_evicted
    res["n_evicted"], res["n_forced"] = ne, r.n_forced
    res["seg_start"], res["seg_len"] = res["seg_start"][:ne], res["seg_len"][:ne]
    if want_seg_cent:
        res["seg_cent"] = res["seg_cent"][:ne]
    return res
