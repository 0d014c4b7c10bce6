"""Oracle work units for a spawn process pool (test infrastructure only).

The GPU parity tests at configuration size hand the oracle many independent
pieces of work: the last Lloyd round of a full-size head split into key
ranges, or whole decode runs of single sequences at several sweep points.
Each function here runs one piece in a fresh interpreter started with the
``spawn`` method (never ``fork`` after the parent touched the GPU). Inputs
come as paths of ``.npy`` files that the workers map read-only; results are
compact: only what the test compares."""
from __future__ import annotations

import numpy as np


def _load(path):
    return np.load(path, mmap_mode="r")


def assign_range(keys_path: str, cent_op_path: str, lo: int, hi: int) -> np.ndarray:
    """oracle.assign of keys[lo:hi] against the operand centroids."""
    import oracle
    keys = np.ascontiguousarray(_load(keys_path)[lo:hi])
    return oracle.assign(keys, np.ascontiguousarray(_load(cent_op_path)))


def decode_run(inputs: dict, kw: dict, attn_steps) -> dict:
    """oracle.decode of one (sequence, layer) from .npy paths; returns the
    flags, r_t, selection sizes, the selections at retrieval steps, the
    attention outputs at attn_steps and the evicted segments."""
    import oracle
    arr = {k: np.ascontiguousarray(_load(p)) for k, p in inputs.items()}
    T = arr["q"].shape[0]
    mask = np.zeros(T, np.uint8)
    mask[np.asarray(attn_steps, dtype=np.int64)] = 1
    o = oracle.decode(arr["keys"], arr["values"], arr["assign"], arr["cent"], arr["q"],
                      arr["k_new"], arr["v_new"], attn_mask=mask, want_seg_cent=True,
                      **kw)
    flagged = np.flatnonzero(o["flag"])
    sel = {}
    if o["sel"] is not None:
        for t in flagged:
            for h in range(o["n_sel"].shape[1]):
                k = o["n_sel"][t, h]
                sel[(int(t), h)] = np.sort(o["sel"][t, h, :k])
    return dict(flag=o["flag"], r32=o["r32"], n_sel=o["n_sel"], n_tok=o["n_tok"], sel=sel,
                out=o["out"][mask.astype(bool)], attn_steps=np.flatnonzero(mask),
                n_evicted=o["n_evicted"], n_forced=o["n_forced"], seg_start=o["seg_start"],
                seg_len=o["seg_len"], seg_cent=o["seg_cent"])
