"""cluster_indexed_kv_gb300 -- LouisKV-style KV-cache retrieval on one GB300.

The compute path is liblkv.so (hand-written CUDA for sm_103a behind the C ABI
in include/lkv.h). This package only marshals torch tensors into that ABI:
``Context`` owns one liblkv context; every method is one C call.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import torch

from . import _lib
from ._lib import LKVError, lkv_config  # noqa: F401

__all__ = ["Context", "LKVError", "build"]


def build(force: bool = False) -> str:
    from .builder import build as _build
    return _build(force=force)


def _dev_ptr(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _event_ptr(ev):
    """cudaEvent_t of a torch.cuda.Event (created now if it never was), or None."""
    if ev is None:
        return None
    if not ev.cuda_event:
        ev.record()  # torch creates the CUDA event at its first record
    return ev.cuda_event


def _opt_ptr(t, name, dtype=None):
    return None if t is None else _dev_ptr(t, name, dtype)


class Context:
    """One liblkv context (pool, index, decode state of every layer)."""

    def __init__(self, *, batch: int, n_layers: int, n_kv_heads: int, group: int,
                 dtype: torch.dtype, local_buf: int, max_clusters: int, max_prefill: int,
                 max_steps: int, max_budget: int, offload: bool = False, head_dim: int = 128,
                 stream: torch.cuda.Stream | None = None):
        if dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("dtype must be torch.float32 or torch.bfloat16")
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        self.cfg = lkv_config(batch, n_layers, n_kv_heads, group, head_dim,
                              _lib.LKV_DTYPE_BF16 if dtype == torch.bfloat16 else _lib.LKV_DTYPE_FP32,
                              local_buf, max_clusters, max_prefill, max_steps, max_budget,
                              1 if offload else 0, self.stream.cuda_stream)
        self.dtype = dtype
        self.batch, self.n_layers, self.n_kv_heads, self.group = batch, n_layers, n_kv_heads, group
        self.n_heads = n_kv_heads * group
        self.local_buf, self.max_clusters, self.max_steps = local_buf, max_clusters, max_steps
        self.u_cap = max_clusters + max_steps
        self._ctx = _lib.lkv_create(self.cfg)

    # -- lifetime
    def close(self):
        if getattr(self, "_ctx", None):
            _lib.lkv_destroy(self._ctx)
            self._ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    # -- calls
    def build_index(self, layer: int, keys: torch.Tensor, values: torch.Tensor,
                    n_clusters: int, iters: int, seed: int) -> None:
        n = keys.shape[-2]
        _lib.lkv_build_index(self._ctx, layer, _dev_ptr(keys, "keys", self.dtype),
                             _dev_ptr(values, "values", self.dtype), n, n_clusters, iters, seed)

    def load_index(self, layer: int, keys: torch.Tensor, values: torch.Tensor, n_clusters: int,
                   assign: torch.Tensor, centroids: torch.Tensor) -> None:
        n = keys.shape[-2]
        _lib.lkv_load_index(self._ctx, layer, _dev_ptr(keys, "keys", self.dtype),
                            _dev_ptr(values, "values", self.dtype), n, n_clusters,
                            _dev_ptr(assign, "assign", torch.int32),
                            _dev_ptr(centroids, "centroids", torch.float32))

    def build_index_async(self, layer: int, keys: torch.Tensor, values: torch.Tensor,
                          n_clusters: int, iters: int, seed: int,
                          ready: "torch.cuda.Event | None" = None,
                          done: "torch.cuda.Event | None" = None) -> None:
        """build_index on the context's stream after `ready` (an event the
        producer recorded when this layer's keys and values were complete);
        `done` is recorded once the build has finished reading them."""
        n = keys.shape[-2]
        _lib.lkv_build_index_async(self._ctx, layer, _dev_ptr(keys, "keys", self.dtype),
                                   _dev_ptr(values, "values", self.dtype), n, n_clusters, iters,
                                   seed, _event_ptr(ready), _event_ptr(done))

    def build_paris(self, layer: int, keys: torch.Tensor, values: torch.Tensor, *, rho: int = 4,
                    n_cand: int = 2048, seed: int = 1) -> None:
        """ParisKV-style token selector for this layer (see lkv_build_paris):
        the pool in token order plus per-token codes; no clusters."""
        n = keys.shape[-2]
        _lib.lkv_build_paris(self._ctx, layer, _dev_ptr(keys, "keys", self.dtype),
                             _dev_ptr(values, "values", self.dtype), n, rho, n_cand, seed)

    def build_pages(self, layer: int, keys: torch.Tensor, values: torch.Tensor, page: int) -> None:
        """Page-mean units (ceil(N / page) pages of consecutive tokens) instead
        of a K-means index."""
        n = keys.shape[-2]
        _lib.lkv_build_pages(self._ctx, layer, _dev_ptr(keys, "keys", self.dtype),
                             _dev_ptr(values, "values", self.dtype), n, page)

    def set_policy(self, trigger: str = "adaptive", interval: int = 1, fill: str = "prefix",
                   page: int = 0, per_head: bool = False) -> None:
        """Retrieval policy: trigger "adaptive" (r_t < tau), "every" or
        "interval"; fill "prefix" (stop at the first unit that does not fit)
        or "skip"; page 0 (segments close at retrievals) or P (P-token pages);
        per_head: a selection per query head (selection records become
        [.., H, u_cap] and [.., H])."""
        trig = {"adaptive": _lib.LKV_TRIGGER_ADAPTIVE, "every": _lib.LKV_TRIGGER_EVERY,
                "interval": _lib.LKV_TRIGGER_INTERVAL}[trigger]
        fl = {"prefix": _lib.LKV_FILL_PREFIX, "skip": _lib.LKV_FILL_SKIP}[fill]
        _lib.lkv_set_policy(self._ctx, trig, interval, fl, page, 1 if per_head else 0)
        self.per_head = bool(per_head)

    def decode_step(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    tau: float, budget: int, out: torch.Tensor, *, n_layers: int = 1,
                    selected_units: torch.Tensor | None = None,
                    n_selected: torch.Tensor | None = None,
                    boundary: torch.Tensor | None = None,
                    r_out: torch.Tensor | None = None) -> None:
        _lib.lkv_decode_step(self._ctx, layer, n_layers, _dev_ptr(q, "q", self.dtype),
                             _dev_ptr(k_new, "k_new", self.dtype),
                             _dev_ptr(v_new, "v_new", self.dtype), float(tau), budget,
                             self.local_buf, _dev_ptr(out, "out", torch.float32),
                             _opt_ptr(selected_units, "selected_units", torch.int32),
                             _opt_ptr(n_selected, "n_selected", torch.int32),
                             _opt_ptr(boundary, "boundary", torch.uint8),
                             _opt_ptr(r_out, "r_out", torch.float32))

    def decode_steps(self, layer: int, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                     tau: float, budget: int, out: torch.Tensor, *, n_layers: int = 1,
                     selected_units: torch.Tensor | None = None,
                     n_selected: torch.Tensor | None = None,
                     boundary: torch.Tensor | None = None,
                     r_out: torch.Tensor | None = None) -> None:
        """q.shape[0] consecutive decode steps (see lkv_decode_steps)."""
        _lib.lkv_decode_steps(self._ctx, layer, n_layers, q.shape[0], _dev_ptr(q, "q", self.dtype),
                              _dev_ptr(k_new, "k_new", self.dtype),
                              _dev_ptr(v_new, "v_new", self.dtype), float(tau), budget,
                              self.local_buf, _dev_ptr(out, "out", torch.float32),
                              _opt_ptr(selected_units, "selected_units", torch.int32),
                              _opt_ptr(n_selected, "n_selected", torch.int32),
                              _opt_ptr(boundary, "boundary", torch.uint8),
                              _opt_ptr(r_out, "r_out", torch.float32))

    def set_profiling(self, enable: bool) -> None:
        _lib.lkv_set_profiling(self._ctx, enable)

    def set_kmeans_filter(self, tensor_cores: bool) -> None:
        """Tensor-core (default) or SIMT distance filter for the K-means
        assignment; the result is the same either way."""
        _lib.lkv_set_kmeans_filter(self._ctx, _lib.LKV_FILTER_TENSOR if tensor_cores
                                   else _lib.LKV_FILTER_SIMT)

    def profile(self, reset: bool = False):
        return _lib.lkv_get_profile(self._ctx, reset)

    def get_index(self, layer: int, seq: int, kv_head: int, n_tokens: int) -> dict:
        cap = self.u_cap
        cent = np.zeros((cap, 128), np.float32)
        ln = np.zeros(cap, np.int32)
        row = np.zeros(cap, np.int32)
        assign = np.zeros(n_tokens, np.int32)
        perm = np.zeros(n_tokens, np.int32)
        u = _lib.lkv_get_index(self._ctx, layer, seq, kv_head, cap, cent.ctypes.data,
                               ln.ctypes.data, row.ctypes.data, assign.ctypes.data,
                               perm.ctypes.data)
        return dict(centroids=cent[:u], unit_len=ln[:u], unit_row=row[:u], assign=assign,
                    perm=perm, n_units=u)

    def decode_state(self, layer: int, seq: int) -> dict:
        s = _lib.lkv_get_decode_state(self._ctx, layer, seq)
        return {name: getattr(s, name) for name, _ in s._fields_}

    def sync(self) -> None:
        _lib.lkv_sync(self._ctx)

    def diag_wait_timeout(self, limit_ns: int) -> None:
        """Failure-path check: a device wait that nothing completes runs out
        after limit_ns; the next sync() raises LKV_ETIMEOUT."""
        _lib.lkv_diag_wait_timeout(self._ctx, limit_ns)
