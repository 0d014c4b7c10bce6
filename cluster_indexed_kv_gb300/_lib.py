"""ctypes binding of liblkv (include/lkv.h): argument marshalling only.

Every function here has the name of the C entry point it calls. There is no
fallback: if liblkv.so has not been built, loading raises immediately.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "liblkv.so")

LKV_OK, LKV_EINVAL, LKV_ENOMEM, LKV_ECUDA, LKV_ECAPACITY, LKV_ESTATE, LKV_ETIMEOUT = range(7)
STATUS_NAMES = {0: "LKV_OK", 1: "LKV_EINVAL", 2: "LKV_ENOMEM", 3: "LKV_ECUDA",
                4: "LKV_ECAPACITY", 5: "LKV_ESTATE", 6: "LKV_ETIMEOUT"}
LKV_DTYPE_FP32, LKV_DTYPE_BF16 = 0, 1

EXPORTED = ("lkv_create", "lkv_destroy", "lkv_build_index", "lkv_load_index",
            "lkv_decode_step", "lkv_decode_steps", "lkv_get_index", "lkv_get_decode_state",
            "lkv_sync", "lkv_last_error", "lkv_set_profiling", "lkv_get_profile",
            "lkv_kmeans_static", "lkv_kmeans_static_status", "lkv_set_kmeans_filter",
            "lkv_diag_wait_timeout", "lkv_uva_read", "lkv_read_ceiling", "lkv_set_policy", "lkv_build_pages",
            "lkv_build_index_async", "lkv_build_paris", "lkv_paris_levels")
LKV_FILTER_TENSOR, LKV_FILTER_SIMT = 0, 1
LKV_TRIGGER_ADAPTIVE, LKV_TRIGGER_EVERY, LKV_TRIGGER_INTERVAL = 0, 1, 2
LKV_FILL_PREFIX, LKV_FILL_SKIP = 0, 1


class lkv_config(C.Structure):
    _fields_ = [
        ("batch", C.c_int32), ("n_layers", C.c_int32), ("n_kv_heads", C.c_int32),
        ("group", C.c_int32), ("head_dim", C.c_int32), ("dtype", C.c_int32),
        ("local_buf", C.c_int32), ("max_clusters", C.c_int32), ("max_prefill", C.c_int64),
        ("max_steps", C.c_int32), ("max_budget", C.c_int32), ("offload", C.c_int32),
        ("stream", C.c_void_p),
    ]


class lkv_policy(C.Structure):
    _fields_ = [("trigger", C.c_int32), ("interval", C.c_int32), ("fill", C.c_int32),
                ("page", C.c_int32), ("per_head", C.c_int32)]


class lkv_paris_params(C.Structure):
    _fields_ = [("rho", C.c_int32), ("n_cand", C.c_int32), ("seed", C.c_uint64)]


class lkv_decode_state(C.Structure):
    _fields_ = [
        ("t", C.c_int32), ("win_start", C.c_int32), ("open_start", C.c_int32),
        ("n_clusters", C.c_int32), ("n_units", C.c_int32), ("n_closed", C.c_int32),
        ("n_evicted", C.c_int32), ("n_forced", C.c_int32), ("n_refined", C.c_int64),
        ("n_inexact", C.c_int64),
    ]


class lkv_kernel_stat(C.Structure):
    _fields_ = [("name", C.c_char * 24), ("launches", C.c_int64), ("total_ms", C.c_double)]


class LKVError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH):
    """Load liblkv.so (raises if it is missing: build it first)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"liblkv.so not found at {path}; build it with "
                "`python -m cluster_indexed_kv_gb300.builder` (needs nvcc)")
        L = C.CDLL(path)
        vp, i32, i64, u64, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_float
        st = C.c_int
        L.lkv_create.argtypes = [C.POINTER(lkv_config), C.POINTER(vp)]
        L.lkv_create.restype = st
        L.lkv_destroy.argtypes = [vp]
        L.lkv_destroy.restype = None
        L.lkv_build_index.argtypes = [vp, i32, vp, vp, i64, i32, i32, u64]
        L.lkv_build_index.restype = st
        L.lkv_build_index_async.argtypes = [vp, i32, vp, vp, i64, i32, i32, u64, vp, vp]
        L.lkv_build_index_async.restype = st
        L.lkv_load_index.argtypes = [vp, i32, vp, vp, i64, i32, vp, vp]
        L.lkv_load_index.restype = st
        L.lkv_decode_step.argtypes = [vp, i32, i32, vp, vp, vp, f32, i32, i32, vp, vp, vp, vp, vp]
        L.lkv_decode_step.restype = st
        L.lkv_decode_steps.argtypes = [vp, i32, i32, i32, vp, vp, vp, f32, i32, i32, vp, vp, vp,
                                       vp, vp]
        L.lkv_decode_steps.restype = st
        L.lkv_set_profiling.argtypes = [vp, i32]
        L.lkv_set_profiling.restype = st
        L.lkv_set_kmeans_filter.argtypes = [vp, i32]
        L.lkv_set_kmeans_filter.restype = st
        L.lkv_get_profile.argtypes = [vp, vp, i32, C.POINTER(i32), vp, i32]
        L.lkv_get_profile.restype = st
        L.lkv_get_index.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, C.POINTER(i32)]
        L.lkv_get_index.restype = st
        L.lkv_get_decode_state.argtypes = [vp, i32, i32, C.POINTER(lkv_decode_state)]
        L.lkv_get_decode_state.restype = st
        L.lkv_kmeans_static.argtypes = [vp, i32, i64, i32, i32, u64, vp, vp, vp]
        L.lkv_kmeans_static.restype = st
        L.lkv_kmeans_static_status.argtypes = [vp]
        L.lkv_kmeans_static_status.restype = st
        L.lkv_uva_read.argtypes = [vp, vp, i64, vp]
        L.lkv_uva_read.restype = st
        L.lkv_read_ceiling.argtypes = [vp, i64, vp]
        L.lkv_read_ceiling.restype = st
        L.lkv_diag_wait_timeout.argtypes = [vp, i64]
        L.lkv_diag_wait_timeout.restype = st
        L.lkv_set_policy.argtypes = [vp, C.POINTER(lkv_policy)]
        L.lkv_set_policy.restype = st
        L.lkv_build_pages.argtypes = [vp, i32, vp, vp, i64, i32]
        L.lkv_build_pages.restype = st
        L.lkv_build_paris.argtypes = [vp, i32, vp, vp, i64, C.POINTER(lkv_paris_params)]
        L.lkv_build_paris.restype = st
        L.lkv_paris_levels.argtypes = [vp, vp]
        L.lkv_paris_levels.restype = st
        L.lkv_sync.argtypes = [vp]
        L.lkv_sync.restype = st
        L.lkv_last_error.argtypes = [vp]
        L.lkv_last_error.restype = C.c_char_p
        _lib = L
        return L


def _check(status: int, ctx) -> None:
    if status != LKV_OK:
        msg = load().lkv_last_error(ctx)
        raise LKVError(status, msg.decode() if msg else "")


def lkv_create(cfg: lkv_config):
    h = C.c_void_p()
    _check(load().lkv_create(C.byref(cfg), C.byref(h)), None)
    return h


def lkv_destroy(ctx) -> None:
    load().lkv_destroy(ctx)


def lkv_build_index(ctx, layer, keys_ptr, values_ptr, n_tokens, n_clusters, iters, seed):
    _check(load().lkv_build_index(ctx, layer, keys_ptr, values_ptr, n_tokens, n_clusters,
                                  iters, seed), ctx)


def lkv_build_index_async(ctx, layer, keys_ptr, values_ptr, n_tokens, n_clusters, iters, seed,
                          ready_event, done_event):
    _check(load().lkv_build_index_async(ctx, layer, keys_ptr, values_ptr, n_tokens, n_clusters,
                                        iters, seed, ready_event, done_event), ctx)


def lkv_load_index(ctx, layer, keys_ptr, values_ptr, n_tokens, n_clusters, assign_ptr, cent_ptr):
    _check(load().lkv_load_index(ctx, layer, keys_ptr, values_ptr, n_tokens, n_clusters,
                                 assign_ptr, cent_ptr), ctx)


def lkv_decode_step(ctx, layer, n_layers, q_ptr, k_ptr, v_ptr, tau, budget, local_buf,
                    out_ptr, sel_ptr, nsel_ptr, boundary_ptr, r_ptr):
    _check(load().lkv_decode_step(ctx, layer, n_layers, q_ptr, k_ptr, v_ptr, tau, budget,
                                  local_buf, out_ptr, sel_ptr, nsel_ptr, boundary_ptr, r_ptr), ctx)


def lkv_decode_steps(ctx, layer, n_layers, n_steps, q_ptr, k_ptr, v_ptr, tau, budget, local_buf,
                     out_ptr, sel_ptr, nsel_ptr, boundary_ptr, r_ptr):
    _check(load().lkv_decode_steps(ctx, layer, n_layers, n_steps, q_ptr, k_ptr, v_ptr, tau,
                                   budget, local_buf, out_ptr, sel_ptr, nsel_ptr, boundary_ptr,
                                   r_ptr), ctx)


def lkv_set_policy(ctx, trigger: int, interval: int, fill: int, page: int, per_head: int = 0) -> None:
    pol = lkv_policy(trigger, interval, fill, page, per_head)
    _check(load().lkv_set_policy(ctx, C.byref(pol)), ctx)


def lkv_build_pages(ctx, layer, keys_ptr, values_ptr, n_tokens, page):
    _check(load().lkv_build_pages(ctx, layer, keys_ptr, values_ptr, n_tokens, page), ctx)


def lkv_build_paris(ctx, layer, keys_ptr, values_ptr, n_tokens, rho, n_cand, seed):
    prm = lkv_paris_params(rho, n_cand, seed)
    _check(load().lkv_build_paris(ctx, layer, keys_ptr, values_ptr, n_tokens, C.byref(prm)), ctx)


def lkv_paris_levels():
    """(thresholds [7], bin means [8]) as lists of floats (host only)."""
    thr, lev = (C.c_float * 7)(), (C.c_float * 8)()
    _check(load().lkv_paris_levels(thr, lev), None)
    return list(thr), list(lev)


def lkv_set_profiling(ctx, enable: bool) -> None:
    _check(load().lkv_set_profiling(ctx, 1 if enable else 0), ctx)


def lkv_set_kmeans_filter(ctx, filter_: int) -> None:
    _check(load().lkv_set_kmeans_filter(ctx, filter_), ctx)


def lkv_get_profile(ctx, reset: bool = False):
    """(dict kernel -> (launches, total_ms), dict of work counters)."""
    stats = (lkv_kernel_stat * 32)()
    n = C.c_int32(0)
    ctr = (C.c_int64 * 6)()
    _check(load().lkv_get_profile(ctx, stats, 32, C.byref(n), ctr, 1 if reset else 0), ctx)
    kern = {stats[i].name.decode(): (stats[i].launches, stats[i].total_ms) for i in range(n.value)}
    names = ("attn_rows", "attn_slices", "score_units", "gather_rows", "sel_units", "sel_tokens")
    return kern, {k: ctr[i] for i, k in enumerate(names)}


def lkv_get_index(ctx, layer, seq, kv_head, capacity, cent_ptr, len_ptr, row_ptr, assign_ptr,
                  perm_ptr) -> int:
    n = C.c_int32(0)
    _check(load().lkv_get_index(ctx, layer, seq, kv_head, capacity, cent_ptr, len_ptr, row_ptr,
                                assign_ptr, perm_ptr, C.byref(n)), ctx)
    return n.value


def lkv_get_decode_state(ctx, layer, seq) -> lkv_decode_state:
    s = lkv_decode_state()
    _check(load().lkv_get_decode_state(ctx, layer, seq, C.byref(s)), ctx)
    return s


def lkv_kmeans_static(keys_ptr, dtype, n_tokens, n_clusters, iters, seed, cent_ptr, assign_ptr,
                      stream_ptr) -> None:
    _check(load().lkv_kmeans_static(keys_ptr, dtype, n_tokens, n_clusters, iters, seed, cent_ptr,
                                    assign_ptr, stream_ptr), None)


def lkv_kmeans_static_status(stream_ptr) -> None:
    _check(load().lkv_kmeans_static_status(stream_ptr), None)


def lkv_uva_read(host_ptr, dev_ptr, nbytes: int, stream_ptr) -> None:
    _check(load().lkv_uva_read(host_ptr, dev_ptr, nbytes, stream_ptr), None)


def lkv_read_ceiling(dev_ptr, nbytes: int, stream_ptr) -> None:
    _check(load().lkv_read_ceiling(dev_ptr, nbytes, stream_ptr), None)


def lkv_diag_wait_timeout(ctx, limit_ns: int) -> None:
    _check(load().lkv_diag_wait_timeout(ctx, limit_ns), ctx)


def lkv_sync(ctx) -> None:
    _check(load().lkv_sync(ctx), ctx)


def lkv_last_error(ctx) -> str:
    m = load().lkv_last_error(ctx)
    return m.decode() if m else ""
