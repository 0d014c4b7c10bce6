"""Benchmark: LouisKV-style retrieval decode at 32K input, batch 8, on one GB300.

One bench step = one pass of the whole hot path over one batch: the prefill
index build (K-means, 20 Lloyd rounds, C = 2048, N = 32768 keys per
(sequence, KV head), 8 sequences x 8 KV heads) followed by T = 8192 decode
steps (boundary test, segment/eviction bookkeeping, group scoring and budget
selection on triggers, sparse attention every step) of all 8 sequences.

Printed (one JSON line, rank 0): value = decode steps/s (one decode step =
all 8 sequences advance one token), k-means Mkeys/s, the attention kernel's
HBM roofline fraction, the oracle timed on the host cores, an end-to-end
number through the C ABI with host buffers, and the SM clocks seen.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--decode-steps T] [--iters I]
Under torchrun (N > 1) every rank runs an independent replica (weak scaling,
no collective on the data path); rank 0 prints the aggregate.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode steps/s (retrieval+sparse attn) @32K, B=8; k-means Mkeys/s; % HBM roofline"
UNIT = "decode steps/s"


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--decode-steps", type=int, default=None)
    p.add_argument("--iters", type=int, default=None)
    p.add_argument("--profile-steps", type=int, default=512)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-probes", action="store_true",
                   help="skip the host-offload/UVA and 4-layer probes of the default workload")
    p.add_argument("--workload", default="b8_32k",
                   help="synthetic workload (default: the 32K-input, batch-8 decode workload)")
    return p.parse_args(argv)


def max_over_ranks(values):
    """Element-wise maximum of a list of floats over all ranks (the list
    itself with one rank)."""
    import torch
    import torch.distributed as td
    if not (td.is_available() and td.is_initialized()) or td.get_world_size() == 1:
        return list(values)
    dev = "cuda" if td.get_backend() == "nccl" else "cpu"
    t = torch.tensor(list(values), dtype=torch.float64, device=dev)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return t.tolist()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload(args):
    import synth
    w = synth.WORKLOADS[args.workload]
    if args.decode_steps:
        w = w.replace(n_steps=args.decode_steps)
    if args.iters:
        w = w.replace(iters=args.iters)
    return w


def config_of(w, world):
    return {"workload": f"{w.name}: B={w.batch}, N={w.n_prefill}, C={w.n_clusters}, "
                        f"iters={w.iters}, T={w.n_steps}, tau={w.tau}, budget={w.budget}, "
                        f"L={w.local_buf}, H_kv={w.n_kv_heads}x{w.group}, d={w.head_dim}, "
                        f"jump_p={w.jump_p}",
            "batch_per_gpu": w.batch, "prefill_tokens": w.n_prefill, "decode_steps": w.n_steps,
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 between timed steps (1.07 GB prefill K/V, "
                  f"{w.n_steps * w.batch * (w.n_heads + 2 * w.n_kv_heads) * 256 / 1e9:.2f} GB decode "
                  "inputs); the roofline pass writes 256 MB, then reads another 256 MB, before every decode step"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(os.path.join("/tmp", f"lkv_clocks_{os.getpid()}.csv"), "w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        self.out.close()
        try:
            os.unlink(self.out.name)
        except OSError:
            pass
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[1]) for r in rows if len(r) > 1) if v is not None]
        mx = [v for v in (num(r[2]) for r in rows if len(r) > 2) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 5 + i and r[5 + i].strip() == "Active"})
        load = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- oracle samples

def oracle_decode_sample(K0, V0, idx, q, kn, vn, w, n_steps, head=0):
    """Seconds per (sequence, KV head) decode step of the oracle, timed on one
    KV head of sequence 0 over n_steps steps (K0, V0: [H_kv, N, d])."""
    import numpy as np
    import oracle
    import synth
    h = head
    g0, g1 = h * w.group, (h + 1) * w.group
    keys = synth.to_oracle(K0[h:h + 1])
    vals = synth.to_oracle(V0[h:h + 1])
    qq = synth.to_oracle(q[:n_steps, 0, 0, g0:g1])
    kk = synth.to_oracle(kn[:n_steps, 0, 0, h:h + 1])
    vv = synth.to_oracle(vn[:n_steps, 0, 0, h:h + 1])
    assign = np.ascontiguousarray(idx["assign"][None])
    cent = np.ascontiguousarray(idx["centroids"][None, :w.n_clusters])
    t0 = time.perf_counter()
    oracle.decode(keys, vals, assign, cent, qq, kk, vv, n_clusters=w.n_clusters,
                  local_buf=w.local_buf, tau=w.tau, budget=w.budget)
    return (time.perf_counter() - t0) / n_steps


def oracle_kmeans_sample(keys_bits, c, n_keys):
    """Seconds for one Lloyd round of the oracle on n_keys keys, c clusters."""
    import numpy as np
    import oracle
    keys = np.ascontiguousarray(keys_bits[:n_keys])
    cent = oracle.bf16_bits_to_f32(keys_bits[:c]).astype(np.float32)
    t0 = time.perf_counter()
    a = oracle.assign(keys, oracle.operand(cent, oracle.BF16))
    oracle.update(keys, a, cent)
    return time.perf_counter() - t0


# Arm "CPU part" numbers of /proc/cpuinfo (implementer 0x41) that name a core
_ARM_PARTS = {"0xd4f": "Arm Neoverse-V2", "0xd40": "Arm Neoverse-V1", "0xd0c": "Arm Neoverse-N1",
              "0xd49": "Arm Neoverse-N2"}


def host_cpu():
    """(logical CPUs, CPU model) of this host."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                if k.strip() in ("model name", "Model", "CPU part") and v.strip():
                    model = v.strip()
                    if k.strip() == "CPU part" and model in _ARM_PARTS:
                        model = f"{_ARM_PARTS[model]} (CPU part {model})"
                    if k.strip() == "model name":
                        break
    except OSError:
        pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return os.cpu_count(), model


def cpu_baseline(K, V, idx0, q, kn, vn, w, n_steps=48, kmeans_keys=1024):
    import synth
    per = oracle_decode_sample(K[0].cpu(), V[0].cpu(), idx0, q, kn, vn, w, n_steps)
    units = w.batch * w.n_kv_heads * w.n_layers
    steps_per_s = 1.0 / (per * units)
    km = oracle_kmeans_sample(synth.to_oracle(K[0, 0]), w.n_clusters, kmeans_keys)
    nproc, model = host_cpu()
    return {"value": steps_per_s, "unit": UNIT, "cores": 1, "kind": "oracle",
            "host_nproc": nproc, "host_cpu": model,
            "sample": f"single-threaded C oracle: 1 (sequence, layer, KV head) x {n_steps} decode "
                      f"steps of the full-size workload (teacher-forced from the GPU index), scaled "
                      f"by B x layers x H_kv = {units}; k-means: one Lloyd round of "
                      f"{kmeans_keys} keys x {w.n_clusters} clusters",
            "kmeans_mkeys_per_s": kmeans_keys / km / 1e6}


# ---------------------------------------------------------------- our arm

def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured")
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_sha256(source, region):
    """SHA-256 of the part of `source` from the line `region[0]` up to the
    line `region[1]` (the kernel and its device helpers)."""
    import hashlib
    with open(os.path.join(ROOT, source)) as f:
        text = f.read()
    i = text.index(region[0])
    j = text.index(region[1], i)
    return hashlib.sha256(text[i:j].encode()).hexdigest()


def ncu_traffic(kernel, units):
    """DRAM bytes per launch from the committed ncu summary, scaled to
    `units` (the launch's work units) when the capture ran a smaller case;
    None when the kernel's source changed after the capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.txt")) as f:
            rec = json.load(f)[kernel]
        if kernel_source_sha256(rec["source"], rec["region"]) != rec["region_sha256"]:
            return None
        return rec["dram_bytes_per_launch"] * units / rec["units_per_launch"]
    except Exception:
        return None


def attn_roofline(kern, ctr, w, eb):
    """(launches, total ms, algorithmic bytes per launch, seconds per launch,
    GB/s) of the attention from a profiled pass: every K and V row attended
    once, plus the queries read and the fp32 outputs written."""
    n_attn, ms_attn = kern["lkv_attn"]
    slices = ctr["attn_slices"]
    alg = (ctr["attn_rows"] * 2 * 128 * eb + slices * w.group * 128 * (eb + 4)) / max(n_attn, 1)
    sec = ms_attn / max(n_attn, 1) / 1e3
    return n_attn, ms_attn, alg, sec, alg / sec / 1e9


class L2Flush:
    """Overwrites L2 before a measured launch: writes a 256 MB buffer (about
    twice the 129 MB L2), then reads another 256 MB with plain loads
    (lkv_read_ceiling). L2 then holds clean lines of data the measured
    kernel does not touch, so the write-back of the written lines is not
    charged to that kernel's first reads."""

    def __init__(self, torch, device="cuda"):
        self.torch = torch
        self.w = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
        self.r = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.int32, device=device)

    def fill_(self, x):
        from cluster_indexed_kv_gb300 import _lib
        self.w.fill_(x)
        _lib.lkv_read_ceiling(self.r.data_ptr(), self.r.numel() * 4,
                              self.torch.cuda.current_stream().cuda_stream)


def read_ceiling(torch, nbytes, flush, hbm_peak, reps=16):
    """Event-timed single launches of lkv_read_ceiling over nbytes of device
    memory, L2 overwritten before each (as in the attention's roofline
    pass): the rate one launch that reads that many bytes reaches."""
    from cluster_indexed_kv_gb300 import _lib
    nbytes = int(nbytes) // 16 * 16
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    ms = 0.0
    for r in range(reps + 2):
        flush.fill_(float(r))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        _lib.lkv_read_ceiling(buf.data_ptr(), nbytes, st.cuda_stream)
        e1.record(st)
        e1.synchronize()
        if r >= 2:
            ms += e0.elapsed_time(e1)
    sec = ms / reps / 1e3
    del buf
    return {"bytes": nbytes, "avg_launch_us": sec * 1e6, "achieved": nbytes / sec / 1e9,
            "frac_of_hbm": nbytes / sec / 1e9 / hbm_peak, "unit": "GB/s",
            "kernel": "lkv_read_ceiling: plain 16-byte loads over a grid that fills the GPU",
            "l2": "256 MB written, then 256 MB read, before every launch"}


def l2_read_ceiling(torch, nbytes, reps=32):
    """Sustained rate at which lkv_read_ceiling reads nbytes of device memory
    that L2 holds: two untimed launches, then `reps` launches back to back
    between one pair of CUDA events (so launch gaps are hidden, as the
    overlapped launches of the decode graph hide them). The timed decode
    graph's attention reads most of its rows from L2, so this is its
    ceiling."""
    from cluster_indexed_kv_gb300 import _lib
    nbytes = int(nbytes) // 16 * 16
    buf = torch.ones(nbytes // 4, dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(2):
        _lib.lkv_read_ceiling(buf.data_ptr(), nbytes, st.cuda_stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(reps):
        _lib.lkv_read_ceiling(buf.data_ptr(), nbytes, st.cuda_stream)
    e1.record(st)
    e1.synchronize()
    sec = e0.elapsed_time(e1) / reps / 1e3
    del buf
    return {"bytes": nbytes, "avg_launch_us": sec * 1e6, "achieved": nbytes / sec / 1e9, "unit": "GB/s",
            "kernel": f"lkv_read_ceiling over a buffer that L2 holds, {reps} launches back to back"}


def in_graph_attention(g_bytes, g_sec, launches, hbm_peak, l2c=None):
    """The attention as the timed decode graph runs it: algorithmic bytes
    per step over the decode time per step, and the DRAM bytes per step of
    a whole 512-step graph from the committed ncu record (cache control
    off). Consecutive steps attend nearly the same rows (the selection
    changes only at retrieval steps), so most of them come from L2: the
    algorithmic rate is not an HBM rate."""
    dram = ncu_traffic("lkv_attn_graph", g_bytes)
    out = {"achieved_alg": g_bytes / g_sec / 1e9, "frac_alg_of_hbm": g_bytes / g_sec / 1e9 / hbm_peak,
           "unit": "GB/s", "alg_bytes_per_step": g_bytes, "us_per_step": g_sec * 1e6,
           "steps": launches, "dram_bytes_per_step": dram,
           "timing": "CUDA events on the context stream around the timed decode graphs; about nine "
                     "attentions overlap, and the time per step includes the boundary and "
                     "selection kernels"}
    if dram is not None:
        out["dram_GBps"] = dram / g_sec / 1e9
        out["dram_frac_of_hbm"] = dram / g_sec / 1e9 / hbm_peak
        out["l2_served_frac"] = 1.0 - dram / g_bytes
    if l2c is not None:
        out["l2_read_ceiling"] = l2c
        out["frac_alg_of_l2_ceiling"] = g_bytes / g_sec / 1e9 / l2c["achieved"]
    return out


def timed_decode(torch, ctx, q, kn, vn, tau, budget, out, warm, n, boundary=None, **kw):
    """Decode steps warm .. warm + n - 1 through the graph path, timed with
    CUDA events on the context stream, after an untimed call for steps
    0 .. warm - 1 (which also captures the decode graphs, so the timed call
    only replays them). Every per-step buffer is passed from the call's own
    first step, as a caller walking full-length buffers chunk by chunk does:
    then both calls present the same graph arguments. Returns steps/s."""
    b0 = {} if boundary is None else {"boundary": boundary[:warm]}
    ctx.decode_steps(0, q[:warm], kn[:warm], vn[:warm], tau, budget, out[:warm], **b0, **kw)
    ctx.sync()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sl = slice(warm, warm + n)
    b1 = {} if boundary is None else {"boundary": boundary[sl]}
    e0.record(ctx.stream)
    ctx.decode_steps(0, q[sl], kn[sl], vn[sl], tau, budget, out[sl], **b1, **kw)
    e1.record(ctx.stream)
    e1.synchronize()
    return n / (e0.elapsed_time(e1) / 1e3)


def graph_attention(ctr, w, eb, dec_ms, launches):
    """The attention as it runs in the timed decode: its algorithmic bytes
    over every timed step (device row counters, so the filling of the local
    buffer is counted as it happened) and the time per launch in the
    pipeline (the timed decode time over the launches; about nine attention
    launches overlap in the graph, and the boundary and selection kernels'
    time is included). Returns (bytes per launch, seconds per launch)."""
    b = ctr["attn_rows"] * 2 * 128 * eb + ctr["attn_slices"] * w.group * 128 * (eb + 4)
    return b / max(launches, 1), dec_ms / 1e3 / max(launches, 1)


def selection_rooflines(kern, ctr, w, eb, hbm_peak, peak_kind):
    """HBM roofline of the scoring + selection kernel from a profiled pass in
    which every slice retrieves. Per slice it reads one centroid-operand row
    per unit (d elements), the group's queries, and a length and a first
    pool row per unit (8 bytes), and writes the selected ids, first rows and
    token offsets (12 bytes a selected unit) and the pool row of every
    selected token (4 bytes)."""
    n, ms = kern["lkv_select"]
    slices = ctr["attn_slices"]
    b = (ctr["score_units"] * (128 * eb + 8) + slices * w.group * 128 * eb
         + ctr["sel_units"] * 12 + ctr["sel_tokens"] * 4) / max(n, 1)
    sec = ms / max(n, 1) / 1e3
    a = b / sec / 1e9 if sec > 0 else None
    return {"k_select": {"bound": "hbm", "achieved": a, "peak": hbm_peak, "unit": "GB/s",
                         "frac": a / hbm_peak if a else None, "alg_bytes_per_launch": b,
                         "avg_launch_us": sec * 1e6, "launches": int(n),
                         "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                         "note": "scoring and budget selection in one kernel"}}


def run_ours(args, rank, world, local):
    import torch
    import synth
    import cluster_indexed_kv_gb300 as lkv

    torch.cuda.set_device(local)
    lkv.build()
    w = workload(args)
    T, NL = w.n_steps, w.n_layers
    dev = "cuda"
    KV = [synth.prefill(w, layer, dev) for layer in range(NL)]
    K, V = KV[0]
    q, kn, vn, _ = synth.decode_inputs(w, dev, n_steps=T)
    prof_T = min(args.profile_steps, T)
    ctx = lkv.Context(batch=w.batch, n_layers=NL, n_kv_heads=w.n_kv_heads, group=w.group,
                      dtype=w.torch_dtype, local_buf=w.local_buf, max_clusters=w.n_clusters,
                      max_prefill=w.n_prefill, max_steps=T, max_budget=w.budget, offload=w.offload)
    stream = ctx.stream
    out = torch.empty(T, w.batch, NL, w.n_heads, 128, device=dev)
    bnd = torch.zeros(T, w.batch, NL, dtype=torch.uint8, device=dev)
    ev = {}

    def build_all():
        for layer, (Kl, Vl) in enumerate(KV):
            ctx.build_index(layer, Kl, Vl, w.n_clusters, w.iters, 1)

    def one_step():
        build_all()
        ev["mid"].record(stream)
        # an NVTX range around the decode lets a profiler select its graphs
        torch.cuda.nvtx.range_push("decode_steps")
        ctx.decode_steps(0, q, kn, vn, w.tau, w.budget, out, n_layers=NL, boundary=bnd)
        torch.cuda.nvtx.range_pop()

    ev["mid"] = torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        one_step()
    ctx.sync()
    ctx.profile(reset=True)
    dist = world > 1 and torch.distributed.is_initialized()
    if dist:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    build_ms = dec_ms = 0.0
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        e0 = torch.cuda.Event(enable_timing=True)
        ev["mid"] = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        one_step()
        e1.record(stream)
        e1.synchronize()
        build_ms += e0.elapsed_time(ev["mid"])
        dec_ms += ev["mid"].elapsed_time(e1)
    torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    kern, ctr_timed = ctx.profile(reset=True)
    launches = int(sum(v[0] for v in kern.values()))
    trig = float(bnd.float().mean().item())
    st = ctx.decode_state(0, 0)
    build_ms, dec_ms, wall_ms = max_over_ranks([build_ms, dec_ms, wall * 1e3])
    K_steps = args.steps
    value = world * T * K_steps / (dec_ms / 1e3)
    mkeys = world * NL * w.batch * w.n_kv_heads * w.n_prefill * w.iters * K_steps / (build_ms / 1e3) / 1e6

    # ---- roofline pass: the decode first advances through the pipelined graph
    # until the local buffer has been full for a while, then prof_T
    # single-step launches run with L2 overwritten before every step and CUDA
    # events around every kernel on the context stream
    flush = L2Flush(torch, dev)
    build_all()
    warm = max(0, min(T - prof_T, max(2 * w.local_buf, 1024)))
    if warm:
        ctx.decode_steps(0, q[:warm], kn[:warm], vn[:warm], w.tau, w.budget, out[:warm],
                         n_layers=NL)
    ctx.set_profiling(True)
    ctx.profile(reset=True)
    for t in range(warm, warm + prof_T):
        flush.fill_(float(t))
        ctx.decode_step(0, q[t], kn[t], vn[t], w.tau, w.budget, out[t], n_layers=NL,
                        boundary=bnd[t])
    kern_p, ctr = ctx.profile(reset=True)
    ctx.set_profiling(False)
    hbm_peak, tc_peak, tc_peak_sus, peak_kind = peaks()
    eb = 2 if w.dtype == "bf16" else 4
    n_attn, ms_attn, alg_bytes, attn_s, achieved = attn_roofline(kern_p, ctr, w, eb)
    g_launches = T * K_steps  # one attention launch per step covers all NL layers
    ceiling = read_ceiling(torch, alg_bytes, flush, hbm_peak)
    l2c = l2_read_ceiling(torch, alg_bytes)
    g_bytes, g_sec = graph_attention(ctr_timed, w, eb, dec_ms, g_launches)
    breakdown = {k: {"launches": int(v[0]), "avg_us": round(v[1] / v[0] * 1e3, 2)}
                 for k, v in kern_p.items() if v[0]}

    # ---- scoring and selection kernels: single-step launches in which every
    # slice retrieves (tau above any r_t), L2 overwritten before every step
    sel_lane = None
    sel_T = min(128, T - warm - prof_T)
    if sel_T >= 16:
        t0 = warm + prof_T
        ctx.set_profiling(True)
        ctx.profile(reset=True)
        for t in range(t0, t0 + sel_T):
            flush.fill_(float(t))
            ctx.decode_step(0, q[t], kn[t], vn[t], 2.0, w.budget, out[t], n_layers=NL)
        kern_s, ctr_s = ctx.profile(reset=True)
        ctx.set_profiling(False)
        sel_lane = selection_rooflines(kern_s, ctr_s, w, eb, hbm_peak, peak_kind)
        sel_lane["steps"] = f"decode steps {t0}..{t0 + sel_T - 1}, tau 2.0 (every slice retrieves)"
        # the chunked selection that the decode graph runs: one launch scores
        # and selects the retrievals of 64 steps side by side
        t1 = t0 + sel_T
        if t1 + 128 <= T:
            ctx.set_profiling(True)
            ctx.profile(reset=True)
            ctx.decode_steps(0, q[t1:t1 + 128], kn[t1:t1 + 128], vn[t1:t1 + 128], 2.0, w.budget,
                             out[t1:t1 + 128], n_layers=NL)
            kern_c, ctr_c = ctx.profile(reset=True)
            ctx.set_profiling(False)
            ch = selection_rooflines(kern_c, ctr_c, w, eb, hbm_peak, peak_kind)["k_select"]
            ch["kernel"] = "k_select_chunk"
            ch["us_per_step"] = ch["avg_launch_us"] / 64
            ch["note"] = ("64 steps per launch, every slice retrieving at every step, no L2 flush "
                          "inside the launch: the steps of a chunk score the same centroid table, "
                          "so most of its rows come from L2")
            sel_lane["k_select_chunk"] = ch
            sel_lane["chunk_steps"] = f"decode steps {t1}..{t1 + 127}, tau 2.0, profiled chunk launches"

    # ---- K-means distance contraction on the tensor cores: one build with
    # CUDA events around every kernel (L2 overwritten first; the keys, 537 MB,
    # exceed L2 anyway)
    flush.fill_(-1.0)
    ctx.set_profiling(True)
    ctx.profile(reset=True)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, 1)
    kern_b, _ = ctx.profile(reset=True)
    ctx.set_profiling(False)
    S = w.batch * w.n_kv_heads
    km_kernel = "kmeans_assign_tc" if kern_b.get("kmeans_assign_tc", (0, 0))[0] else "kmeans_assign"
    n_km, ms_km = kern_b[km_kernel]
    km_flops = 2.0 * S * w.n_prefill * w.n_clusters * 128
    km_s = ms_km / max(n_km, 1) / 1e3
    km_tf = km_flops / km_s / 1e12
    build_breakdown = {k: {"launches": int(v[0]), "avg_us": round(v[1] / v[0] * 1e3, 2)}
                       for k, v in kern_b.items() if v[0]}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K_steps,
        "warmup": args.warmup, "ms_per_step": wall_ms / K_steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": config_of(w, world),
        "tokens_per_s": value * w.batch,
        "kmeans_mkeys_per_s": mkeys,
        "decode_ms_per_bench_step": dec_ms / K_steps, "build_ms_per_bench_step": build_ms / K_steps,
        "trigger_rate": trig, "kmeans_refined_keys_total": st["n_refined"],
        "roofline": {"kernel": "lkv_attn", "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                     "unit": "GB/s", "frac": achieved / hbm_peak,
                     "traffic": ncu_traffic("lkv_attn", alg_bytes),
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                     "alg_bytes_per_launch": alg_bytes, "avg_launch_us": attn_s * 1e6,
                     "launches": int(n_attn), "l2": "single-step launches; before every step 256 MB written, then 256 MB read",
                     "single_launch_read_ceiling": ceiling,
                     "frac_of_single_launch_ceiling": achieved / ceiling["achieved"],
                     "in_graph": in_graph_attention(g_bytes, g_sec, g_launches, hbm_peak, l2c)},
        "roofline_kmeans_assign": {
            "kernel": "k_assign_tc" if km_kernel == "kmeans_assign_tc" else "k_assign_simt",
            "bound": "tensor", "achieved": km_tf, "peak": tc_peak, "unit": "TFLOP/s",
            "frac": km_tf / tc_peak, "frac_of_sustained": km_tf / tc_peak_sus,
            "traffic": ncu_traffic("k_assign_tc", S) if km_kernel == "kmeans_assign_tc" else None,
            "peak_source": f"{peak_kind} bf16_tflops (cuBLAS burst)",
            "flops_per_launch": km_flops, "avg_launch_us": km_s * 1e6, "launches": int(n_km)},
        "roofline_selection_lane": sel_lane,
        "kernel_breakdown_us": breakdown,
        "build_breakdown_us": build_breakdown,
        "gpu_launches": launches,
        "clocks": clk,
    }

    # ---- end to end through the C ABI with host buffers: every decode step's
    # inputs come from pinned host memory and its outputs go back to it. The
    # steps go in chunks of 2048 (one decode graph each); a chunk's
    # host-to-device copy (its own stream) overlaps the previous chunk's
    # decode, and its device-to-host copy (a third stream) overlaps the next.
    if not args.no_e2e:
        qh, knh, vnh = (x.cpu().pin_memory() for x in (q, kn, vn))
        outh = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d = (q[0].numel() + kn[0].numel() + vn[0].numel()) * eb
        d2h = out[0].numel() * 4
        chunk = 2048
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

        def e2e_pass():
            build_all()
            ctx.sync()
            torch.cuda.synchronize()
            ea, eb_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(s_in)
            for c0 in range(0, T, chunk):
                n = min(chunk, T - c0)
                with torch.cuda.stream(s_in):
                    q[c0:c0 + n].copy_(qh[c0:c0 + n], non_blocking=True)
                    kn[c0:c0 + n].copy_(knh[c0:c0 + n], non_blocking=True)
                    vn[c0:c0 + n].copy_(vnh[c0:c0 + n], non_blocking=True)
                    inputs_in = torch.cuda.Event()
                    inputs_in.record(s_in)
                stream.wait_event(inputs_in)
                ctx.decode_steps(0, q[c0:c0 + n], kn[c0:c0 + n], vn[c0:c0 + n], w.tau, w.budget,
                                 out[c0:c0 + n], n_layers=NL)
                decoded = torch.cuda.Event()
                decoded.record(stream)
                s_out.wait_event(decoded)
                with torch.cuda.stream(s_out):
                    outh[c0:c0 + n].copy_(out[c0:c0 + n], non_blocking=True)
            eb_.record(s_out)
            eb_.synchronize()
            return ea.elapsed_time(eb_)

        e2e_pass()  # untimed: captures the decode graphs this call sequence uses
        e2e_ms = e2e_pass()
        result["e2e"] = {"value": world * T / (e2e_ms / 1e3), "unit": UNIT,
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    idx0 = ctx.get_index(0, 0, 0, w.n_prefill) if want_cpu else None
    ctx.close()
    if not args.no_probes and args.workload == "b8_32k":
        del out, flush
        torch.cuda.empty_cache()
        result["uva_gather"] = offload_probe(torch, hbm_peak)
        torch.cuda.empty_cache()
        result["multi_layer"] = multi_layer_probe(torch, w, hbm_peak, peak_kind)
        torch.cuda.empty_cache()
        result["policy_baselines"] = policy_probe(torch, w)
        torch.cuda.empty_cache()
        result["async_build"] = async_build_probe(torch)
        torch.cuda.empty_cache()
        result["paris_selector"] = paris_probe(torch, w)
        torch.cuda.empty_cache()
    if want_cpu:
        result["cpu_baseline"] = cpu_baseline(K, V, idx0, q, kn, vn, w)
    return result


def offload_probe(torch, hbm_peak):
    """The host-offload shape on one layer (8 KV heads x 131072 keys in pinned
    host memory, C = 8192, budget 2048, L = 512): the UVA gather's rate on
    steps where every slice retrieves, against the ceiling of a plain UVA
    read of 1 GiB of pinned host memory on the same link (lkv_uva_read), and
    the decode rate of this shape through the pipelined graph at tau 0.7."""
    import synth
    import cluster_indexed_kv_gb300 as lkv
    from cluster_indexed_kv_gb300 import _lib
    W0, T1, T2 = 128, 256, 128
    w = synth.WORKLOADS["offload"].replace(n_layers=1, iters=2, n_steps=W0 + T1 + T2)
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    ctx = lkv.Context(batch=1, n_layers=1, n_kv_heads=w.n_kv_heads, group=w.group,
                      dtype=w.torch_dtype, local_buf=w.local_buf, max_clusters=w.n_clusters,
                      max_prefill=w.n_prefill, max_steps=w.n_steps, max_budget=w.budget,
                      offload=True)
    ctx.build_index(0, K, V, w.n_clusters, w.iters, 1)
    del K, V
    out = torch.empty(w.n_steps, 1, 1, w.n_heads, 128, device="cuda")
    ctx.sync()
    steps_per_s = timed_decode(torch, ctx, q, kn, vn, w.tau, w.budget, out, W0, T1)
    ctx.set_profiling(True)
    ctx.profile(reset=True)
    for t in range(W0 + T1, W0 + T1 + T2):
        ctx.decode_step(0, q[t], kn[t], vn[t], 2.0, w.budget, out[t])
    kern, ctr = ctx.profile(reset=True)
    ctx.close()
    n_g, ms_g = kern["lkv_gather_offload"]
    g_bytes = ctr["gather_rows"] * 2 * 128 * 2
    achieved = g_bytes / (ms_g / 1e3) / 1e9
    # the link's ceiling: plain streaming read of pinned host memory over UVA
    nbytes = 1 << 30
    host = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    host.fill_(1)
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = float("inf")
    for _ in range(4):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        _lib.lkv_uva_read(host.data_ptr(), dst.data_ptr(), nbytes, torch.cuda.current_stream().cuda_stream)
        b.record()
        b.synchronize()
        best = min(best, a.elapsed_time(b))
    ceiling = nbytes / (best / 1e3) / 1e9
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    dst.copy_(host, non_blocking=True)
    b.record()
    b.synchronize()
    dma = nbytes / (a.elapsed_time(b) / 1e3) / 1e9
    return {"kernel": "k_gather_offload", "bound": "host link", "achieved": achieved,
            "peak": ceiling, "unit": "GB/s", "frac": achieved / ceiling,
            "peak_source": "lkv_uva_read: plain 16-byte UVA reads of 1 GiB of pinned host memory "
                           "on this box (best of 4)",
            "dma_h2d_GBps": dma, "bytes": g_bytes, "launches": int(n_g),
            "avg_launch_us": ms_g / max(n_g, 1) * 1e3,
            "workload": "1 layer of the host-offload shape: 8 KV heads x 131072 keys in pinned "
                        "host memory, C=8192, budget 2048, L=512; gather timed on 128 steps "
                        "where every slice retrieves",
            "offload_decode_steps_per_s": steps_per_s,
            "offload_decode_note": f"{T1} steps at tau {w.tau} through the pipelined graph"}


def multi_layer_probe(torch, w0, hbm_peak, peak_kind):
    """The 32K-input, batch-8 workload with 4 attention layers decoded in one
    call per step (4 x 64 slices, about 200 MB of selected and local-buffer
    rows per step, more than L2 holds): decode steps/s through the pipelined
    graph, and the attention roofline of one 4-layer launch with L2
    overwritten before every step."""
    import synth
    import cluster_indexed_kv_gb300 as lkv
    NL, W0, T1, T2 = 4, 512, 1024, 64
    w = w0.replace(n_layers=NL, n_steps=W0 + T1 + T2)
    ctx = lkv.Context(batch=w.batch, n_layers=NL, n_kv_heads=w.n_kv_heads, group=w.group,
                      dtype=w.torch_dtype, local_buf=w.local_buf, max_clusters=w.n_clusters,
                      max_prefill=w.n_prefill, max_steps=w.n_steps, max_budget=w.budget)
    for layer in range(NL):
        K, V = synth.prefill(w, layer, "cuda")
        ctx.build_index(layer, K, V, w.n_clusters, w.iters, 1 + layer)
        del K, V
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    out = torch.empty(w.n_steps, w.batch, NL, w.n_heads, 128, device="cuda")
    ctx.sync()
    steps_per_s = timed_decode(torch, ctx, q, kn, vn, w.tau, w.budget, out, W0, T1, n_layers=NL)
    flush = L2Flush(torch)
    ctx.set_profiling(True)
    ctx.profile(reset=True)
    for t in range(W0 + T1, W0 + T1 + T2):
        flush.fill_(float(t))
        ctx.decode_step(0, q[t], kn[t], vn[t], w.tau, w.budget, out[t], n_layers=NL)
    kern, ctr = ctx.profile(reset=True)
    ctx.close()
    n_attn, _, alg, sec, achieved = attn_roofline(kern, ctr, w, 2)
    return {"workload": f"b8_32k x {NL} layers (one decode call per step for all layers)",
            "decode_steps_per_s": steps_per_s, "tokens_per_s": steps_per_s * w.batch,
            "decode_note": f"steps {W0}..{W0 + T1 - 1} through the pipelined graph (graphs "
                           f"captured by the untimed steps before)",
            "attn_roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                              "unit": "GB/s", "frac": achieved / hbm_peak,
                              "alg_bytes_per_launch": alg, "avg_launch_us": sec * 1e6,
                              "launches": int(n_attn), "peak_source": f"{peak_kind} hbm_gbs",
                              "l2": "before every step 256 MB written, then 256 MB read"}}


def policy_probe(torch, w0):
    """The retrieval policies on the 32K-input, batch-8 workload, each over
    the same inputs: the method (retrieval when r_t < tau, K-means clusters
    and boundary segments), retrieval at every step, at every 32nd step, and
    the page-granular every-step baseline (16-token pages of the input, as
    many units as clusters, and 16-token output pages). Per policy: decode
    steps/s through the pipelined graph (steps 512..2047, after untimed
    steps 0..511 that capture the graphs), then 256 single-step
    launches with CUDA events around every kernel (L2 overwritten before
    every step) for the share of the step that goes to scoring + selection
    (the retrieval; the K/V rows are read where they lie by the attention)."""
    import synth
    import cluster_indexed_kv_gb300 as lkv
    W0, T1, T2 = 512, 1536, 256
    w = w0.replace(n_steps=W0 + T1 + T2, iters=4)
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    out = torch.empty(w.n_steps, w.batch, 1, w.n_heads, 128, device="cuda")
    flush = L2Flush(torch)
    rows = {}
    policies = [("method: adaptive r_t < tau, clusters + segments", dict(), 0),
                ("every-step retrieval, clusters + segments", dict(trigger="every"), 0),
                ("every 32nd step, clusters + segments", dict(trigger="interval", interval=32), 0),
                ("every-step retrieval, 16-token pages in and out", dict(trigger="every", page=16), 16),
                ("method with a selection per query head (not group-consistent)", dict(per_head=True), 0)]
    for name, pol, pages in policies:
        ctx = lkv.Context(batch=w.batch, n_layers=1, n_kv_heads=w.n_kv_heads, group=w.group,
                          dtype=w.torch_dtype, local_buf=w.local_buf, max_clusters=w.n_clusters,
                          max_prefill=w.n_prefill, max_steps=w.n_steps, max_budget=w.budget)
        if pages:
            ctx.build_pages(0, K, V, pages)
        else:
            ctx.build_index(0, K, V, w.n_clusters, w.iters, 1)
        ctx.set_policy(**pol)
        bnd = torch.zeros(w.n_steps, w.batch, 1, dtype=torch.uint8, device="cuda")
        ctx.sync()
        sps = timed_decode(torch, ctx, q, kn, vn, w.tau, w.budget, out, W0, T1, boundary=bnd)
        ctx.set_profiling(True)
        ctx.profile(reset=True)
        for t in range(W0 + T1, W0 + T1 + T2):
            flush.fill_(float(t))
            ctx.decode_step(0, q[t], kn[t], vn[t], w.tau, w.budget, out[t], boundary=bnd[t])
        kern, ctr = ctx.profile(reset=True)
        ctx.close()
        ms = {k: v[1] for k, v in kern.items() if v[0]}
        total = sum(ms.values())
        retr = ms.get("lkv_select", 0.0) + ms.get("lkv_score", 0.0) + ms.get("lkv_gather_offload", 0.0)
        rows[name] = {"decode_steps_per_s": sps, "retrieval_rate": float(bnd.float().mean().item()),
                      "retrieval_share_of_step": retr / total if total else None,
                      "single_step_us": {k: round(v / T2 * 1e3, 2) for k, v in ms.items()},
                      "attended_rows_per_step": ctr["attn_rows"] / T2,
                      "attended_bytes_per_step": ctr["attn_rows"] * 2 * 128 * 2 / T2,
                      "selected_tokens_per_retrieval": ctr["sel_tokens"] / max(
                          1, int(bnd[W0 + T1:].sum().item()) * w.n_kv_heads)}
    return {"workload": "b8_32k (4 Lloyd rounds for the clustered rows)", "policies": rows,
            "note": "share = scoring+selection kernel time / all decode kernel time of the "
                    "single-step launches (the pages' breakdown also counts the host transfer "
                    "of an offloaded cache; here the rows stay in HBM). selected tokens per "
                    "retrieval count every query head's own selection in the per-head row (what "
                    "separate per-head gathers would move); its attended rows are the union "
                    "the kernel reads once per group"}


def paris_probe(torch, w0):
    """The ParisKV-style token selector on the 32K-input, batch-8 workload
    (same inputs, budget 1024 tokens, rho 4, 2560 candidates = 7.8% of the
    prefill): decode steps/s through the pipelined graph with the method's
    adaptive trigger and with retrieval at every step (steps 512..2047, after
    untimed steps that capture the graphs), then 128 single-step
    launches at every step (L2 overwritten before each) for the selection
    kernel's time and its HBM roofline (bucket bytes of every region token,
    codes and scales of every candidate, 16 + 128 bytes)."""
    import synth
    import cluster_indexed_kv_gb300 as lkv
    W0, T1, T2 = 512, 1536, 128
    w = w0.replace(n_steps=W0 + T1 + T2)
    K, V = synth.prefill(w, 0, "cuda")
    q, kn, vn, _ = synth.decode_inputs(w, "cuda")
    out = torch.empty(w.n_steps, w.batch, 1, w.n_heads, 128, device="cuda")
    flush = L2Flush(torch)
    res = {"workload": "b8_32k, ParisKV-style selector (rho 4, 2560 candidates, budget 1024 tokens)"}
    for name, pol in (("adaptive", dict()), ("every_step", dict(trigger="every"))):
        ctx = lkv.Context(batch=w.batch, n_layers=1, n_kv_heads=w.n_kv_heads, group=w.group,
                          dtype=w.torch_dtype, local_buf=w.local_buf, max_clusters=w.n_clusters,
                          max_prefill=w.n_prefill, max_steps=w.n_steps, max_budget=w.budget)
        ctx.build_paris(0, K, V, rho=4, n_cand=2560, seed=1)
        ctx.set_policy(**pol)
        ctx.sync()
        res[f"decode_steps_per_s_{name}"] = timed_decode(torch, ctx, q, kn, vn, w.tau, w.budget, out, W0, T1)
        if name == "every_step":
            ctx.set_profiling(True)
            ctx.profile(reset=True)
            for t in range(W0 + T1, W0 + T1 + T2):
                flush.fill_(float(t))
                ctx.decode_step(0, q[t], kn[t], vn[t], w.tau, w.budget, out[t])
            kern, ctr = ctx.profile(reset=True)
            n_sel, ms_sel = kern["lkv_select"]
            sec = ms_sel / n_sel / 1e3
            region = ctr["score_units"] / n_sel           # region tokens per launch
            cand = min(2560, region / (w.batch * w.n_kv_heads)) * w.batch * w.n_kv_heads
            alg = region * 16 + cand * 128
            res["select_us"] = sec * 1e6
            res["select_roofline"] = {"bound": "hbm", "achieved": alg / sec / 1e9, "unit": "GB/s",
                                      "alg_bytes_per_launch": alg,
                                      "note": "bucket bytes of every region token + codes and scales "
                                              "of every candidate"}
            res["single_step_us"] = {k: round(v[1] / v[0] * 1e3, 2) for k, v in kern.items() if v[0]}
        ctx.close()
    return res


def async_build_probe(torch):
    """Index build pipelined behind a prefill stand-in: 4 layers of the
    32K-input shape (8 KV heads x 32768 keys, C = 2048, 20 Lloyd rounds).
    The stand-in for a layer's prefill forward is a chain of cuBLAS bf16
    GEMMs [32768 x 4096] x [4096 x 4096] with the FLOPs of one Qwen3-8B-shaped
    layer at 32K tokens (projections and MLP 2*N*193M, causal attention
    2*N^2*d*H: 21.4 TFLOP, 19 GEMMs). Timed alone, the builds alone, then the
    prefill with layer l's build (lkv_build_index_async on the context's own
    stream) waiting for layer l's event: hidden fraction = 1 - (overlapped -
    prefill) / builds."""
    import synth
    import cluster_indexed_kv_gb300 as lkv
    NL = 4
    w = synth.WORKLOADS["long_in"].replace(n_layers=NL)
    KV = [synth.prefill(w, l, "cuda") for l in range(NL)]
    side = torch.cuda.Stream()
    ctx = lkv.Context(batch=1, n_layers=NL, n_kv_heads=w.n_kv_heads, group=w.group,
                      dtype=w.torch_dtype, local_buf=w.local_buf, max_clusters=w.n_clusters,
                      max_prefill=w.n_prefill, max_steps=w.n_steps, max_budget=w.budget, stream=side)
    x0 = torch.randn(w.n_prefill, 4096, device="cuda", dtype=torch.bfloat16)
    wm = torch.randn(4096, 4096, device="cuda", dtype=torch.bfloat16) / 64.0
    n_gemm = 19
    main = torch.cuda.current_stream()

    def prefill_layer(x):
        for _ in range(n_gemm):
            x = x @ wm
        return x

    def timed(fn):
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        fn()
        main.wait_stream(side)
        b.record(main)
        b.synchronize()
        return a.elapsed_time(b)

    def pre_only():
        x = x0
        for _ in range(NL):
            x = prefill_layer(x)

    def build_only():
        with torch.cuda.stream(side):
            side.wait_stream(main)
            for l in range(NL):
                ctx.build_index(l, KV[l][0], KV[l][1], w.n_clusters, w.iters, 1 + l)

    def overlapped():
        x = x0
        for l in range(NL):
            x = prefill_layer(x)
            ev = torch.cuda.Event()
            ev.record(main)
            ctx.build_index_async(l, KV[l][0], KV[l][1], w.n_clusters, w.iters, 1 + l, ready=ev)

    for fn in (pre_only, build_only, overlapped):
        timed(fn)  # warm-up
    res = {}
    for name, fn in (("prefill_ms", pre_only), ("build_ms", build_only), ("overlapped_ms", overlapped)):
        res[name] = sorted(timed(fn) for _ in range(3))[1]
    ctx.close()
    hidden = 1.0 - (res["overlapped_ms"] - res["prefill_ms"]) / res["build_ms"]
    return {"workload": "4 layers x (1 sequence, 8 KV heads, 32768 keys, C=2048, 20 rounds)",
            **res, "hidden_fraction": hidden,
            "prefill_slowdown": res["overlapped_ms"] / res["prefill_ms"] - 1.0,
            "prefill_standin": f"{n_gemm} cuBLAS bf16 GEMMs [32768x4096]x[4096x4096] per layer",
            "note": "median of 3; the pages report TTFT +3.5% over FullCache with their overlap "
                    "(another model, GPU and prefill; context only)"}


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """The oracle timed as it stands on the host cores, same metric and
    workload; each step is a bounded sample (one (sequence, KV head))."""
    import numpy as np
    import torch
    import oracle
    import synth
    w = workload(args)
    if rank != 0:
        return None
    n_steps = 32
    K, V = synth.prefill(w, 0, "cpu", seqs=[0], heads=[0])
    q, kn, vn, _ = synth.decode_inputs(w, "cpu", n_steps=n_steps, seqs=[0])
    # the sampled head's index, built by the oracle itself (one Lloyd round)
    km = oracle.kmeans(synth.to_oracle(K[0, 0]), w.n_clusters, 1, 1)
    idx = {"assign": km["assign"], "centroids": km["cent"]}
    Kf = torch.zeros(1, w.n_kv_heads, w.n_prefill, 128, dtype=K.dtype)
    Vf = torch.zeros_like(Kf)
    Kf[0, 0], Vf[0, 0] = K[0, 0], V[0, 0]
    for _ in range(args.warmup):
        oracle_decode_sample(Kf[0], Vf[0], idx, q, kn, vn, w, 4)
    per = [oracle_decode_sample(Kf[0], Vf[0], idx, q, kn, vn, w, n_steps) for _ in range(args.steps)]
    value = 1.0 / (float(np.mean(per)) * w.batch * w.n_kv_heads)
    sample = (f"single-threaded C oracle: 1 (sequence, KV head) x {n_steps} decode steps per step "
              f"of the full-size workload, index from one oracle Lloyd round; scaled by "
              f"B x H_kv = {w.batch * w.n_kv_heads}")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": float(np.mean(per)) * w.batch * w.n_kv_heads * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w, world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "host_nproc": host_cpu()[0], "host_cpu": host_cpu()[1],
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if world > 1:
        import torch
        import torch.distributed as td
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        td.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            res = run_reference(args, rank, world)
        else:
            res = run_ours(args, rank, world, local)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            import torch.distributed as td
            td.destroy_process_group()


if __name__ == "__main__":
    main()
