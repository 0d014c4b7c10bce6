"""Pipelined index build (lkv_build_index_async): the K-means of layer l runs
on the context's own stream beside a producer stream that is still working
("LouisKV ... Long Input-Output Sequences", 关键设计 2: clustering and offload
overlap the prefill forward). The index must be bit-identical to a serial
build, the build must not start before the producer's ready event (the key
buffers hold zeros until then) and the producer may overwrite the buffers
once the done event has passed."""
import numpy as np
import pytest
import torch

import synth
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _busy(x, w, n):
    for _ in range(n):
        x = torch.tanh(x @ w)
    return x


@pytest.mark.parametrize("offload", [False, True])
def test_async_build_waits_and_matches_serial(offload):
    import cluster_indexed_kv_gb300 as lkv
    w = synth.WORKLOADS["long_in"].replace(batch=2, n_layers=3, n_kv_heads=2, n_prefill=3000,
                                           n_components=60, n_clusters=64, iters=4, n_steps=40,
                                           local_buf=16, budget=200, offload=offload)
    NL, T = w.n_layers, w.n_steps
    prod = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    kw = dict(batch=w.batch, n_layers=NL, n_kv_heads=w.n_kv_heads, group=w.group,
              dtype=w.torch_dtype, local_buf=w.local_buf, max_clusters=w.n_clusters,
              max_prefill=w.n_prefill, max_steps=T, max_budget=w.budget, offload=offload)
    ctx_a = lkv.Context(stream=side, **kw)
    ctx_s = lkv.Context(**kw)
    KV = [synth.prefill(w, l, "cuda") for l in range(NL)]
    bufK = [torch.zeros_like(K) for K, _ in KV]
    bufV = [torch.zeros_like(V) for _, V in KV]
    x = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16)
    wm = torch.randn(2048, 2048, device="cuda", dtype=torch.bfloat16) / 45.0
    done = [torch.cuda.Event() for _ in range(NL)]
    torch.cuda.synchronize()
    for l in range(NL):
        x = _busy(x, wm, 40)                       # the producer's layer l
        bufK[l].copy_(KV[l][0])
        bufV[l].copy_(KV[l][1])
        ready = torch.cuda.Event()
        ready.record(prod)
        ctx_a.build_index_async(l, bufK[l], bufV[l], w.n_clusters, w.iters, 7 + l, ready=ready,
                                done=done[l])
    for l in range(NL):                            # reuse the buffers once each build is done
        prod.wait_event(done[l])
        bufK[l].zero_()
        bufV[l].zero_()
    for l in range(NL):
        ctx_s.build_index(l, KV[l][0], KV[l][1], w.n_clusters, w.iters, 7 + l)
    for l in range(NL):
        for b in range(w.batch):
            for h in range(w.n_kv_heads):
                a = ctx_a.get_index(l, b, h, w.n_prefill)
                s = ctx_s.get_index(l, b, h, w.n_prefill)
                assert a["n_units"] == s["n_units"] == w.n_clusters
                for k in ("assign", "perm", "unit_len", "unit_row"):
                    assert np.array_equal(a[k], s[k]), (l, b, h, k)
                assert np.array_equal(a["centroids"].view(np.uint32), s["centroids"].view(np.uint32))
    # the pools hold the right rows: decoding from both gives the same outputs
    q, kn, vn, _ = synth.decode_inputs(w, "cuda", n_steps=T)
    outs = []
    for ctx in (ctx_a, ctx_s):
        out = torch.zeros(T, w.batch, NL, w.n_heads, 128, device="cuda")
        with torch.cuda.stream(ctx.stream):
            ctx.stream.wait_stream(prod)
            for t in range(T):
                ctx.decode_step(0, q[t], kn[t], vn[t], w.tau, w.budget, out[t], n_layers=NL)
        ctx.sync()
        outs.append(out.cpu().numpy())
    assert np.array_equal(outs[0], outs[1])
    ctx_a.close()
    ctx_s.close()
