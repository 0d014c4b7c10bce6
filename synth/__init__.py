"""Seeded synthetic workloads shaped like the LouisKV evaluation settings.

This module holds only input generation (no retrieval arithmetic); the CUDA
path and the oracle both consume the tensors it makes. Every tensor comes from
its own ``torch.Generator`` stream keyed by (workload seed, kind, sequence,
layer, head), so any slice can be regenerated alone. Values are drawn in fp32
and rounded to nearest-even bf16 for the bf16 workloads.

Recipe (stand-in for LongBench / reasoning sets / RULER, which are not used):
  * prefill keys: Gaussian mixture -- component means N(0,1)^d, each key picks
    a component uniformly and adds 0.3 * N(0,1)^d; values N(0,1)^d;
  * queries: per (layer, head) random walk q_t = sqrt(d) * normalize(q_{t-1}
    + 0.2 * N(0,1)^d); with probability ``jump_p`` per (sequence, step) -- one
    draw shared by all heads and layers -- q_t is a fresh N(0,1)^d draw;
  * new decode keys: N(0,1)^d, or (``new_key="query_dir"``) sqrt(d) *
    normalize(mean of the group's query heads) + 0.5 * N(0,1)^d; new values
    N(0,1)^d.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import torch

KIND_COMPONENTS, KIND_CHOICE, KIND_KNOISE, KIND_VALUES = 1, 2, 3, 4
KIND_Q0, KIND_QNOISE, KIND_QFRESH, KIND_JUMP = 5, 6, 7, 8
KIND_KNEW, KIND_VNEW = 9, 10


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_layers: int
    n_kv_heads: int
    group: int
    head_dim: int
    dtype: str               # "fp32" | "bf16"
    n_prefill: int           # N prefill tokens per (sequence, layer, kv head)
    n_components: int        # mixture components of the prefill keys
    n_clusters: int          # C
    iters: int               # Lloyd rounds
    n_steps: int             # T decode steps
    jump_p: float
    tau: float
    budget: int              # token budget per (sequence, layer, kv head)
    local_buf: int           # L local-buffer tokens
    new_key: str = "gauss"   # "gauss" | "query_dir"
    offload: bool = False    # prefill K/V pool in pinned host memory
    seed: int = 1

    @property
    def n_heads(self) -> int:
        return self.n_kv_heads * self.group

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five evaluation shapes (Qwen3-8B-like GQA heads: 8 KV heads x 4 query
# heads, head_dim 128) plus the 32K-input, batch-8 decode workload.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 4, 128, "fp32", 2048, 32, 32, 10, 64, 0.05,
                     0.7, 256, 128, seed=1),
    "long_in": Workload("long_in", 1, 1, 8, 4, 128, "bf16", 32768, 2048, 2048, 20,
                        256, 0.05, 0.7, 1024, 256, seed=2),
    "long_out": Workload("long_out", 8, 1, 8, 4, 128, "bf16", 2048, 128, 128, 20,
                         16384, 0.02, 0.7, 1024, 512, new_key="query_dir", seed=3),
    "offload": Workload("offload", 1, 36, 8, 4, 128, "bf16", 131072, 8192, 8192, 20,
                        512, 0.05, 0.7, 2048, 512, offload=True, seed=4),
    "sweep": Workload("sweep", 32, 1, 8, 4, 128, "bf16", 32768, 2048, 2048, 20, 8192,
                      0.03, 0.7, 1024, 512, seed=5),
    "b8_32k": Workload("b8_32k", 8, 1, 8, 4, 128, "bf16", 32768, 2048, 2048, 20, 8192,
                       0.03, 0.7, 1024, 512, seed=6),
}


def _stream(w: Workload, kind: int, seq: int, layer: int, head: int,
            device) -> torch.Generator:
    key = f"{w.seed}/{kind}/{seq}/{layer}/{head}".encode()
    s = int.from_bytes(hashlib.blake2b(key, digest_size=8).digest(), "little")
    g = torch.Generator(device=device)
    g.manual_seed(s & 0x7FFFFFFFFFFFFFFF)
    return g


def _normal(shape, gen, device):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)


def prefill(w: Workload, layer: int = 0, device="cpu", seqs=None, heads=None):
    """Prefill keys and values of one layer: [B, H_kv, N, d] in the workload
    dtype (``seqs`` / ``heads`` restrict to a subset, same values)."""
    seqs = range(w.batch) if seqs is None else seqs
    heads = range(w.n_kv_heads) if heads is None else heads
    N, d = w.n_prefill, w.head_dim
    K = torch.empty(len(seqs), len(heads), N, d, dtype=w.torch_dtype, device=device)
    V = torch.empty_like(K)
    for bi, b in enumerate(seqs):
        for hi, h in enumerate(heads):
            comps = _normal((w.n_components, d), _stream(w, KIND_COMPONENTS, b, layer, h, device), device)
            choice = torch.randint(0, w.n_components, (N,), device=device,
                                   generator=_stream(w, KIND_CHOICE, b, layer, h, device))
            noise = _normal((N, d), _stream(w, KIND_KNOISE, b, layer, h, device), device)
            K[bi, hi] = (comps[choice] + 0.3 * noise).to(w.torch_dtype)
            V[bi, hi] = _normal((N, d), _stream(w, KIND_VALUES, b, layer, h, device), device).to(w.torch_dtype)
    return K, V


def _normalize_sqrt_d(x: torch.Tensor, d: int) -> torch.Tensor:
    return math.sqrt(d) * x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def decode_inputs(w: Workload, device="cpu", n_steps: int | None = None,
                  seqs=None, layers=None):
    """Per-step decode inputs.

    Returns q [T, B, layers, H, d], k_new and v_new [T, B, layers, H_kv, d]
    in the workload dtype, and the jump mask [T, B] (bool).
    """
    T = w.n_steps if n_steps is None else n_steps
    seqs = range(w.batch) if seqs is None else seqs
    layers = range(w.n_layers) if layers is None else layers
    H, Hkv, G, d = w.n_heads, w.n_kv_heads, w.group, w.head_dim
    nb, nl = len(seqs), len(layers)
    q = torch.empty(T, nb, nl, H, d, dtype=w.torch_dtype, device=device)
    kn = torch.empty(T, nb, nl, Hkv, d, dtype=w.torch_dtype, device=device)
    vn = torch.empty_like(kn)
    jumps = torch.zeros(T, nb, dtype=torch.bool, device=device)
    for bi, b in enumerate(seqs):
        u = torch.rand(T, generator=_stream(w, KIND_JUMP, b, 0, 0, device), device=device)
        jumps[:, bi] = u < w.jump_p
        jumps[0, bi] = False
        for li, l in enumerate(layers):
            cur = _normal((H, d), _stream(w, KIND_Q0, b, l, 0, device), device)
            noise = _normal((T, H, d), _stream(w, KIND_QNOISE, b, l, 0, device), device)
            fresh = _normal((T, H, d), _stream(w, KIND_QFRESH, b, l, 0, device), device)
            walk = torch.empty(T, H, d, dtype=torch.float32, device=device)
            walk[0] = cur
            jb = jumps[:, bi].tolist()
            for t in range(1, T):
                cur = fresh[t] if jb[t] else _normalize_sqrt_d(cur + 0.2 * noise[t], d)
                walk[t] = cur
            q[:, bi, li] = walk.to(w.torch_dtype)
            knoise = _normal((T, Hkv, d), _stream(w, KIND_KNEW, b, l, 0, device), device)
            if w.new_key == "query_dir":
                gm = walk.view(T, Hkv, G, d).mean(dim=2)
                kn[:, bi, li] = (_normalize_sqrt_d(gm, d) + 0.5 * knoise).to(w.torch_dtype)
            else:
                kn[:, bi, li] = knoise.to(w.torch_dtype)
            vn[:, bi, li] = _normal((T, Hkv, d), _stream(w, KIND_VNEW, b, l, 0, device),
                                    device).to(w.torch_dtype)
    return q, kn, vn, jumps


def to_oracle(x: torch.Tensor):
    """numpy view for the oracle: bf16 as uint16 bit patterns, fp32 as is."""
    import numpy as np
    x = x.detach().contiguous().cpu()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    return x.numpy()
