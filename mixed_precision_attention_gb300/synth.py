"""Seeded synthetic Q/K/V for causal GQA prefill attention.

This module only draws inputs; it holds none of the attention arithmetic, so
both the CUDA path and the CPU oracle can be fed from it.

The recipe stands in for the Llama-3.2-3B Q/K/V dumps that the APA blog
("APA: sloppy attention, exact where it counts", rfriedmann.de) measures on,
which are not available.  It reproduces the structure those dumps have and the
method depends on:

* a shared per-KV-head direction ``u`` so that queries and keys of one head are
  correlated (Q = u + 0.5 n, K = u + 0.5 n');
* a few outlier channels (x8 on Q and K, before RoPE), the channel spread that
  the blog's "Mean-centred K" trick is about;
* rotary position embedding (half split, theta = 500000, Llama-3 style), with
  keys at positions 0..Nkv-1 and queries tail-aligned at Nkv-Nq .. Nkv-1;
* an attention sink: key row 0 scaled by ``sink_gain`` after RoPE, so tile 0
  carries a large share of every row's softmax mass (blog, "Why this can work
  at all");
* V ~ N(0, 1).

Normals are drawn as float32 (numpy ``Generator(PCG64(seed + b))`` per
sequence b, in the order u [Hkv, d]; outlier channels per KV head; nQ per query
head; nK per KV head; V per KV head).  RoPE angles and their cos / sin are
computed in float64 and rounded to float32; the rest is float32 arithmetic,
rounded to bfloat16 with round-to-nearest-even.
"""
from __future__ import annotations

import hashlib
import os
from dataclasses import dataclass, field

import numpy as np

ROPE_THETA = 500000.0


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, generator knobs and the hot-test eps."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nkv: int
    d: int
    causal: bool = True
    eps: float = 0.005
    seed: int = 0
    sink_gains: tuple = (4.0,)
    n_outliers: int = 4
    outlier_gain: float = 8.0
    eps_sweep: tuple = field(default=())

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def visible_pairs(self) -> int:
        """(query row, key) pairs that causal tail-aligned masking leaves visible."""
        if not self.causal:
            return self.B * self.Hq * self.Nq * self.Nkv
        off = self.Nkv - self.Nq
        per_head = self.Nq * (off + 1) + self.Nq * (self.Nq - 1) // 2
        return self.B * self.Hq * per_head

    @property
    def flops_exact(self) -> float:
        """Algorithmic flops of exact attention: 2d for QK^T and 2d for PV per visible pair."""
        return 4.0 * self.d * self.visible_pairs


# The five workloads: a tiny case, the 2048-query x 122880-key Llama-3.2-3B
# layer chunk, a full 8k self-attention prefill with an eps sweep, a batched
# 32k prefill and a short-query / long-KV case with head dim 256.
WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hq=2, Hkv=1, Nq=128, Nkv=512, d=64,
                     sink_gains=(4.0,), n_outliers=0),
    "llama3b_2048x122880": Workload("llama3b_2048x122880", B=1, Hq=24, Hkv=8,
                                    Nq=2048, Nkv=122880, d=128),
    "prefill_8k": Workload("prefill_8k", B=1, Hq=32, Hkv=8, Nq=8192, Nkv=8192,
                           d=128, eps_sweep=(0.0, 0.001, 0.005, 0.02, float("inf"))),
    "batched_32k": Workload("batched_32k", B=4, Hq=32, Hkv=8, Nq=32768,
                            Nkv=32768, d=128, sink_gains=(2.0, 4.0, 8.0, 16.0)),
    "shortq_131k_d256": Workload("shortq_131k_d256", B=2, Hq=32, Hkv=8, Nq=128,
                                 Nkv=131072, d=256, sink_gains=(8.0,)),
}


def f32_to_bf16_bits(x: np.ndarray, out: np.ndarray | None = None) -> np.ndarray:
    """Round finite float32 values to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = u >> np.uint32(16)
    r &= np.uint32(1)
    r += u
    r += np.uint32(0x7FFF)
    r >>= np.uint32(16)
    if out is None:
        return r.astype(np.uint16)
    out[...] = r
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rope_tables(n_pos: int, d: int):
    half = d // 2
    inv_freq = ROPE_THETA ** (-(2.0 * np.arange(half, dtype=np.float64)) / d)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Half-split rotary embedding, float32."""
    half = x.shape[-1] // 2
    out = np.empty_like(x)
    x1, x2 = x[..., :half], x[..., half:]
    np.multiply(x1, cos, out=out[..., :half])
    out[..., :half] -= x2 * sin
    np.multiply(x2, cos, out=out[..., half:])
    out[..., half:] += x1 * sin
    return out


def generate(w: Workload, seed: int | None = None):
    """Returns (q, k, v) as uint16 bfloat16 bit arrays in BHSD layout.

    q: [B, Hq, Nq, d]; k, v: [B, Hkv, Nkv, d].
    """
    base = w.seed if seed is None else seed
    B, Hq, Hkv, Nq, Nkv, d, G = w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.d, w.G
    assert Hq % Hkv == 0 and Nkv >= Nq and d % 2 == 0
    off = Nkv - Nq
    cos, sin = _rope_tables(Nkv, d)
    q = np.empty((B, Hq, Nq, d), dtype=np.uint16)
    k = np.empty((B, Hkv, Nkv, d), dtype=np.uint16)
    v = np.empty((B, Hkv, Nkv, d), dtype=np.uint16)
    from concurrent.futures import ThreadPoolExecutor
    pool = ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1))
    jobs = []

    def finish_q(dst, x, c, si):
        f32_to_bf16_bits(_rope(x, c, si), out=dst)

    def finish_k(dst, x, gain):
        y = _rope(x, cos, sin)
        y[0] *= np.float32(gain)
        f32_to_bf16_bits(y, out=dst)

    for b in range(B):
        rng = np.random.Generator(np.random.PCG64(base + b))
        gain = w.sink_gains[b % len(w.sink_gains)]
        f32 = np.float32
        u = rng.standard_normal((Hkv, d), dtype=f32)
        outl = [np.sort(rng.choice(d, size=w.n_outliers, replace=False))
                if w.n_outliers else np.zeros(0, dtype=np.int64) for _ in range(Hkv)]
        for h in range(Hq):
            hk = h // G
            x = rng.standard_normal((Nq, d), dtype=f32)
            x *= f32(0.5)
            x += u[hk][None, :]
            x[:, outl[hk]] *= f32(w.outlier_gain)
            jobs.append(pool.submit(finish_q, q[b, h], x, cos[off:off + Nq], sin[off:off + Nq]))
        for h in range(Hkv):
            x = rng.standard_normal((Nkv, d), dtype=f32)
            x *= f32(0.5)
            x += u[h][None, :]
            x[:, outl[h]] *= f32(w.outlier_gain)
            jobs.append(pool.submit(finish_k, k[b, h], x, gain))
        for h in range(Hkv):
            jobs.append(pool.submit(f32_to_bf16_bits, rng.standard_normal((Nkv, d), dtype=f32), v[b, h]))
        # bound the memory held by pending float32 copies
        while sum(not j.done() for j in jobs) > 16:
            jobs[[j.done() for j in jobs].index(False)].result()
    for j in jobs:
        j.result()
    pool.shutdown()
    return q, k, v


def small(B=1, Hq=2, Hkv=1, Nq=128, Nkv=512, d=64, causal=True, eps=0.005,
          seed=0, sink_gain=4.0, n_outliers=0, name="small") -> Workload:
    """A small workload of arbitrary shape with the same generator."""
    return Workload(name, B=B, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, d=d, causal=causal,
                    eps=eps, seed=seed, sink_gains=(sink_gain,), n_outliers=n_outliers)


def sha256(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def to_torch_bf16(a: np.ndarray, device=None):
    """Views uint16 bfloat16 bits as a torch.bfloat16 tensor (copied to ``device``)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t
