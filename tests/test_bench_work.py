"""bench.py's algorithmic work counts (the numerators of its roofline figures)
against a brute-force count over every (row, key) pair of a tiny layer: visible
pairs per (16-row group, 64-key tile), hot and cold pairs, the flops of both
passes, and the per-block union of hot tiles that pass 2 walks."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mixed_precision_attention_gb300 import synth  # noqa: E402


def _brute(w, hot):
    """hot: bool [B, Hkv, ngroups, T].  Counts by walking every packed row and key."""
    G, R, T, off = w.G, w.G * w.Nq, (w.Nkv + 63) // 64, w.Nkv - w.Nq
    pairs = hot_pairs = 0
    union = set()
    vis_blocks = set()
    for b in range(w.B):
        for h in range(w.Hkv):
            for p in range(R):
                last = p // G + off if w.causal else w.Nkv - 1
                for j in range(min(last + 1, w.Nkv)):
                    t = j // 64
                    pairs += 1
                    vis_blocks.add((b, h, p // 128, t))
                    if hot[b, h, p // 16, t]:
                        hot_pairs += 1
                        union.add((b, h, p // 128, t))
    return pairs, hot_pairs, len(union), len(vis_blocks)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("shape", [dict(B=1, Hq=6, Hkv=2, Nq=50, Nkv=300, d=64),
                                   dict(B=2, Hq=4, Hkv=1, Nq=100, Nkv=130, d=128)])
def test_work_counts_match_brute_force(shape, causal):
    w = synth.small(causal=causal, **shape)
    T = (w.Nkv + 63) // 64
    ng = (w.G * w.Nq + 15) // 16
    rng = np.random.default_rng(5)
    hot = rng.random((w.B, w.Hkv, ng, T)) < 0.3
    words = (T + 31) // 32
    mask = np.zeros((w.B, w.Hkv, ng, words), np.uint32)
    for t in range(T):
        mask[..., t // 32] |= hot[..., t].astype(np.uint32) << np.uint32(t % 32)
    got = bench.algorithmic(w, mask)
    pairs, hot_pairs, union, vis_blocks = _brute(w, hot)
    assert got["pairs"] == pairs and got["hot_pairs"] == hot_pairs
    assert got["cold_pairs"] == pairs - hot_pairs
    # QK^T (2d) and the ones product of the row sums (N = 16: 32) on every pair, PV on cold ones
    assert got["F1"] == pairs * (2 * w.d + 32) + (pairs - hot_pairs) * 2 * w.d
    assert got["F2"] == hot_pairs * 4 * w.d
    assert got["block_tiles_hot"] == union and got["block_tiles_vis"] == vis_blocks


def test_all_hot_and_none_hot():
    w = synth.small(B=1, Hq=3, Hkv=1, Nq=70, Nkv=500, d=64)
    T, ng = (w.Nkv + 63) // 64, (w.G * w.Nq + 15) // 16
    full = np.full((1, 1, ng, (T + 31) // 32), 0xFFFFFFFF, np.uint32)
    got = bench.algorithmic(w, full)
    assert got["hot_pairs"] == got["pairs"] and got["block_tiles_hot"] == got["block_tiles_vis"]
    got = bench.algorithmic(w, np.zeros_like(full))
    assert got["hot_pairs"] == 0 and got["F2"] == 0 and got["block_tiles_hot"] == 0


def test_stage_bytes_follow_where_the_kv_quantizer_runs():
    # the K/V quantizer's traffic counts in the pass-1 stage when it runs inside
    # that launch, in the quantizer stage otherwise; the total is the same
    w = synth.WORKLOADS["llama3b_2048x122880"]
    assert bench.pass1_hosts_kv_quantizer(w, 152)   # 128 pass-1 CTAs, 24 SMs spare
    assert not bench.pass1_hosts_kv_quantizer(synth.WORKLOADS["batched_32k"], 152)
    assert bench.pass1_hosts_kv_quantizer(synth.WORKLOADS["shortq_131k_d256"], 152)  # 64 one-block CTAs
    q_in, p1_in = bench.stage_bytes(w, True)
    q_out, p1_out = bench.stage_bytes(w, False)
    assert q_in + p1_in == q_out + p1_out and q_out > q_in and p1_in > p1_out
    kv = w.B * w.Hkv * w.Nkv * w.d
    # statistics read K and V once (bf16); the quantizer reads them again and writes
    # 0.5625 B of codes and scales per element and the 2-B FP16 copy of V
    assert q_out - q_in == 2 * kv * 2 + 2 * kv * 0.5625 + kv * 2
