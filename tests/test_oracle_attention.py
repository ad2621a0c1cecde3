"""Pins for the oracle's exact attention, merge and APA emulation (CPU only).

Independent references: PyTorch's scaled_dot_product_attention in float64,
the merge identity of the APA blog ("The merge that makes it exact"),
special cases that reduce APA to exact attention, the cold-verdict safety
invariant ("Cold verdicts are safe"), the tile order ("Tile order") and the
frame collapse of APA 0.2.0 ("The bug: a sink that drowned the tail").
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mixed_precision_attention_gb300 import synth


def _sdpa_reference(q, k, v, causal):
    qf = torch.from_numpy(synth.bf16_bits_to_f32(q).astype(np.float64))
    kf = torch.from_numpy(synth.bf16_bits_to_f32(k).astype(np.float64))
    vf = torch.from_numpy(synth.bf16_bits_to_f32(v).astype(np.float64))
    G = qf.shape[1] // kf.shape[1]
    kf, vf = kf.repeat_interleave(G, 1), vf.repeat_interleave(G, 1)
    Nq, Nkv, d = qf.shape[2], kf.shape[2], qf.shape[3]
    mask = None
    if causal:  # tail-aligned: query row i sees keys j <= i + Nkv - Nq
        i = torch.arange(Nq)[:, None]
        j = torch.arange(Nkv)[None, :]
        mask = j <= i + (Nkv - Nq)
    out = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, attn_mask=mask)
    s = qf @ kf.transpose(-1, -2) / math.sqrt(d)
    if mask is not None:
        s = s.masked_fill(~mask, float("-inf"))
    return out.numpy(), torch.logsumexp(s, -1).numpy()


@pytest.mark.parametrize("shape", [
    dict(B=1, Hq=2, Hkv=1, Nq=128, Nkv=512, d=64, causal=True),
    dict(B=2, Hq=6, Hkv=2, Nq=37, Nkv=101, d=64, causal=True),
    dict(B=1, Hq=4, Hkv=4, Nq=20, Nkv=70, d=128, causal=False),
])
def test_exact_matches_torch_sdpa(shape):
    causal = shape.pop("causal")
    w = synth.small(causal=causal, n_outliers=2, **shape)
    q, k, v = synth.generate(w)
    out, lse = oracle.exact(q, k, v, causal=causal)
    ref, ref_lse = _sdpa_reference(q, k, v, causal)
    assert np.max(np.abs(out - ref)) < 1e-12
    assert np.max(np.abs(lse - ref_lse)) < 1e-11


def test_exact_row_subset():
    w = synth.small(B=1, Hq=4, Hkv=2, Nq=50, Nkv=300, d=64)
    q, k, v = synth.generate(w)
    full, full_lse = oracle.exact(q, k, v)
    rows = np.array([[0, 3, 49], [0, 0, 0], [0, 2, 17]])
    part, part_lse = oracle.exact(q, k, v, rows=rows)
    for b, h, i in rows:
        assert np.array_equal(part[b, h, i], full[b, h, i]) and part_lse[b, h, i] == full_lse[b, h, i]
    assert np.isnan(part[0, 1, 5]).all()


def _state(s, V):
    """(m, l, o) of a set of keys by the plain definition, log2 units."""
    if len(s) == 0:
        return -np.inf, 0.0, np.zeros(V.shape[1])
    m = s.max()
    p = np.exp2(s - m)
    return m, p.sum(), p @ V


def test_merge_identity_disjoint_key_sets():
    rng = np.random.default_rng(4)
    for trial in range(50):
        n, d = int(rng.integers(2, 300)), 16
        s = rng.standard_normal(n) * rng.uniform(0.1, 30)
        V = rng.standard_normal((n, d))
        full_m, full_l, full_o = _state(s, V)
        ref = full_o / full_l
        sel = rng.random(n) < rng.uniform(0, 1)
        a, b = _state(s[sel], V[sel]), _state(s[~sel], V[~sel])
        out, lg = oracle.merge(*a, *b)
        assert np.max(np.abs(out - ref)) <= 1e-12 * max(1.0, np.abs(ref).max())
        assert abs(lg - (full_m + math.log2(full_l))) < 1e-12 * max(1.0, abs(full_m))
    # an empty state is the identity
    s = rng.standard_normal(10)
    V = rng.standard_normal((10, 4))
    st = _state(s, V)
    out, _ = oracle.merge(*st, -np.inf, 0.0, np.zeros(4))
    assert np.allclose(out, st[2] / st[1], rtol=0, atol=1e-15)


SHAPES = [
    dict(B=1, Hq=2, Hkv=1, Nq=128, Nkv=512, d=64, causal=True),     # tiny
    dict(B=1, Hq=3, Hkv=1, Nq=45, Nkv=1000, d=64, causal=True),     # G=3, ragged tail, partial last group
    dict(B=2, Hq=4, Hkv=2, Nq=24, Nkv=300, d=128, causal=False),    # non-causal, ragged
    dict(B=1, Hq=2, Hkv=1, Nq=64, Nkv=4096, d=64, causal=True),     # many tiles: cold tiles exist
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("eps", [0.0, 0.005, 0.05, np.inf])
def test_apa_without_quantization_is_exact(shape, eps):
    """With no operand quantized, every tile is exact in one of the two passes, so
    the merged result is exact attention whatever the hot/cold split: this pins
    the frame bookkeeping (lazy max, cold frame, rescales), the tile order
    covering every tile once, the merge and the centring constant in the LSE."""
    sh = dict(shape)
    causal = sh.pop("causal")
    w = synth.small(causal=causal, n_outliers=2, sink_gain=8.0, **sh)
    q, k, v = synth.generate(w)
    ex, ex_lse = oracle.exact(q, k, v, causal=causal)
    r = oracle.apa(q, k, v, causal=causal, eps=eps, quant=0)
    assert np.max(np.abs(r["out"] - ex)) < 1e-12
    assert np.max(np.abs(r["lse"] - ex_lse)) < 1e-11


@pytest.mark.parametrize("shape", SHAPES)
def test_apa_eps0_is_exact(shape):
    sh = dict(shape)
    causal = sh.pop("causal")
    w = synth.small(causal=causal, n_outliers=2, **sh)
    q, k, v = synth.generate(w)
    ex, ex_lse = oracle.exact(q, k, v, causal=causal)
    r = oracle.apa(q, k, v, causal=causal, eps=0.0)
    assert np.max(np.abs(r["out"] - ex)) < 1e-12
    assert np.max(np.abs(r["lse"] - ex_lse)) < 1e-11


def test_apa_single_tile_is_exact():
    # Nkv <= 64: one tile, judged against an empty running sum, so always hot
    w = synth.small(B=1, Hq=4, Hkv=2, Nq=40, Nkv=64, d=64, n_outliers=2)
    q, k, v = synth.generate(w)
    ex, _ = oracle.exact(q, k, v)
    for eps in (1e-4, 0.005, 0.5, 1e6):
        r = oracle.apa(q, k, v, eps=eps)
        assert np.max(np.abs(r["out"] - ex)) < 1e-12
        assert np.all(r["hot_mask"] == 1)


def _hot_bits(mask, T):
    bits = np.unpackbits(mask.view(np.uint8), bitorder="little").reshape(mask.shape[:-1] + (-1,))
    return bits[..., :T].astype(bool)


def _visible_tiles(Hq, Hkv, Nq, Nkv, causal, grp):
    rows = oracle.group_rows(Hq, Hkv, Nq, 0, 0, grp)
    last = max(p + Nkv - Nq for _, _, p in rows) if causal else Nkv - 1
    return last // 64


@pytest.mark.parametrize("eps", [0.001, 0.005, 0.02])
def test_hot_test_invariants(eps):
    """Cold verdicts stay cold against the final sum; lambda counts every tile;
    tile 0 is always hot; verdicts follow the order 0, diagonal, ..., 1."""
    Hq, Hkv, Nq, Nkv, d = 2, 1, 64, 4096, 64
    w = synth.small(B=1, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, d=d, sink_gain=4.0, n_outliers=2)
    q, k, v = synth.generate(w)
    r = oracle.apa(q, k, v, eps=eps, diag=True)
    T = Nkv // 64
    hot = _hot_bits(r["hot_mask"][0, 0], T)
    ell, lam = r["ell"], r["lam"]
    n_cold = 0
    for grp in range(hot.shape[0]):
        assert hot[grp, 0]  # tile 0 judged first, against lambda = 0
        tmax = _visible_tiles(Hq, Hkv, Nq, Nkv, True, grp)
        order = [0] + list(range(tmax, 0, -1))
        assert not hot[grp, tmax + 1:].any()
        for rr in range(16):
            e = ell[grp, rr]
            seen = ~np.isnan(e)
            # lambda is the running sum over all tiles seen, hot ones included
            assert abs(lam[grp, rr] - e[seen].sum()) <= 1e-9 * lam[grp, rr]
            # cold verdicts are never revoked by later tiles
            cold = seen & ~hot[grp]
            n_cold += cold.sum()
            assert np.all(e[cold] <= eps * lam[grp, rr] * (1 + 1e-9))
        # each verdict in visiting order: hot iff some row's tile sum exceeds eps times
        # the sum of the tiles judged before it (all in the row's final frame)
        before = np.zeros(16)
        for t in order:
            e = ell[grp, :, t]
            vis = ~np.isnan(e)
            ratio = np.where(vis, e, 0.0)
            thr = eps * before
            if t == 0:
                expect = True
            else:
                margin = np.abs(ratio - thr) <= 1e-9 * np.maximum(thr, 1e-300)
                if np.any(margin & vis):
                    continue  # too close to the threshold to call in FP64
                expect = bool(np.any(vis & (ratio > thr)))
            assert hot[grp, t] == expect, (grp, t)
            before += ratio
    assert n_cold > 0


def test_apa_accuracy_against_exact():
    # the long middle goes to FP4, yet the merged output stays close to exact
    # (256 tiles: the hot share shrinks as the context grows)
    w = synth.small(B=1, Hq=2, Hkv=1, Nq=32, Nkv=16384, d=128, sink_gain=4.0, n_outliers=4)
    q, k, v = synth.generate(w)
    ex, _ = oracle.exact(q, k, v)
    r = oracle.apa(q, k, v, eps=0.005)
    cos = (ex * r["out"]).sum() / np.linalg.norm(ex) / np.linalg.norm(r["out"])
    hot_frac = _hot_bits(r["hot_mask"][0, 0], 256).mean()
    assert cos > 0.999 and hot_frac < 0.3
    allfp4 = oracle.apa(q, k, v, eps=np.inf)
    assert not allfp4["hot_mask"].any()
    cos4 = (ex * allfp4["out"]).sum() / np.linalg.norm(ex) / np.linalg.norm(allfp4["out"])
    assert 0.8 < cos4 < cos


def _sink_row_case():
    """One 16-row group whose rows see a dominant sink key and a thin, coherent tail.

    Sink: log2 score ~15 above the tail; the tail holds ~8 % of the mass spread
    over 47 tiles, and its values point against the sink's, so dropping it
    changes the output norm (the situation of the blog's worst pair)."""
    d, Nq, Nkv = 64, 16, 48 * 64
    rng = np.random.default_rng(5)
    q = np.zeros((1, 1, Nq, d), np.float32)
    q[..., 0] = 8.0
    q[..., 1:] = 0.01 * rng.standard_normal((Nq, d - 1))
    k = np.zeros((1, 1, Nkv, d), np.float32)
    k[0, 0, :, 0] = 0.05 * rng.standard_normal(Nkv)
    k[0, 0, :, 1:] = rng.standard_normal((Nkv, d - 1))
    k[0, 0, 0, 0] = 15.0 / math.log2(math.e) * math.sqrt(d) / 8.0
    v = 0.3 * rng.standard_normal((1, 1, Nkv, d)).astype(np.float32)
    v[0, 0, :, 0] -= 5.0
    v[0, 0, 0, 0] = 10.0
    b = synth.f32_to_bf16_bits
    return b(q), b(k), b(v)


def test_offset0_collapse_and_cold_frame_fix():
    """With the cold-frame offset at 0 (APA 0.2.0) the sink sets the frame and the
    cold tail rounds to zero: the output norm equals the hot part alone.  With
    offset 32 (0.3.0) the tail survives and the output is close to exact."""
    q, k, v = _sink_row_case()
    eps = 0.01
    ex, _ = oracle.exact(q, k, v)
    r0 = oracle.apa(q, k, v, eps=eps, cold_offset=0.0)
    r32 = oracle.apa(q, k, v, eps=eps, cold_offset=32.0)
    hot = _hot_bits(r32["hot_mask"][0, 0], 48)[0]
    assert hot[0] and hot.sum() <= 2
    assert np.array_equal(r0["hot_mask"], r32["hot_mask"])
    # the hot part alone: exact softmax over the hot tiles' keys only
    keys = np.concatenate([np.arange(t * 64, t * 64 + 64) for t in np.nonzero(hot)[0]])
    kf = synth.bf16_bits_to_f32(k[0, 0]).astype(np.float64)
    vf = synth.bf16_bits_to_f32(v[0, 0]).astype(np.float64)
    qf = synth.bf16_bits_to_f32(q[0, 0]).astype(np.float64)
    for i in range(16):
        nvis = i + 48 * 64 - 16 + 1
        kk = keys[keys < nvis]
        s = qf[i] @ kf[kk].T / 8.0
        p = np.exp(s - s.max())
        hot_part = p @ vf[kk] / p.sum()
        n0, nh, nex = np.linalg.norm(r0["out"][0, 0, i]), np.linalg.norm(hot_part), np.linalg.norm(ex[0, 0, i])
        assert abs(n0 - nh) < 1e-3 * nh  # collapse: output == hot part
        assert abs(nex - nh) > 0.1 * nex  # ... which is far from exact
        err32 = np.linalg.norm(r32["out"][0, 0, i] - ex[0, 0, i]) / nex
        assert err32 < 0.02


def test_apa_deterministic():
    w = synth.small(B=1, Hq=2, Hkv=1, Nq=64, Nkv=2048, d=64)
    q, k, v = synth.generate(w)
    a = oracle.apa(q, k, v, eps=0.005)
    b = oracle.apa(q, k, v, eps=0.005)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["hot_mask"], b["hot_mask"])


def test_apa_group_subset_matches_full():
    w = synth.small(B=2, Hq=4, Hkv=2, Nq=40, Nkv=700, d=64)
    q, k, v = synth.generate(w)
    full = oracle.apa(q, k, v, eps=0.005)
    units = np.array([[1, 1, 4], [0, 0, 0], [1, 0, 2]])
    part = oracle.apa(q, k, v, eps=0.005, units=units)
    for b, h, g in units:
        for (bb, hq, pos) in oracle.group_rows(4, 2, 40, b, h, g):
            assert np.array_equal(part["out"][bb, hq, pos], full["out"][bb, hq, pos])
        assert np.array_equal(part["hot_mask"][b, h, g], full["hot_mask"][b, h, g])


def test_eps0_marks_every_visible_tile_hot_even_when_fp4_mass_underflows():
    """eps = 0 is the all-exact run: a tile whose FP4 row sums round to zero (its
    scores sit far below the frame) is still hot and is computed exactly."""
    q, k, v = _sink_row_case()
    kf = synth.bf16_bits_to_f32(k).copy()
    kf[0, 0, 5 * 64:6 * 64, 0] = -60.0  # tile 5: ~70 log2 units below the sink
    k2 = synth.f32_to_bf16_bits(kf)
    probe = oracle.apa(q, k2, v, eps=1e-12, diag=True)
    assert np.all(probe["ell"][0, :, 5] == 0.0)  # the FP4 mass of tile 5 underflows
    r = oracle.apa(q, k2, v, eps=0.0)
    assert _hot_bits(r["hot_mask"][0, 0], 48)[0].all()
    ex, _ = oracle.exact(q, k2, v)
    assert np.max(np.abs(r["out"] - ex)) < 1e-12
