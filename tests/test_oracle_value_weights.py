"""The oracle's value-norm-weighted hot test (the APA page, "Honest limits": the
plain test bounds a cold tile's share of the softmax mass, not its share of the
output, and a test weighted by value norm is proposed for rows where the two part).
Reading: w_t = (largest key value norm in tile t) / (mean key value norm of the
head); a tile is hot iff some row's l_t * w_t * 2^(m~ - m) exceeds eps * lambda.
Pinned against the definition recomputed here in numpy and against the verdicts
re-derived from the oracle's own tile sums."""
import numpy as np
import pytest

import oracle
from mixed_precision_attention_gb300 import synth

VW = oracle.QUANT_ALL | oracle.QUANT_VWEIGHT


def _weights_numpy(vh):
    """Same definition, written with numpy float32 steps: per-key norm, tile max, mean."""
    x = synth.bf16_bits_to_f32(vh).astype(np.float32)
    Nkv = x.shape[0]
    sq = x * x  # fp32 squares
    acc = np.zeros(Nkv, np.float32)
    for c in range(x.shape[1]):  # channel order
        acc = (acc + sq[:, c]).astype(np.float32)
    n = np.sqrt(acc).astype(np.float32)
    T = (Nkv + 63) // 64
    amax = np.array([n[t * 64:(t + 1) * 64].max() for t in range(T)], np.float32)
    nbar = np.float32(n.astype(np.float64).sum() / Nkv)
    if nbar == 0:
        return np.ones(T, np.float32)
    return (amax.astype(np.float64) / np.float64(nbar)).astype(np.float32)


def _hot_bits(mask, T):
    bits = np.unpackbits(mask.view(np.uint8), bitorder="little").reshape(mask.shape[:-1] + (-1,))
    return bits[..., :T].astype(bool)


def test_weights_match_the_definition():
    rng = np.random.default_rng(11)
    for Nkv, d in ((1000, 64), (4096, 128), (70, 96)):
        vf = rng.standard_normal((1, 1, Nkv, d)).astype(np.float32)
        vf[0, 0, rng.integers(0, Nkv, 9)] *= 30.0  # a few large-norm keys
        vh = synth.f32_to_bf16_bits(vf)
        w = oracle.value_weights(vh)[0, 0]
        ref = _weights_numpy(vh[0, 0])
        # the mean's summation order differs (tile then range vs flat): a few ulp
        np.testing.assert_allclose(w, ref, rtol=3e-6, atol=0)
        # closed form: a tile of the mean norm has weight 1; the largest tile is >= 1
        assert w.max() >= 1.0


def test_weights_closed_forms():
    # every key the same norm: every weight is exactly 1
    v = np.zeros((1, 1, 640, 64), np.float32)
    v[..., 0] = 3.0
    assert np.all(oracle.value_weights(synth.f32_to_bf16_bits(v)) == 1.0)
    # one tile of keys at norm 5, the rest at norm 1, all of 640 keys: mean = (64*5 + 576)/640
    v = np.zeros((1, 1, 640, 64), np.float32)
    v[..., 1] = 1.0
    v[0, 0, 128:192, 1] = 5.0
    w = oracle.value_weights(synth.f32_to_bf16_bits(v))[0, 0]
    nbar = (64 * 5 + 576) / 640
    np.testing.assert_allclose(w, np.where(np.arange(10) == 2, 5 / nbar, 1 / nbar), rtol=1e-7)
    # all-zero values: weights are 1 (no division by zero)
    assert np.all(oracle.value_weights(np.zeros((1, 1, 200, 64), np.uint16)) == 1.0)


@pytest.mark.parametrize("eps", [0.002, 0.02])
def test_weighted_verdicts_follow_the_weighted_test(eps):
    """Each verdict in visiting order: hot iff some row's tile sum times w_t exceeds
    eps times the sum of the tiles judged before it (the row's final frame)."""
    Hq, Hkv, Nq, Nkv, d = 2, 1, 64, 4096, 64
    w = synth.small(B=1, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, d=d, sink_gain=4.0, n_outliers=2, seed=7)
    q, k, v = synth.generate(w)
    vf = synth.bf16_bits_to_f32(v).copy()
    vf[0, 0, 20 * 64:21 * 64] *= 12.0  # one tile of large-norm values
    vf[0, 0, 40 * 64:41 * 64] *= 0.05  # one of small-norm values
    v = synth.f32_to_bf16_bits(vf)
    wt = oracle.value_weights(v)[0, 0].astype(np.float64)
    assert wt[20] > 5 and wt[40] < 0.2
    r = oracle.apa(q, k, v, eps=eps, quant=VW, diag=True)
    T = Nkv // 64
    hot = _hot_bits(r["hot_mask"][0, 0], T)
    ell = r["ell"]
    checked = 0
    for grp in range(hot.shape[0]):
        assert hot[grp, 0]
        seen_any = ~np.isnan(ell[grp]).all(0)
        tmax = int(np.nonzero(seen_any)[0].max())
        order = [0] + list(range(tmax, 0, -1))
        before = np.zeros(16)
        for t in order:
            e = ell[grp, :, t]
            vis = ~np.isnan(e)
            ratio = np.where(vis, e, 0.0)
            if t != 0:
                thr = eps * before
                lhs = ratio * wt[t]
                margin = np.abs(lhs - thr) <= 1e-9 * np.maximum(thr, 1e-300)
                if not np.any(margin & vis):
                    assert hot[grp, t] == bool(np.any(vis & (lhs > thr))), (grp, t)
                    checked += 1
            before += ratio
    assert checked > 50


def test_weighting_bounds_each_cold_tile_share_of_the_output():
    """What the weighting buys: under the plain test a cold tile's share of the
    softmax mass is at most eps, so its share of the output is at most eps times
    its largest value norm; under the weighted test the output share of every cold
    tile is at most eps times the head's mean value norm, whatever its own norm.
    Verdicts also move monotonically with the weight (the running sums do not
    depend on them): w >= 1 keeps every plain hot tile hot, w <= 1 every cold one cold."""
    Hq, Hkv, Nq, Nkv, d = 2, 1, 64, 4096, 64
    w = synth.small(B=1, Hq=Hq, Hkv=Hkv, Nq=Nq, Nkv=Nkv, d=d, sink_gain=4.0, n_outliers=2, seed=9)
    q, k, v = synth.generate(w)
    vf = synth.bf16_bits_to_f32(v).copy()
    vf[0, 0, 10 * 64:12 * 64] *= 40.0
    v = synth.f32_to_bf16_bits(vf)
    eps = 0.02
    # tile max and head mean of the key value norms, from the definition in FP64
    n = np.sqrt((synth.bf16_bits_to_f32(v[0, 0]).astype(np.float64) ** 2).sum(-1))
    a = n.reshape(-1, 64).max(-1)
    nbar = n.mean()
    wt = oracle.value_weights(v)[0, 0]
    np.testing.assert_allclose(wt, a / nbar, rtol=1e-6)
    a0 = oracle.apa(q, k, v, eps=eps, diag=True)
    a1 = oracle.apa(q, k, v, eps=eps, quant=VW, diag=True)
    h0, h1 = _hot_bits(a0["hot_mask"][0, 0], 64), _hot_bits(a1["hot_mask"][0, 0], 64)
    up, down = wt >= 1.0, wt <= 1.0
    assert np.all(h1[:, up] >= h0[:, up])
    assert np.all(h1[:, down] <= h0[:, down])
    assert h1[:, 10:12].sum() > h0[:, 10:12].sum()
    over_plain = 0
    for r, h in ((a0, h0), (a1, h1)):
        ell, lam = r["ell"], r["lam"]
        for grp in range(h.shape[0]):
            for rr in range(16):
                e = ell[grp, rr]
                cold = ~np.isnan(e) & ~h[grp]
                share = np.where(cold, np.nan_to_num(e), 0.0) * a / lam[grp, rr]
                if r is a1:
                    assert np.all(share <= eps * nbar * (1 + 1e-5))
                else:
                    assert np.all(np.where(cold, np.nan_to_num(e), 0.0) <= eps * lam[grp, rr] * (1 + 1e-9))
                    over_plain += int((share > eps * nbar * (1 + 1e-5)).sum())
    assert over_plain > 0  # the plain test leaves some large-norm tile cold above that bound


def test_weighted_eps_limits():
    w = synth.small(B=1, Hq=2, Hkv=1, Nq=64, Nkv=1024, d=64, n_outliers=1, seed=2)
    q, k, v = synth.generate(w)
    for eps in (0.0, np.inf):
        a0 = oracle.apa(q, k, v, eps=eps)
        a1 = oracle.apa(q, k, v, eps=eps, quant=VW)
        assert np.array_equal(a0["hot_mask"], a1["hot_mask"])
        assert np.array_equal(a0["out"], a1["out"])
