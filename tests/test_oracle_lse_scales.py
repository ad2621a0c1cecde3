"""The oracle's least-squared-error block scales ("Second hunt" on the APA page:
every block scale picked from a small set of candidates by least squared error
instead of the nearest one).  Reading: candidates are the nearest UE4M3 code and
its two neighbours.  Pinned against an FP64 brute force written here."""
import numpy as np

import oracle
from mixed_precision_attention_gb300 import synth

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_rne(y):
    """Nearest E2M1 magnitude (ties to the even code), saturating at 6, sign kept."""
    a = np.minimum(np.abs(y), 6.0)
    d = np.abs(a[..., None] - E2M1)
    best = d.min(-1, keepdims=True)
    tie = np.isclose(d, best, rtol=0, atol=1e-12)
    idx = np.where(tie, np.arange(8), 99)
    even = np.where(tie & (np.arange(8) % 2 == 0), np.arange(8), 99).min(-1)
    pick = np.where(even < 99, even, idx.min(-1))
    return np.sign(y) * E2M1[pick]


def _sse(xb, scale):
    return float(((xb - _e2m1_rne(xb / scale) * scale) ** 2).sum())


def test_lse_scale_is_the_least_squared_error_candidate():
    rng = np.random.default_rng(5)
    # mixed magnitudes: normal and subnormal block scales, outliers that saturate
    x = (rng.standard_normal((600, 16)) * np.exp(rng.uniform(-9, 4, (600, 1)))).astype(np.float32)
    x[::7, 3] *= 9.0
    s = oracle.head_scale(float(np.abs(x).max()))
    c0, f0 = oracle.quantize_blocks(x, s)
    c1, f1 = oracle.quantize_blocks(x, s, lse=True)
    f0, f1 = f0[:, 0].astype(int), f1[:, 0].astype(int)  # one scale per 16-value row
    ue = np.vectorize(oracle.ue4m3_value)
    changed = 0
    for b in range(x.shape[0]):
        xb = x[b].astype(np.float64)
        if f0[b] == 0:
            assert f1[b] == 0 and not c1[b].any()
            continue
        cands = [c for c in (f0[b] - 1, f0[b], f0[b] + 1) if 1 <= c <= 126]
        sse = {c: _sse(xb, ue(c) * s) for c in cands}
        assert f1[b] in sse
        assert sse[f1[b]] <= min(sse.values()) * (1 + 1e-5) + 1e-30
        assert sse[f1[b]] <= sse[f0[b]] * (1 + 1e-6) + 1e-30
        # the codes are those of the chosen scale
        assert np.array_equal(np.vectorize(oracle.e2m1_value)(c1[b].astype(int)), _e2m1_rne(xb / (ue(f1[b]) * s)))
        changed += f1[b] != f0[b]
    assert changed > 0.05 * x.shape[0]  # the choice is not always the nearest


def test_lse_scales_reduce_k_quantization_error():
    w = synth.small(B=1, Hq=2, Hkv=1, Nq=128, Nkv=1024, d=64, n_outliers=2, seed=4)
    q, k, v = synth.generate(w)
    kf = synth.bf16_bits_to_f32(k[0, 0]).astype(np.float64)
    dec, sc = np.vectorize(oracle.e2m1_value), np.vectorize(oracle.ue4m3_value)
    errs = []
    for lse in (False, True):
        r = oracle.quantize_kv(k, v, lse=lse)
        kd = dec(r["kcodes"][0, 0].astype(int)) * np.repeat(sc(r["ksf"][0, 0].astype(int)), 16, -1) * r["s_k"][0, 0]
        errs.append(np.linalg.norm(kd - (kf - r["mu"][0, 0])))
    # per block the chosen scale minimizes the squared error, so the total can only drop
    # (the attention output through the softmax has no such guarantee)
    assert errs[1] < errs[0]
