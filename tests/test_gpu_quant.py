"""The CUDA NVFP4 quantizer against the oracle: codes, scales, key mean and
head scales bit-exact (blog, "Pass 1: FP4 everywhere, with a hot test" and
"Mean-centred K")."""
import numpy as np
import pytest

import oracle
from mixed_precision_attention_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu

CASES = [
    dict(B=1, Hq=2, Hkv=1, Nq=128, Nkv=512, d=64, n_outliers=0),      # the tiny workload
    dict(B=2, Hq=6, Hkv=2, Nq=37, Nkv=1000, d=128, n_outliers=4),    # G=3, ragged keys and rows
    dict(B=1, Hq=4, Hkv=2, Nq=20, Nkv=333, d=256, n_outliers=4),     # d=256, ragged
    dict(B=1, Hq=32, Hkv=8, Nq=256, Nkv=4096, d=128, n_outliers=4),  # prefill-shaped
]


def _quant_gpu(q, k, v):
    import mixed_precision_attention_gb300 as apa
    r = apa.quantize(_gpu.to_dev(q), _gpu.to_dev(k), _gpu.to_dev(v))
    apa.check_error()
    return {n: t.cpu().numpy() for n, t in r.items()}


@pytest.mark.parametrize("case", CASES)
def test_quantizer_bit_exact(case):
    w = synth.small(sink_gain=4.0, **case)
    q, k, v = synth.generate(w)
    B, Hq, Hkv, Nq, Nkv, d = w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.d
    g = _quant_gpu(q, k, v)
    ok = oracle.quantize_kv(k, v)
    oq = oracle.quantize_q(q)
    # key mean and FP32 head scales: bitwise
    assert np.array_equal(g["mu"].view(np.uint32), ok["mu"].view(np.uint32))
    assert np.array_equal(g["s_k"], ok["s_k"].astype(np.float32))
    assert np.array_equal(g["s_v"], ok["s_v"].astype(np.float32))
    assert np.array_equal(g["s_q"], oq["s_q"].astype(np.float32))
    kc, ksf, vc, vsf = _gpu.decode_kv_blob(g["kv_blob"], B, Hkv, Nkv, d)
    assert np.array_equal(kc[:, :, :Nkv], ok["kcodes"])
    assert np.array_equal(ksf[:, :, :Nkv], ok["ksf"])
    assert not kc[:, :, Nkv:].any() and not ksf[:, :, Nkv:].any()
    Npad = ok["vcodes"].shape[-1]
    assert np.array_equal(vc[..., :Npad], ok["vcodes"])
    assert np.array_equal(vsf[..., :Npad // 16], ok["vsf"])
    assert not vc[..., Npad:].any() and not vsf[..., Npad // 16:].any()
    qc, qsf, pad_c, pad_s = _gpu.decode_q_blob(g["q_blob"], B, Hq, Hkv, Nq, d)
    assert np.array_equal(qc, oq["codes"]) and np.array_equal(qsf, oq["sf"])
    assert not pad_c.any() and not pad_s.any()


def test_quantizer_adversarial_blocks():
    """Ties, zeros, an all-zero head and tiny blocks with subnormal scales."""
    B, Hq, Hkv, Nq, Nkv, d = 1, 2, 2, 64, 256, 64
    rng = np.random.default_rng(7)
    qf = rng.standard_normal((B, Hq, Nq, d)).astype(np.float32)
    kf = rng.standard_normal((B, Hkv, Nkv, d)).astype(np.float32)
    vf = rng.standard_normal((B, Hkv, Nkv, d)).astype(np.float32)
    qf[0, 1] = 0.0                                   # an all-zero head: scale 1, every code 0
    vf[0, 0, :16, :] = 0.0                           # zero V blocks
    kf[0, 1, 5, :] = np.tile([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], 8)  # E2M1 midpoints
    qf[0, 0, 3, :16] = 1e-6                          # a tiny block next to large ones
    qf[0, 0, 3, 16:] = 100.0
    vf[0, 1, 32:48, 7] = 3e-7 * np.arange(16)        # subnormal UE4M3 block scale
    q, k, v = (synth.f32_to_bf16_bits(a) for a in (qf, kf, vf))
    g = _quant_gpu(q, k, v)
    ok = oracle.quantize_kv(k, v)
    oq = oracle.quantize_q(q)
    kc, ksf, vc, vsf = _gpu.decode_kv_blob(g["kv_blob"], B, Hkv, Nkv, d)
    assert np.array_equal(kc, ok["kcodes"]) and np.array_equal(ksf, ok["ksf"])
    assert np.array_equal(vc, ok["vcodes"]) and np.array_equal(vsf, ok["vsf"])
    qc, qsf, _, _ = _gpu.decode_q_blob(g["q_blob"], B, Hq, Hkv, Nq, d)
    assert np.array_equal(qc, oq["codes"]) and np.array_equal(qsf, oq["sf"])
    assert g["s_q"][0, 1] == 1.0 and not qc[0, 1].any()
    assert (vsf[0, 1, 7, 2] < 8)  # the subnormal scale really occurs


def test_quantizer_deterministic():
    w = synth.small(B=1, Hq=4, Hkv=2, Nq=100, Nkv=2000, d=128, n_outliers=4)
    q, k, v = synth.generate(w)
    a, b = _quant_gpu(q, k, v), _quant_gpu(q, k, v)
    for n in a:
        assert np.array_equal(a[n], b[n])


@pytest.mark.parametrize("case", [CASES[1], CASES[2]])
def test_q_residual_blob_bit_exact(case):
    # the FP4 residual term of Q (Q2 = FP4(Q - Q1) under the same head scale)
    import mixed_precision_attention_gb300 as apa
    w = synth.small(sink_gain=4.0, **case)
    q, k, v = synth.generate(w)
    r = apa.quantize(_gpu.to_dev(q), _gpu.to_dev(k), _gpu.to_dev(v), q_residual=True)
    apa.check_error()
    oq = oracle.quantize_q(q, residual=True)
    qc, qsf, _, _ = _gpu.decode_q_blob(r["q_blob"].cpu().numpy(), w.B, w.Hq, w.Hkv, w.Nq, w.d)
    assert np.array_equal(qc, oq["codes"]) and np.array_equal(qsf, oq["sf"])
    c2, s2, pad_c, pad_s = _gpu.decode_q_blob(r["q2_blob"].cpu().numpy(), w.B, w.Hq, w.Hkv, w.Nq, w.d)
    assert np.array_equal(c2, oq["codes2"]) and np.array_equal(s2, oq["sf2"])
    assert not pad_c.any() and not pad_s.any()
    assert oq["sf2"].any()  # the residual is not trivially zero


@pytest.mark.parametrize("case", [CASES[0], CASES[1], CASES[2]])
def test_lse_scales_bit_exact(case):
    # least-squared-error block scales (APA_FLAG_LSE_SCALES) for K, V, Q and the residual Q
    import mixed_precision_attention_gb300 as apa
    w = synth.small(sink_gain=4.0, **case)
    q, k, v = synth.generate(w)
    B, Hq, Hkv, Nq, Nkv, d = w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.d
    r = apa.quantize(_gpu.to_dev(q), _gpu.to_dev(k), _gpu.to_dev(v), q_residual=True, lse_scales=True)
    apa.check_error()
    g = {n: t.cpu().numpy() for n, t in r.items()}
    ok = oracle.quantize_kv(k, v, lse=True)
    oq = oracle.quantize_q(q, residual=True, lse=True)
    kc, ksf, vc, vsf = _gpu.decode_kv_blob(g["kv_blob"], B, Hkv, Nkv, d)
    assert np.array_equal(kc[:, :, :Nkv], ok["kcodes"]) and np.array_equal(ksf[:, :, :Nkv], ok["ksf"])
    Npad = ok["vcodes"].shape[-1]
    assert np.array_equal(vc[..., :Npad], ok["vcodes"]) and np.array_equal(vsf[..., :Npad // 16], ok["vsf"])
    qc, qsf, _, _ = _gpu.decode_q_blob(g["q_blob"], B, Hq, Hkv, Nq, d)
    assert np.array_equal(qc, oq["codes"]) and np.array_equal(qsf, oq["sf"])
    c2, s2, _, _ = _gpu.decode_q_blob(g["q2_blob"], B, Hq, Hkv, Nq, d)
    assert np.array_equal(c2, oq["codes2"]) and np.array_equal(s2, oq["sf2"])
    near = oracle.quantize_kv(k, v)
    assert (near["ksf"] != ok["ksf"]).any()  # the choice is not just the nearest scale


def test_e2m1_rounding_of_every_bf16_value_in_range():
    """Every bf16 value x with |x| <= 6, signed zeros included, through the GPU
    quantizer with head scale 1 and block scale 1 (a head maximum of 2688 and a 6
    in every block), so each code is the plain E2M1 rounding of x: nearest of
    0, 0.5, 1, 1.5, 2, 3, 4, 6, ties to the even code, sign kept.  Checked
    against that rule written out here and against the oracle."""
    pos = np.arange(0x0000, 0x40C1, dtype=np.uint16)          # +0 .. 6.0
    vals = np.concatenate([pos, pos | np.uint16(0x8000)])   # and -0 .. -6.0
    d = 128
    nb = (len(vals) + 14) // 15                              # 15 values + one 6.0 per block
    blocks = np.full((nb, 16), 0x40C0, np.uint16)
    flat = blocks[:, 1:].reshape(-1)
    flat[:len(vals)] = vals
    flat[len(vals):] = 0x40C0
    blocks[:, 1:] = flat.reshape(nb, 15)
    rows = (nb * 16 + d - 1) // d
    qrow = np.full(rows * d, 0x40C0, np.uint16)
    qrow[:nb * 16] = blocks.reshape(-1)
    q = np.zeros((1, 1, rows + 1, d), np.uint16)
    q[0, 0, :rows] = qrow.reshape(rows, d)
    q[0, 0, rows, 0] = synth.f32_to_bf16_bits(np.array([2688.0], np.float32))[0]  # head maximum: scale 1
    kv = synth.f32_to_bf16_bits(np.ones((1, 1, 64, d), np.float32))
    g = _quant_gpu(q, kv, kv)
    assert g["s_q"][0, 0] == 1.0
    qc, qsf, _, _ = _gpu.decode_q_blob(g["q_blob"], 1, 1, 1, rows + 1, d)
    codes = qc[0, 0, :rows].reshape(-1)[:nb * 16].reshape(nb, 16)
    assert (qsf[0, 0, :rows].reshape(-1)[:nb] == 0x38).all()   # UE4M3 1.0 for every test block
    # the rule, independently
    x = synth.bf16_bits_to_f32(vals).astype(np.float64)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    dist = np.abs(np.abs(x)[:, None] - grid)
    best = dist.min(1, keepdims=True)
    cand = np.where(dist == best, np.arange(8), 99)
    even = np.where((dist == best) & (np.arange(8) % 2 == 0), np.arange(8), 99).min(1)
    idx = np.where(even < 99, even, cand.min(1))
    want = idx | (np.signbit(x).astype(np.int64) << 3)
    got = codes[:, 1:].reshape(-1)[:len(vals)]
    assert np.array_equal(got.astype(np.int64), want)
    # and the oracle agrees on the whole tensor
    oq = oracle.quantize_q(q)
    assert np.array_equal(qc, oq["codes"]) and np.array_equal(qsf, oq["sf"])


# The key mean sums per-tile FP32 sums in FP64 per range of 64 tiles, then the
# ranges: these cases span 30 and 32 ranges (the 2048 x 122880 layer's keys with
# two of its KV heads, and the short-query d = 256 shape's 131072 keys), so the
# multi-range reduction is compared bit for bit.
LONG_CASES = [
    dict(B=1, Hq=6, Hkv=2, Nq=64, Nkv=122880, d=128, n_outliers=4),
    dict(B=1, Hq=4, Hkv=1, Nq=128, Nkv=131072, d=256, n_outliers=4),
]


@pytest.mark.parametrize("case", LONG_CASES)
def test_quantizer_bit_exact_many_ranges(case):
    w = synth.small(sink_gain=4.0, **case)
    q, k, v = synth.generate(w)
    assert (w.Nkv + 63) // 64 > 64 * 16  # more than 16 ranges of 64 tiles
    g = _quant_gpu(q, k, v)
    ok = oracle.quantize_kv(k, v)
    oq = oracle.quantize_q(q)
    assert np.array_equal(g["mu"].view(np.uint32), ok["mu"].view(np.uint32))
    assert np.array_equal(g["s_k"], ok["s_k"].astype(np.float32))
    assert np.array_equal(g["s_v"], ok["s_v"].astype(np.float32))
    assert np.array_equal(g["s_q"], oq["s_q"].astype(np.float32))
    kc, ksf, vc, vsf = _gpu.decode_kv_blob(g["kv_blob"], w.B, w.Hkv, w.Nkv, w.d)
    assert np.array_equal(kc, ok["kcodes"]) and np.array_equal(ksf, ok["ksf"])
    assert np.array_equal(vc, ok["vcodes"]) and np.array_equal(vsf, ok["vsf"])
    qc, qsf, _, _ = _gpu.decode_q_blob(g["q_blob"], w.B, w.Hq, w.Hkv, w.Nq, w.d)
    assert np.array_equal(qc, oq["codes"]) and np.array_equal(qsf, oq["sf"])
