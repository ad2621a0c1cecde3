"""The oracle's Q two-term residual ("Second hunt" on the APA page: Q2 is the
FP4 residual Q - Q1 in the same scale, accumulated against the same K), pinned
by bounds computed independently of the oracle's arithmetic."""
import numpy as np

import oracle
from mixed_precision_attention_gb300 import synth

_dec = np.vectorize(oracle.e2m1_value)
_sc = np.vectorize(oracle.ue4m3_value)


def _deq(codes, sf, s):
    return _dec(codes.astype(int)) * np.repeat(_sc(sf.astype(int)), 16, -1) * s


def test_residual_term_bounds_and_reduces_the_error():
    w = synth.small(B=1, Hq=3, Hkv=1, Nq=96, Nkv=128, d=64, n_outliers=2, seed=7)
    q, _, _ = synth.generate(w)
    r = oracle.quantize_q(q, residual=True)
    single = oracle.quantize_q(q)
    assert np.array_equal(r["codes"], single["codes"]) and np.array_equal(r["sf"], single["sf"])
    x = synth.bf16_bits_to_f32(q).astype(np.float64)
    s = r["s_q"][..., None, None]
    d1 = _deq(r["codes"], r["sf"], s)
    d2 = _deq(r["codes2"], r["sf2"], s)
    res = x - d1                                   # the residual, in FP64 here
    amax_r = np.repeat(np.abs(res).reshape(*res.shape[:-1], -1, 16).max(-1), 16, -1)
    # the second term is the FP4 quantization of the residual: within one E2M1
    # half-gap (1) of its block scale, which rounds amax_r / 6 to UE4M3 (rel. <= 1/16)
    # or clamps it at the smallest UE4M3 value; plus the FP32 roundings of the residual
    step2 = np.maximum(amax_r / 6 * (1 + 1 / 16), 2.0 ** -9 * s)
    err2 = np.abs(x - d1 - d2)
    assert np.all(err2 <= step2 * (1 + 1e-6) + 1e-6 * np.abs(x))
    # and it shrinks the error of Q1 alone by a large factor overall
    assert np.linalg.norm(err2) < 0.25 * np.linalg.norm(res)


def test_representable_q_has_zero_residual():
    # values on the E2M1 x UE4M3 grid of their own block scale are exact in Q1
    rng = np.random.default_rng(0)
    vals = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    codes = rng.choice(vals, size=(4, 64)) * rng.choice([-1.0, 1.0], size=(4, 64))
    codes[:, ::16] = 6.0                           # every block reaches 6: scale code exact
    s = oracle.head_scale(6.0 * 2.0)               # head max 12 -> s = 12 / 2688
    scale = 2.0                                    # block scale UE4M3 2.0, applied on top of s
    xf = (codes * scale * s).astype(np.float32)
    c1, f1 = oracle.quantize_blocks(xf, s)
    c2, f2 = np.zeros_like(c1), np.zeros_like(f1)
    lib = oracle._load()
    lib.oracle_quantize_residual_blocks(oracle._ptr(np.ascontiguousarray(xf)), xf.size // 16, s,
                                        oracle._ptr(c1), oracle._ptr(f1), oracle._ptr(c2), oracle._ptr(f2), 0)
    assert np.array_equal(_deq(c1, f1, s).astype(np.float32), xf)  # Q1 holds them up to the FP32 rounding
    assert not c2.any() and not f2.any()


def test_two_term_q_moves_apa_closer_to_exact():
    w = synth.small(B=1, Hq=2, Hkv=1, Nq=128, Nkv=2048, d=64, n_outliers=2, seed=11)
    q, k, v = synth.generate(w)
    ex, _ = oracle.exact(q, k, v)
    # Q the only quantized operand, every tile cold: the error is the FP4 rounding of Q
    one = oracle.apa(q, k, v, eps=float("inf"), quant=oracle.QUANT_Q)["out"]
    two = oracle.apa(q, k, v, eps=float("inf"), quant=oracle.QUANT_Q | oracle.QUANT_Q2)["out"]
    e1, e2 = np.abs(one - ex).max(), np.abs(two - ex).max()
    assert e2 < 0.3 * e1, (e1, e2)
    # with every operand quantized the second term still helps
    a1 = oracle.apa(q, k, v, eps=float("inf"))["out"]
    a2 = oracle.apa(q, k, v, eps=float("inf"), quant=oracle.QUANT_ALL | oracle.QUANT_Q2)["out"]
    assert np.linalg.norm(a2 - ex) < np.linalg.norm(a1 - ex)
