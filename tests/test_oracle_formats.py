"""Pins for the oracle's NVFP4 formats and quantizer (CPU only).

Each test checks the oracle against something other than itself: values the
APA blog prints, brute-force enumeration, or PyTorch's float8_e4m3fn cast.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from mixed_precision_attention_gb300 import synth


def test_e2m1_value_set_matches_page(golden):
    vals = sorted({oracle.e2m1_value(c) for c in range(16)})
    assert vals == sorted(set(golden["e2m1_values"]))
    assert max(vals) == 6.0


def _nearest_even_bruteforce(x):
    """Nearest E2M1 value by exhaustive search; ties go to the code with an even mantissa bit."""
    best = None
    for code in range(8):
        val = oracle.e2m1_value(code)
        err = abs(abs(x) - val)
        key = (err, code & 1)  # smaller error first, then even code
        if best is None or key < best[0]:
            best = (key, code)
    return best[1] | (8 if math.copysign(1.0, x) < 0 else 0)


def test_e2m1_rounding_bruteforce():
    mags = [0.0, 0.125, 0.25, 0.2500001, 0.5, 0.75, 0.7499999, 1.0, 1.25, 1.2500001, 1.5, 1.75,
            1.7499999, 2.0, 2.5, 2.5000002, 3.0, 3.5, 3.4999998, 4.0, 5.0, 5.0000005, 6.0]
    mags += list(np.linspace(0, 6, 2401)[1:])
    for m in mags:
        for x in (m, -m):
            assert oracle.e2m1_code(x) == _nearest_even_bruteforce(x), x
    # saturation beyond the largest value
    for x in (6.5, 7.0, 100.0, 1e30):
        assert oracle.e2m1_code(x) == 7 and oracle.e2m1_code(-x) == 15


def test_ue4m3_matches_torch_float8_cast(golden):
    # every representable value and every midpoint between neighbours, plus a dense grid
    reps = np.array([oracle.ue4m3_value(c) for c in range(0x7F)])
    assert reps.max() == golden["ue4m3_max"]
    mids = (reps[1:] + reps[:-1]) / 2
    grid = np.concatenate([reps, mids, np.geomspace(2.0 ** -11, 448, 20000)]).astype(np.float32)
    ref = torch.from_numpy(grid).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([oracle.ue4m3_code(float(x)) for x in grid])
    assert np.array_equal(ours, ref)
    # decoded values agree with torch's decoding for every finite non-negative code
    dec = torch.arange(0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(reps.astype(np.float32), dec)
    # saturation: anything at or above 448 is the largest finite code
    for x in (448.0, 460.0, 1e6):
        assert oracle.ue4m3_code(x) == 0x7E


def test_head_scale_maps_max_to_2688(golden):
    assert golden["head_max_maps_to"] == 6 * golden["ue4m3_max"]
    rng = np.random.default_rng(1)
    for _ in range(200):
        x = (rng.standard_normal(64) * 10 ** rng.uniform(-3, 3)).astype(np.float32)
        A = float(np.abs(x).max())
        s = oracle.head_scale(A)
        codes, sf = oracle.quantize_blocks(x, s)
        i = int(np.abs(x).argmax())
        blk = i // 16
        assert sf[blk] == 0x7E  # scale 448
        assert codes[i] & 7 == 7  # element 6
        deq = oracle.e2m1_value(int(codes[i])) * oracle.ue4m3_value(int(sf[blk])) * s
        assert abs(abs(deq) - A) <= 2 * np.spacing(np.float32(A))
    assert oracle.head_scale(0.0) == 1.0


def test_quantizer_error_bound_and_zero_blocks():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((512, 64)) * np.exp(rng.uniform(-6, 6, (512, 1)))).astype(np.float32)
    x[3, 16:32] = 0.0  # an all-zero block
    A = float(np.abs(x).max())
    s = oracle.head_scale(A)
    codes, sf = oracle.quantize_blocks(x, s)
    vals = np.vectorize(oracle.e2m1_value)(codes.astype(int))
    scales = np.vectorize(oracle.ue4m3_value)(sf.astype(int))
    step = np.repeat(scales, 16, axis=-1) * s
    deq = vals * step
    err = np.abs(x - deq)
    normal = np.repeat(sf, 16, axis=-1) >= 8
    # normal scales: the E2M1 grid's largest half-gap is 1 (between 4 and 6); saturation costs less
    assert np.all(err[normal] <= step[normal] * (1 + 1e-6))
    # subnormal scales carry fewer mantissa bits, so a block maximum may saturate at 6
    sub = ~normal
    assert sub.any()
    assert np.all(err[sub] <= np.maximum(step[sub], np.abs(x[sub]) - 6 * step[sub]) * (1 + 1e-6))
    assert sf[3, 1] == 0 and np.all(codes[3, 16:32] == 0)


def test_key_mean_against_exact_sum():
    rng = np.random.default_rng(3)
    for Nkv, d in [(1, 64), (64, 64), (200, 128), (4096, 64)]:
        kf = (rng.standard_normal((Nkv, d)) + 3.0).astype(np.float32)
        kb = synth.f32_to_bf16_bits(kf)
        exact = np.array([math.fsum(col) for col in synth.bf16_bits_to_f32(kb).astype(np.float64).T]) / Nkv
        mu = oracle.key_mean(kb)
        # FP32 sums of <= 64 bf16 values: rounding error <= 64 * 2^-24 relative to the tile magnitude
        tol = 64 * 2.0 ** -24 * (np.abs(synth.bf16_bits_to_f32(kb)).max()) + np.spacing(np.abs(exact).astype(np.float32))
        assert np.all(np.abs(mu - exact) <= tol)
    # more than one 64-tile range: still the mean within the FP32 tile-sum rounding bound
    kf = (rng.standard_normal((64 * 64 * 3 + 100, 64)) + 3.0).astype(np.float32)
    kb = synth.f32_to_bf16_bits(kf)
    exact = np.array([math.fsum(col) for col in synth.bf16_bits_to_f32(kb).astype(np.float64).T]) / kb.shape[0]
    assert np.all(np.abs(oracle.key_mean(kb) - exact) <= 64 * 2.0 ** -24 * 8.0 + np.spacing(np.float32(4.0)))
    # all keys equal: the mean is that value exactly
    kb = synth.f32_to_bf16_bits(np.full((300, 64), 1.5, np.float32))
    assert np.all(oracle.key_mean(kb) == 1.5)


def test_quantize_kv_dequantizes_to_centred_keys_and_values():
    w = synth.small(Nkv=200, Nq=40, d=64, n_outliers=4)
    q, k, v = synth.generate(w)
    r = oracle.quantize_kv(k, v)
    kf = synth.bf16_bits_to_f32(k[0, 0]).astype(np.float64)
    vf = synth.bf16_bits_to_f32(v[0, 0]).astype(np.float64)
    assert np.allclose(r["mu"][0, 0], kf.mean(0), atol=1e-5)
    dec = np.vectorize(oracle.e2m1_value)
    sc = np.vectorize(oracle.ue4m3_value)
    kd = dec(r["kcodes"][0, 0].astype(int)) * np.repeat(sc(r["ksf"][0, 0].astype(int)), 16, -1) * r["s_k"][0, 0]
    kc = kf - r["mu"][0, 0]
    assert np.max(np.abs(kd - kc)) <= np.abs(kc).max() / 6 * 1.2  # at most one E2M1 half-gap of the block scale
    assert (kd * kc).sum() / np.linalg.norm(kd) / np.linalg.norm(kc) > 0.99
    vd = dec(r["vcodes"][0, 0].astype(int)) * np.repeat(sc(r["vsf"][0, 0].astype(int)), 16, -1) * r["s_v"][0, 0]
    vd = vd[:, :200].T  # V^T, padded to 208 keys
    assert (vd * vf).sum() / np.linalg.norm(vd) / np.linalg.norm(vf) > 0.99
    assert np.all(r["vcodes"][0, 0][:, 200:] == 0)


def test_blob_size_matches_page(golden):
    # K and V^T codes (d/2 bytes per key each) plus one UE4M3 scale per 16 values of each
    d = 128
    per_tile = golden["key_tile"] * (d // 2) * 2 + golden["key_tile"] * d // golden["values_per_scale"] * 2
    assert per_tile == golden["blob_bytes_per_tile_d128"] == 72 * d
    tiles = 122880 // golden["key_tile"]
    assert round(tiles * 8 * per_tile / 2 ** 20, 1) == golden["fp4_kv_copy_mib_8heads_122880keys"]
    # the window: sink tile + 2 ring slots of 96 tiles per KV head, 8 heads
    assert round((1 + 2 * 96) * 8 * per_tile / 2 ** 20, 1) == golden["fp4_kv_window_mib_8heads"]
