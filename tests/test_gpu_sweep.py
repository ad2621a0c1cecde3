"""A seeded sweep of random shapes: the CUDA path against the oracle on shapes
no one picked by hand (batch, GQA group size, head dim, ragged query and key
counts, causal or not), so that an index or tail mistake tied to some
combination shows up.  The bounds are those of the hand-picked cases in
test_gpu_attention.py (eps = 0 against exact attention; eps > 0 against the
APA emulation, with mask agreement and the cold-tile bound) and, for the
quantizer, bit-exactness as in test_gpu_quant.py."""
import numpy as np
import pytest

import oracle
from mixed_precision_attention_gb300 import synth
from tests import _gpu
from tests.test_gpu_attention import _check_apa

pytestmark = pytest.mark.gpu


def _draw(n, seed):
    """n random shapes, small enough that the FP64 oracle finishes each in seconds."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(rng.choice([64, 128, 256]))
        G = int(rng.choice([1, 2, 3, 4, 5, 8]))
        Hkv = int(rng.choice([1, 2]))
        B = int(rng.choice([1, 2])) if Hkv == 1 else 1
        Nq = int(rng.integers(1, 200 if d < 256 else 120))
        Nkv = int(Nq + rng.integers(0, 2000 if d < 256 else 1200))
        out.append(dict(B=B, Hq=G * Hkv, Hkv=Hkv, Nq=Nq, Nkv=max(Nkv, 1), d=d,
                        causal=bool(rng.integers(0, 2)), n_outliers=int(rng.choice([0, 2])),
                        seed=int(rng.integers(0, 1 << 30))))
    return out


ATTN = _draw(16, 2024)
QUANT = _draw(12, 77)


def _id(c):
    return "B{B}_Hq{Hq}_Hkv{Hkv}_q{Nq}_k{Nkv}_d{d}_{c}".format(c="causal" if c["causal"] else "full", **c)


def _workload(c):
    kw = {k: v for k, v in c.items() if k != "causal"}
    return synth.small(causal=c["causal"], sink_gain=4.0, **kw)


@pytest.mark.parametrize("case", ATTN, ids=[_id(c) for c in ATTN])
def test_random_shape_matches_oracle(case, record_property):
    w = _workload(case)
    q, k, v = synth.generate(w)
    causal = case["causal"]
    # eps = 0: exact attention
    ex, ex_lse = oracle.exact(q, k, v, causal=causal)
    out, lse, _ = _gpu.run_apa(q, k, v, causal=causal, eps=0.0)
    assert np.abs(out - ex).max() <= 4e-3
    assert np.abs(lse - ex_lse).max() <= 1e-3
    # eps > 0: the APA emulation, its hot masks and the cold-tile bound
    _check_apa(w, q, k, v, 0.005, causal=causal, record=record_property)


@pytest.mark.parametrize("case", ATTN[::3], ids=[_id(c) for c in ATTN[::3]])
def test_random_shape_all_fp4(case):
    w = _workload(case)
    q, k, v = synth.generate(w)
    ref = oracle.apa(q, k, v, causal=case["causal"], eps=np.inf)
    out, lse, mask = _gpu.run_apa(q, k, v, causal=case["causal"], eps=np.inf)
    assert np.abs(out - ref["out"]).max() <= 1e-2
    assert np.abs(lse - ref["lse"]).max() <= 1e-2
    assert not mask.any()


@pytest.mark.parametrize("case", QUANT, ids=[_id(c) for c in QUANT])
def test_random_shape_quantizer_bit_exact(case):
    import mixed_precision_attention_gb300 as apa
    w = _workload(case)
    q, k, v = synth.generate(w)
    B, Hq, Hkv, Nq, Nkv, d = w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.d
    r = apa.quantize(_gpu.to_dev(q), _gpu.to_dev(k), _gpu.to_dev(v))
    apa.check_error()
    g = {n: t.cpu().numpy() for n, t in r.items()}
    ok, oq = oracle.quantize_kv(k, v), oracle.quantize_q(q)
    assert np.array_equal(g["mu"].view(np.uint32), ok["mu"].view(np.uint32))
    assert np.array_equal(g["s_k"], ok["s_k"].astype(np.float32))
    assert np.array_equal(g["s_v"], ok["s_v"].astype(np.float32))
    assert np.array_equal(g["s_q"], oq["s_q"].astype(np.float32))
    kc, ksf, vc, vsf = _gpu.decode_kv_blob(g["kv_blob"], B, Hkv, Nkv, d)
    assert np.array_equal(kc[:, :, :Nkv], ok["kcodes"]) and np.array_equal(ksf[:, :, :Nkv], ok["ksf"])
    Npad = ok["vcodes"].shape[-1]
    assert np.array_equal(vc[..., :Npad], ok["vcodes"]) and np.array_equal(vsf[..., :Npad // 16], ok["vsf"])
    qc, qsf, pad_c, pad_s = _gpu.decode_q_blob(g["q_blob"], B, Hq, Hkv, Nq, d)
    assert np.array_equal(qc, oq["codes"]) and np.array_equal(qsf, oq["sf"])
    assert not pad_c.any() and not pad_s.any()


@pytest.mark.parametrize("case", ATTN[1::3], ids=[_id(c) for c in ATTN[1::3]])
def test_random_shape_host_and_paged_equal_device(case):
    """The host entry point (per-(b, KV head) sub-problems, the last in the one-block
    form, with the separate K/V quantizer) and the paged entry point (K/V through a
    shuffled block table) give the device call's results bit for bit."""
    import torch

    import mixed_precision_attention_gb300 as apa
    from tests.test_gpu_paged import _paged
    w = _workload(case)
    q, k, v = synth.generate(w)
    causal = case["causal"]
    dev = _gpu.run_apa(q, k, v, causal=causal, eps=0.005)
    hq, hk, hv = (synth.to_torch_bf16(a).pin_memory() for a in (q, k, v))
    out, lse, mask = apa.attention_host(hq, hk, hv, causal=causal, eps=0.005, return_hot_mask=True)
    assert np.array_equal(out.numpy().astype(np.float64), dev[0])
    assert np.array_equal(lse.numpy().astype(np.float64), dev[1])
    assert np.array_equal(mask.numpy().view(np.uint32), dev[2])
    kp, vp, table = _paged(k, v, seed=w.Nkv)
    out, lse, mask = apa.attention_paged(_gpu.to_dev(q), _gpu.to_dev(kp), _gpu.to_dev(vp),
                                         torch.from_numpy(table).cuda(), w.Nkv, causal=causal, eps=0.005,
                                         return_hot_mask=True)
    apa.check_error()
    assert np.array_equal(out.cpu().numpy().astype(np.float64), dev[0])
    assert np.array_equal(lse.cpu().numpy().astype(np.float64), dev[1])
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), dev[2])
    torch.cuda.synchronize()
