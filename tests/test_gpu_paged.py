"""apa_attention_paged: K and V in pages of 64 keys from a shared pool, addressed
through a per-sequence block table (the blog, "What else is in the box": pass 2
reads through a block table).  The results must be those of apa_attention on the
same keys laid out contiguously, bit for bit: the same arithmetic, other
addresses.  The pool's unused pages and the rows past Nkv in each sequence's last
page hold NaN, which must never reach a result."""
import numpy as np
import pytest

from mixed_precision_attention_gb300 import synth
from tests import _gpu

pytestmark = pytest.mark.gpu

SHAPES = {
    "gqa3_ragged": dict(B=1, Hq=3, Hkv=1, Nq=45, Nkv=1000, d=64, n_outliers=2),
    "batch_ragged_d128": dict(B=2, Hq=8, Hkv=2, Nq=100, Nkv=1100, d=128, n_outliers=4),
    "d256": dict(B=1, Hq=4, Hkv=2, Nq=64, Nkv=700, d=256, n_outliers=4),
    "aligned": dict(B=2, Hq=4, Hkv=2, Nq=128, Nkv=2048, d=128, n_outliers=2),
}
NAN_BF16 = 0x7FC0


def _paged(k, v, seed=0, spare=5):
    """Pool [num_pages, Hkv, 64, d] with the sequences' tiles at shuffled pages."""
    B, Hkv, Nkv, d = k.shape
    T = (Nkv + 63) // 64
    rng = np.random.default_rng(seed)
    num_pages = B * T + spare
    order = rng.permutation(num_pages)[:B * T].reshape(B, T).astype(np.int32)
    kp = np.full((num_pages, Hkv, 64, d), NAN_BF16, np.uint16)
    vp = np.full_like(kp, NAN_BF16)
    for b in range(B):
        for t in range(T):
            n = min(64, Nkv - 64 * t)
            kp[order[b, t], :, :n] = k[b, :, 64 * t:64 * t + n]
            vp[order[b, t], :, :n] = v[b, :, 64 * t:64 * t + n]
    table = np.full((B, T + 3), -7, np.int32)  # entries past T are never read
    table[:, :T] = order
    return kp, vp, table


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("eps", [0.005, 0.0, float("inf")])
@pytest.mark.parametrize("causal", [True, False])
def test_paged_equals_contiguous(name, eps, causal):
    import torch

    import mixed_precision_attention_gb300 as apa
    w = synth.small(causal=causal, sink_gain=4.0, **SHAPES[name])
    q, k, v = synth.generate(w)
    kp, vp, table = _paged(k, v, seed=w.Nkv)
    dev = _gpu.run_apa(q, k, v, causal=causal, eps=eps)
    out, lse, mask = apa.attention_paged(_gpu.to_dev(q), _gpu.to_dev(kp), _gpu.to_dev(vp),
                                         torch.from_numpy(table).cuda(), w.Nkv, causal=causal, eps=eps,
                                         return_hot_mask=True)
    apa.check_error()
    assert np.array_equal(out.cpu().numpy().astype(np.float64), dev[0])
    assert np.array_equal(lse.cpu().numpy().astype(np.float64), dev[1])
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), dev[2])


def test_paged_bad_table_entry_is_reported():
    # a page index outside the pool reads page 0 (no out-of-bounds access) and the
    # call reports a device bounds error
    import torch

    import mixed_precision_attention_gb300 as apa
    w = synth.small(**SHAPES["gqa3_ragged"])
    q, k, v = synth.generate(w)
    kp, vp, table = _paged(k, v)
    table[0, 3] = kp.shape[0] + 10
    apa.attention_paged(_gpu.to_dev(q), _gpu.to_dev(kp), _gpu.to_dev(vp), torch.from_numpy(table).cuda(), w.Nkv,
                        eps=0.005)
    with pytest.raises(apa.ApaError):
        apa.check_error()
    apa.check_error()  # reported once, then cleared
