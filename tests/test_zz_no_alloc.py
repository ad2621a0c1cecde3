"""apa_quantize_noalloc: the quantizer for callers that cannot allocate device
memory while they run (their own arena owns the GPU, or a plugin interface gives
them buffers but no allocator).  It keeps its temporary statistics in a fixed
array inside the library instead of allocating them.

Checked through the C ABI against apa_quantize on two calls in a row: the
second call must not see anything the first left in the shared array.  The
quantizer is bit-exact, so the outputs must be identical byte for byte.

This file sorts last so that a run stopping at the first failure has already
run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

from mixed_precision_attention_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

OUTS = ("kv_blob", "q_blob", "mu", "s_q", "s_k", "s_v")


def _buffers(lib, B, Hq, Hkv, Nq, Nkv, d):
    import torch
    return dict(kv_blob=torch.zeros(lib.apa_kv_blob_bytes(B, Hkv, Nkv, d), dtype=torch.uint8, device="cuda"),
                q_blob=torch.zeros(lib.apa_q_blob_bytes(B, Hq, Hkv, Nq, d), dtype=torch.uint8, device="cuda"),
                mu=torch.zeros((B, Hkv, d), dtype=torch.float32, device="cuda"),
                s_q=torch.zeros((B, Hq), dtype=torch.float32, device="cuda"),
                s_k=torch.zeros((B, Hkv), dtype=torch.float32, device="cuda"),
                s_v=torch.zeros((B, Hkv), dtype=torch.float32, device="cuda"))


def _call(fn, q, k, v, shape, bufs):
    import torch
    B, Hq, Hkv, Nq, Nkv, d = shape
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = fn(P(q), P(k), P(v), B, Hq, Hkv, Nq, Nkv, d, *(P(bufs[n]) for n in OUTS), stream)
    assert st == 0, _lib.status_string(st)
    assert _lib.load().apa_check_error(stream) == 0
    return {n: bufs[n].cpu().numpy() for n in OUTS}


def test_noalloc_quantizer_matches_allocating_one_on_two_calls():
    import torch
    lib = _lib.load()
    workloads = [synth.small(B=2, Hq=8, Hkv=2, Nq=300, Nkv=5000, d=128, n_outliers=4, seed=1, sink_gain=8.0),
                 synth.small(B=1, Hq=3, Hkv=1, Nq=45, Nkv=1000, d=64, n_outliers=2, seed=2)]
    for w in workloads:  # two calls in a row, different problems
        q, k, v = (synth.to_torch_bf16(a, "cuda") for a in synth.generate(w))
        shape = (w.B, w.Hq, w.Hkv, w.Nq, w.Nkv, w.d)
        assert lib.apa_quantize_noalloc_scratch_bytes(w.B, w.Hq, w.Hkv, w.Nkv, w.d) <= 16 * 2 ** 20
        ref = _call(lib.apa_quantize, q, k, v, shape, _buffers(lib, *shape))
        got = _call(lib.apa_quantize_noalloc, q, k, v, shape, _buffers(lib, *shape))
        for n in OUTS:
            assert np.array_equal(ref[n].view(np.uint8), got[n].view(np.uint8)), n
        torch.cuda.synchronize()
