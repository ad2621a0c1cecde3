"""The C-ABI library builds, loads and exports what include/apa.h declares; its
host-side argument checks return the documented statuses (CPU only: no call
here reaches the GPU)."""
import ctypes
import math

import pytest

from mixed_precision_attention_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    seen = set()
    for s in range(0, -11, -1):
        text = _lib.status_string(s)
        assert text and text != "unknown status"
        seen.add(text)
    assert len(seen) == 11
    assert _lib.status_string(-99) == "unknown status"


P = ctypes.c_void_p
OK_PTR = (P(0x10000), P(0x20000), P(0x30000))


def _call(lib, q=OK_PTR[0], k=OK_PTR[1], v=OK_PTR[2], B=1, Hq=2, Hkv=1, Nq=128, Nkv=512, d=64, causal=1,
          eps=0.005, out=P(0x40000)):
    # every case below is rejected before anything is enqueued, so the fake
    # pointers are never dereferenced
    return lib.apa_attention(q, k, v, B, Hq, Hkv, Nq, Nkv, d, causal, eps, out, None, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), -1), (dict(k=None), -1), (dict(v=None), -1), (dict(out=None), -1),
    (dict(B=0), -2), (dict(Hq=3, Hkv=2), -2), (dict(Nq=0), -2), (dict(Nkv=100, Nq=128), -2),
    (dict(Nkv=64 * 65536), -2),
    (dict(eps=-0.1), -3), (dict(eps=math.nan), -3),
    (dict(d=96), -4), (dict(d=32), -4), (dict(d=512), -4),
    (dict(v=P(0x30008)), -8),
])
def test_argument_errors(lib, kw, status):
    assert _call(lib, **kw) == status


def test_sizes(lib):
    # one 9216-byte blob per 64-key tile at d = 128 (135.0 MiB at 8 heads x 122880 keys)
    assert lib.apa_kv_blob_bytes(1, 8, 122880, 128) == 1920 * 8 * 9216
    assert lib.apa_kv_blob_bytes(1, 1, 65, 128) == 2 * 9216
    # 128 packed rows x 72 d bytes per Q block; GQA packs G * Nq rows
    assert lib.apa_q_blob_bytes(1, 24, 8, 2048, 128) == 8 * 48 * 72 * 128
    # eps = 0 (all exact): the FP16 copy of V (8 heads x 122880 keys x 128 x 2 B) and the head maxima
    assert lib.apa_workspace_bytes(1, 24, 8, 2048, 122880, 128, 0.0) == 8 * 122880 * 128 * 2 + 256
    assert lib.apa_workspace_bytes(1, 24, 8, 2048, 122880, 128, 0.005) > 141557760
    assert lib.apa_workspace_bytes(1, 3, 2, 16, 64, 64, 0.005) == 0  # Hq % Hkv != 0
    # eps = 0 at d = 256 with a long walk (2048 tiles, one block): two parts' states too
    assert lib.apa_workspace_bytes(1, 1, 1, 16, 131072, 256, 0.0) >= 131072 * 256 * 2 + 2 * 128 * (256 * 4 + 8)
    assert lib.apa_workspace_bytes(1, 1, 1, 16, 65536, 256, 0.0) < 65536 * 256 * 2 + 128 * 256 * 4
    # eps > 0 at d = 256: pass 2's walk over the hot list splits one part per 512 tiles.
    # From 1022 to 1023 tiles the workspace grows by one tile's share; from 1023 to 1024
    # by that plus two parts' states (2 x 128 rows of O and (m, l)) and a q.mu term per
    # row, each rounded up to 256 bytes
    ws = lambda nkv: lib.apa_workspace_bytes(1, 1, 1, 16, nkv, 256, 0.005)  # noqa: E731
    tile = ws(65472) - ws(65408)
    parts = 2 * 128 * 256 * 4 + 2 * 128 * 8 + 128 * 4
    assert parts <= ws(65536) - ws(65472) - tile <= parts + 3 * 255


def test_workspace_too_small_is_rejected(lib):
    need = lib.apa_workspace_bytes(1, 2, 1, 128, 512, 64, 0.005)
    st = lib.apa_attention_ws(*OK_PTR, 1, 2, 1, 128, 512, 64, 1, 0.005, P(0x40000), None, None,
                              P(0x50000), need - 1, None)
    assert st == -6
    st = lib.apa_attention_ws(*OK_PTR, 1, 2, 1, 128, 512, 64, 1, 0.005, P(0x40000), None, None,
                              P(0x50010), need, None)  # not 256-byte aligned
    assert st == -6


def test_option_flags(lib):
    # the residual-Q option needs one more Q blob; unknown bits are rejected before any work
    base = lib.apa_workspace_bytes_ex(1, 2, 1, 128, 512, 64, 0.005, 0)
    assert base == lib.apa_workspace_bytes(1, 2, 1, 128, 512, 64, 0.005)
    q2 = lib.apa_workspace_bytes_ex(1, 2, 1, 128, 512, 64, 0.005, 1)
    assert q2 >= base + lib.apa_q_blob_bytes(1, 2, 1, 128, 64)
    assert lib.apa_workspace_bytes_ex(1, 2, 1, 128, 512, 64, 0.005, 2) == base  # the scale choice needs no memory
    # the value-weighted test keeps two floats per (b, KV head, tile): 8 tiles here
    vw = lib.apa_workspace_bytes_ex(1, 2, 1, 128, 512, 64, 0.005, 4)
    assert base + 2 * 8 * 4 <= vw <= base + 2 * 256
    assert lib.apa_workspace_bytes_ex(1, 2, 1, 128, 512, 64, 0.005, 16) == 0
    st = lib.apa_attention_ex(*OK_PTR, 1, 2, 1, 128, 512, 64, 1, 0.005, 16, P(0x40000), None, None, None, 0, None)
    assert st == -10
    # the ones-MMA row sums and the residual Q term share TMEM columns: refused together
    st = lib.apa_attention_ex(*OK_PTR, 1, 2, 1, 128, 512, 64, 1, 0.005, 9, P(0x40000), None, None, None, 0, None)
    assert st == -10
    z = P(0x60000)
    st = lib.apa_quantize_ex(*OK_PTR, 1, 2, 1, 128, 512, 64, 16, z, z, None, z, z, z, z, None)
    assert st == -10
    st = lib.apa_attention_ex(*OK_PTR, 1, 2, 1, 128, 512, 64, 1, 0.005, 4, P(0x40000), None, None,
                              P(0x50000), vw - 1, None)
    assert st == -6
    st = lib.apa_attention_ex(*OK_PTR, 1, 2, 1, 128, 512, 64, 1, 0.005, 1, P(0x40000), None, None,
                              P(0x50000), q2 - 1, None)
    assert st == -6


def test_quantize_argument_errors(lib):
    z = P(0x60000)
    assert lib.apa_quantize(*OK_PTR, 1, 2, 1, 128, 512, 64, None, z, z, z, z, z, None) == -1
    assert lib.apa_quantize(*OK_PTR, 1, 2, 1, 128, 512, 80, z, z, z, z, z, z, None) == -4


def test_noalloc_quantizer_rejects_oversized_problems(lib):
    # statistics of the 2 x 8 heads x 131072 keys x d=256 problem need ~34 MB, more
    # than the fixed 16 MiB array: rejected before anything touches the GPU
    z = P(0x60000)
    need = lib.apa_quantize_noalloc_scratch_bytes(2, 32, 8, 131072, 256)
    assert need > 16 * 2 ** 20
    assert lib.apa_quantize_noalloc(*OK_PTR, 2, 32, 8, 128, 131072, 256, z, z, z, z, z, z, None) == -9
    assert _lib.status_string(-9) != "unknown status"
    assert lib.apa_quantize_noalloc_scratch_bytes(1, 24, 8, 122880, 128) <= 16 * 2 ** 20
    assert lib.apa_quantize_noalloc(*OK_PTR, 1, 2, 1, 128, 512, 64, None, z, z, z, z, z, None) == -1


def test_paged_argument_errors(lib):
    # rejected on the host before anything is enqueued
    z = P(0x70000)
    # a null block table
    assert lib.apa_attention_paged(*OK_PTR, 10, None, 8, 1, 2, 1, 128, 512, 64, 1, 0.005, z, None, None, None) == -1
    # max_pages below ceil(Nkv / 64), and an empty pool
    assert lib.apa_attention_paged(*OK_PTR, 10, z, 7, 1, 2, 1, 128, 512, 64, 1, 0.005, z, None, None, None) == -2
    assert lib.apa_attention_paged(*OK_PTR, 0, z, 8, 1, 2, 1, 128, 512, 64, 1, 0.005, z, None, None, None) == -2
    # the usual shape checks still apply
    assert lib.apa_attention_paged(*OK_PTR, 10, z, 8, 1, 3, 2, 128, 512, 64, 1, 0.005, z, None, None, None) == -2
