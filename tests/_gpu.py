"""Helpers for the GPU parity tests: decoding the library's NVFP4 blobs into
logical code arrays (the layout documented in apa_internal.h / include/apa.h),
running the CUDA path on numpy inputs, and the comparison metrics."""
import numpy as np

from mixed_precision_attention_gb300 import synth

TILE = 64


def blob_bytes(d):
    return 64 * d + 1024 * ((d + 127) // 128)


def decode_kv_blob(blob, B, Hkv, Nkv, d):
    """-> kcodes [B,Hkv,T*64,d], ksf [B,Hkv,T*64,d/16], vcodes [B,Hkv,d,T*64], vsf [B,Hkv,d,T*4]."""
    T = (Nkv + TILE - 1) // TILE
    bb = blob_bytes(d)
    x = np.asarray(blob, np.uint8).reshape(B, Hkv, T, bb)
    # K codes: key n, byte x -> elements 2x (low nibble), 2x+1 (high)
    n = np.arange(64)[:, None]
    xb = np.arange(d // 2)[None, :]
    off = (n // 8) * (4 * d) + (xb // 16) * 128 + (n % 8) * 16 + xb % 16
    kb = x[..., off]  # [B,Hkv,T,64,d/2]
    kcodes = np.stack([kb & 15, kb >> 4], -1).reshape(B, Hkv, T * 64, d)
    cb = np.arange(d // 16)[None, :]
    kbk, k16 = cb // 4, cb % 4
    soff = 64 * d + (kbk // 2) * 512 + (n % 32) * 16 + ((n // 32) + 2 * (kbk % 2)) * 4 + k16
    ksf = x[..., soff].reshape(B, Hkv, T * 64, d // 16)
    # V^T codes: channel c, byte x -> keys 2x, 2x+1 of the tile
    c = np.arange(d)[:, None]
    xv = np.arange(32)[None, :]
    voff = 32 * d + (c // 8) * 256 + (xv // 16) * 128 + (c % 8) * 16 + xv % 16
    vb = x[..., voff]  # [B,Hkv,T,d,32]
    vcodes = np.stack([vb & 15, vb >> 4], -1).reshape(B, Hkv, T, d, 64).transpose(0, 1, 3, 2, 4).reshape(B, Hkv, d, T * 64)
    k16v = np.arange(4)[None, :]
    r = c % 128
    vsoff = 64 * d + 512 * ((d + 127) // 128) + (c // 128) * 512 + (r % 32) * 16 + (r // 32) * 4 + k16v
    vsf = x[..., vsoff].transpose(0, 1, 3, 2, 4).reshape(B, Hkv, d, T * 4)
    return kcodes, ksf, vcodes, vsf


def decode_q_blob(blob, B, Hq, Hkv, Nq, d):
    """-> codes [B,Hq,Nq,d], sf [B,Hq,Nq,d/16], and the padding rows' codes / scales."""
    G = Hq // Hkv
    R = G * Nq
    nblk = (R + 127) // 128
    qb = 72 * d
    x = np.asarray(blob, np.uint8).reshape(B, Hkv, nblk, qb)
    p = np.arange(128)[:, None]
    xb = np.arange(d // 2)[None, :]
    off = (p // 8) * (4 * d) + (xb // 16) * 128 + (p % 8) * 16 + xb % 16
    cbytes = x[..., off]  # [B,Hkv,nblk,128,d/2]
    codes = np.stack([cbytes & 15, cbytes >> 4], -1).reshape(B, Hkv, nblk * 128, d)
    cb = np.arange(d // 16)[None, :]
    soff = 64 * d + (cb // 4) * 512 + (p % 32) * 16 + (p // 32) * 4 + cb % 4
    sf = x[..., soff].reshape(B, Hkv, nblk * 128, d // 16)
    # unpack rows p = pos*G + g -> head h*G + g, position pos
    out_c = codes[:, :, :R].reshape(B, Hkv, Nq, G, d).transpose(0, 1, 3, 2, 4).reshape(B, Hq, Nq, d)
    out_s = sf[:, :, :R].reshape(B, Hkv, Nq, G, d // 16).transpose(0, 1, 3, 2, 4).reshape(B, Hq, Nq, d // 16)
    return out_c, out_s, codes[:, :, R:], sf[:, :, R:]


def to_dev(a, dev="cuda"):
    return synth.to_torch_bf16(a, dev)


def run_apa(q, k, v, causal=True, eps=0.005, hot_mask=True, **options):
    import mixed_precision_attention_gb300 as apa
    out, lse, mask = apa.attention(to_dev(q), to_dev(k), to_dev(v), causal=causal, eps=eps, return_hot_mask=hot_mask,
                                   **options)
    apa.check_error()
    return (out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64),
            None if mask is None else mask.cpu().numpy().view(np.uint32))


def cosine(a, b):
    a, b = np.asarray(a, np.float64).ravel(), np.asarray(b, np.float64).ravel()
    return float(a @ b / np.linalg.norm(a) / np.linalg.norm(b))


def hot_bits(mask, T):
    m = np.ascontiguousarray(mask, np.uint32)
    bits = np.unpackbits(m.view(np.uint8), bitorder="little").reshape(m.shape[:-1] + (-1,))
    return bits[..., :T].astype(bool)


def group_visible(Hq, Hkv, Nq, Nkv, causal, ng, T):
    """[ng, T] bool: tile t has a key visible to some row of 16-row group g."""
    G = Hq // Hkv
    R = G * Nq
    vis = np.zeros((ng, T), bool)
    for g in range(ng):
        last_row = min(R, (g + 1) * 16) - 1
        last = (last_row // G + Nkv - Nq) if causal else Nkv - 1
        vis[g, : min(T, last // 64 + 1)] = True
    return vis
