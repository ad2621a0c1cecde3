"""CPU oracle for adaptive-precision attention -- TEST INFRASTRUCTURE ONLY.

A plain FP64 statement of the method of "APA: sloppy attention, exact where it
counts" (rfriedmann.de blog) in ``apa_oracle.c``, loaded through ctypes.  Only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  It shares no code with the CUDA path
(``mixed_precision_attention_gb300``); both are fed by the seeded generator in
``mixed_precision_attention_gb300.synth``, which holds no attention arithmetic.

Every array in and out is numpy.  bf16 inputs are uint16 bit arrays in BHSD
layout: q [B, Hq, Nq, d], k and v [B, Hkv, Nkv, d].
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "apa_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

QUANT_Q, QUANT_K, QUANT_V, QUANT_P = 1, 2, 4, 8
QUANT_ALL = 15
QUANT_Q2 = 16  # Q as two FP4 terms, Q1 + FP4(Q - Q1) (needs QUANT_Q)
QUANT_LSE = 32  # least-squared-error block scales for Q, K and V
QUANT_VWEIGHT = 64  # value-norm-weighted hot test (not a quantization)
TILE = 64
GROUP_ROWS = 16


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (FP contraction off, so x86 and Arm agree)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                               "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_e2m1_code.argtypes = [f64]; lib.oracle_e2m1_code.restype = i32
            lib.oracle_e2m1_value.argtypes = [i32]; lib.oracle_e2m1_value.restype = f64
            lib.oracle_ue4m3_code.argtypes = [f64]; lib.oracle_ue4m3_code.restype = i32
            lib.oracle_ue4m3_value.argtypes = [i32]; lib.oracle_ue4m3_value.restype = f64
            lib.oracle_head_scale.argtypes = [f64]; lib.oracle_head_scale.restype = f64
            lib.oracle_quantize_blocks.argtypes = [P, i64, f64, P, P]; lib.oracle_quantize_blocks.restype = None
            lib.oracle_key_mean.argtypes = [P, i32, i32, P]; lib.oracle_key_mean.restype = None
            lib.oracle_merge.argtypes = [f64, f64, P, f64, f64, P, i32, P]; lib.oracle_merge.restype = f64
            lib.oracle_exact.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, P, i64, P, P]
            lib.oracle_exact.restype = None
            lib.oracle_quantize_kv_head.argtypes = [P, P, i32, i32, P, P, P, P, P, P, P, i32]
            lib.oracle_quantize_kv_head.restype = None
            lib.oracle_quantize_q_head.argtypes = [P, i32, i32, P, P, P, P, P, i32]
            lib.oracle_quantize_residual_blocks.argtypes = [P, i64, f64, P, P, P, P, i32]
            lib.oracle_quantize_blocks_mode.argtypes = [P, i64, f64, P, P, i32]
            lib.oracle_value_weights.argtypes = [P, i32, i32, P]
            lib.oracle_value_weights.restype = None
            lib.oracle_quantize_blocks_mode.restype = None
            lib.oracle_quantize_residual_blocks.restype = None
            lib.oracle_quantize_q_head.restype = None
            lib.oracle_apa.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, f64, f64, f64, i32,
                                       P, i64, P, P, P, P, P, P]
            lib.oracle_p_tile.argtypes = [P, f64, f64, i32, P, P, P, P]
            lib.oracle_p_tile.restype = f64
            lib.oracle_apa.restype = i32
            lib.oracle_num_threads.argtypes = []; lib.oracle_num_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def num_threads() -> int:
    return _load().oracle_num_threads()


# ----------------------------------------------------------------- formats
def e2m1_code(x: float) -> int:
    return _load().oracle_e2m1_code(float(x))


def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def ue4m3_code(x: float) -> int:
    return _load().oracle_ue4m3_code(float(x))


def ue4m3_value(code: int) -> float:
    return _load().oracle_ue4m3_value(int(code))


def head_scale(amax: float) -> float:
    return _load().oracle_head_scale(float(amax))


def quantize_blocks(x: np.ndarray, s: float, lse: bool = False):
    """Quantizes float32 values in blocks of 16 (last axis) with head scale s;
    lse: least-squared-error block scales instead of the nearest ones.

    Returns (codes uint8 same shape as x, sf uint8 with the last axis / 16)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape[-1] % 16 == 0
    codes = np.empty(x.shape, dtype=np.uint8)
    sf = np.empty(x.shape[:-1] + (x.shape[-1] // 16,), dtype=np.uint8)
    _load().oracle_quantize_blocks_mode(_ptr(x), x.size // 16, float(s), _ptr(codes), _ptr(sf), int(lse))
    return codes, sf


def key_mean(k_head: np.ndarray) -> np.ndarray:
    """Per-channel key mean of one KV head, k_head [Nkv, d] bf16 bits -> float32 [d]."""
    k_head = _u16(k_head)
    Nkv, d = k_head.shape
    mu = np.empty(d, dtype=np.float32)
    _load().oracle_key_mean(_ptr(k_head), Nkv, d, _ptr(mu))
    return mu


def merge(m1, l1, o1, m2, l2, o2):
    """Merges two (m, l, o) states (log2 units).  Returns (out, log2 of merged sum)."""
    o1 = np.ascontiguousarray(o1, dtype=np.float64)
    o2 = np.ascontiguousarray(o2, dtype=np.float64)
    out = np.empty_like(o1)
    lg = _load().oracle_merge(float(m1), float(l1), _ptr(o1), float(m2), float(l2), _ptr(o2), o1.size, _ptr(out))
    return out, lg


# ----------------------------------------------------------------- quantizer
def quantize_kv(k: np.ndarray, v: np.ndarray, lse: bool = False):
    """NVFP4 codes of K (centred) and V^T for every (b, KV head).

    Returns dict with mu [B,Hkv,d] f32, kcodes [B,Hkv,Nkv,d] u8, ksf [B,Hkv,Nkv,d/16],
    s_k [B,Hkv] f64, vcodes [B,Hkv,d,Npad], vsf [B,Hkv,d,Npad/16], s_v [B,Hkv]."""
    k, v = _u16(k), _u16(v)
    B, Hkv, Nkv, d = k.shape
    Npad = (Nkv + 15) // 16 * 16
    r = dict(mu=np.empty((B, Hkv, d), np.float32), kcodes=np.empty((B, Hkv, Nkv, d), np.uint8),
             ksf=np.empty((B, Hkv, Nkv, d // 16), np.uint8), s_k=np.empty((B, Hkv)),
             vcodes=np.empty((B, Hkv, d, Npad), np.uint8), vsf=np.empty((B, Hkv, d, Npad // 16), np.uint8),
             s_v=np.empty((B, Hkv)))
    lib = _load()
    for b in range(B):
        for h in range(Hkv):
            sk, sv = ctypes.c_double(), ctypes.c_double()
            lib.oracle_quantize_kv_head(_ptr(np.ascontiguousarray(k[b, h])), _ptr(np.ascontiguousarray(v[b, h])),
                                        Nkv, d, _ptr(r["mu"][b, h]), _ptr(r["kcodes"][b, h]),
                                        _ptr(r["ksf"][b, h]), ctypes.byref(sk), _ptr(r["vcodes"][b, h]),
                                        _ptr(r["vsf"][b, h]), ctypes.byref(sv), int(lse))
            r["s_k"][b, h], r["s_v"][b, h] = sk.value, sv.value
    return r


def quantize_q(q: np.ndarray, residual: bool = False, lse: bool = False):
    """NVFP4 codes of Q per (b, query head): codes [B,Hq,Nq,d], sf [B,Hq,Nq,d/16], s_q [B,Hq];
    with residual=True also codes2 / sf2, the FP4 residual term Q - Q1 in the same head scale."""
    q = _u16(q)
    B, Hq, Nq, d = q.shape
    codes = np.empty((B, Hq, Nq, d), np.uint8)
    sf = np.empty((B, Hq, Nq, d // 16), np.uint8)
    codes2 = np.empty_like(codes) if residual else None
    sf2 = np.empty_like(sf) if residual else None
    s_q = np.empty((B, Hq))
    lib = _load()
    for b in range(B):
        for h in range(Hq):
            s = ctypes.c_double()
            lib.oracle_quantize_q_head(_ptr(np.ascontiguousarray(q[b, h])), Nq, d, _ptr(codes[b, h]),
                                       _ptr(sf[b, h]), ctypes.byref(s),
                                       _ptr(codes2[b, h]) if residual else None,
                                       _ptr(sf2[b, h]) if residual else None, int(lse))
            s_q[b, h] = s.value
    r = dict(codes=codes, sf=sf, s_q=s_q)
    if residual:
        r.update(codes2=codes2, sf2=sf2)
    return r


def value_weights(v: np.ndarray):
    """Value-norm weight of every 64-key tile per (b, KV head): [B, Hkv, T] float32."""
    v = _u16(v)
    B, Hkv, Nkv, d = v.shape
    T = (Nkv + TILE - 1) // TILE
    w = np.empty((B, Hkv, T), np.float32)
    lib = _load()
    for b in range(B):
        for h in range(Hkv):
            lib.oracle_value_weights(_ptr(np.ascontiguousarray(v[b, h])), Nkv, d, _ptr(w[b, h]))
    return w


# ----------------------------------------------------------------- attention
def exact(q, k, v, causal=True, rows=None):
    """Exact FP64 attention.  rows: optional int array [n, 3] of (b, hq, pos).

    Returns (out [B,Hq,Nq,d] f64, lse [B,Hq,Nq] f64, natural log); rows that
    were not asked for are NaN."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    out = np.full((B, Hq, Nq, d), np.nan)
    lse = np.full((B, Hq, Nq), np.nan)
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    _load().oracle_exact(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d, int(causal), _ptr(r),
                         0 if r is None else len(r), _ptr(out), _ptr(lse))
    return out, lse


def n_groups(Hq, Hkv, Nq):
    return ((Hq // Hkv) * Nq + GROUP_ROWS - 1) // GROUP_ROWS


TAU = 4.0           # lazy-maximum threshold, log2 units ("Lazy maximum")
COLD_OFFSET = 32.0  # a hot tile lifts the frame at most to c - 32 ("The bug", the decoupled cold frame)


def p_tile(s, m, tau=TAU, quantize=True):
    """P of one row over one 64-key tile, encoded in FP4 as pass 1 does.

    s: 64 scores in log2 units (-inf = not visible); m: the row's frame before
    the tile.  Returns dict(c=tile max, mt=frame P is computed in, sc=[4] group
    scales, p=[64] dequantized P, ell=sum of p)."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    assert s.shape == (TILE,)
    c, mt = ctypes.c_double(), ctypes.c_double()
    sc = np.empty(TILE // 16)
    p = np.empty(TILE)
    ell = _load().oracle_p_tile(_ptr(s), float(m), float(tau), int(quantize), ctypes.byref(c), ctypes.byref(mt),
                                _ptr(sc), _ptr(p))
    return dict(c=c.value, mt=mt.value, sc=sc, p=p, ell=ell)


def apa(q, k, v, causal=True, eps=0.005, tau=TAU, cold_offset=COLD_OFFSET, quant=QUANT_ALL, units=None,
        diag=False):
    """APA emulation (pass 1, hot test, exact pass 2, merge) in FP64.

    units: optional int array [n, 3] of (b, hkv, group) 16-row groups; None = all.
    Returns dict(out, lse, hot_mask[, ell, lam]); rows of groups not asked for are NaN.
    hot_mask: uint32 [B, Hkv, ceil(R/16), ceil(T/32)], bit t%32 of word t/32.
    ell [n, 16, T]: each row's FP4 tile sum in the row's final frame (NaN = unseen);
    lam [n, 16]: final running sum lambda;
    frame [n, 16, T, 3]: per row and tile seen, the tile maximum c, the frame m~
    its P was computed in, and the row's frame after the tile (NaN = unseen)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    T = (Nkv + TILE - 1) // TILE
    ng = n_groups(Hq, Hkv, Nq)
    out = np.full((B, Hq, Nq, d), np.nan)
    lse = np.full((B, Hq, Nq), np.nan)
    hot = np.zeros((B, Hkv, ng, (T + 31) // 32), np.uint32)
    u = None if units is None else np.ascontiguousarray(units, dtype=np.int32)
    nu = B * Hkv * ng if u is None else len(u)
    ell = np.full((nu, GROUP_ROWS, T), np.nan) if diag else None
    lam = np.full((nu, GROUP_ROWS), np.nan) if diag else None
    frame = np.full((nu, GROUP_ROWS, T, 3), np.nan) if diag else None
    rc = _load().oracle_apa(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nkv, d, int(causal), float(eps),
                            float(tau), float(cold_offset), int(quant), _ptr(u), 0 if u is None else len(u),
                            _ptr(out), _ptr(lse), _ptr(hot), _ptr(ell), _ptr(lam), _ptr(frame))
    if rc != 0:
        raise ValueError("unsupported shape for the oracle")
    r = dict(out=out, lse=lse, hot_mask=hot)
    if diag:
        r["ell"], r["lam"], r["frame"] = ell, lam, frame
    return r


def group_rows(Hq, Hkv, Nq, b, hkv, grp):
    """(b, hq, pos) of the rows of one 16-row group (packed row p = pos*G + g)."""
    G = Hq // Hkv
    R = G * Nq
    return [(b, hkv * G + p % G, p // G) for p in range(grp * GROUP_ROWS, min(R, (grp + 1) * GROUP_ROWS))]
