"""Pins for the oracle's FP4 encoding of P and its frames (CPU only).

Pass 1 of "APA: sloppy attention, exact where it counts" encodes P directly in
FP4 ("Pass 1: FP4 everywhere, with a hot test", step 2: one scale per 16-key
group, folded into the exponent bias), with UE4M3 group scales that put each
group maximum near 6 ("Second hunt"), the scale exponent clamped at -6 ("The
bug: a sink that drowned the tail"), a lazy maximum with tau = 4 ("Lazy
maximum") and the decoupled cold frame max(m, c - 32) of a hot tile ("The bug").

The expected values below are worked out by hand from those rules (the
derivation is in the comments), not by re-running the oracle's formulas.  Each
plausible mistake is then planted in a copy of the oracle's source, and a pin
must reject it.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

import oracle
from mixed_precision_attention_gb300 import synth

NEG = -math.inf


def _row(groups):
    """64 scores from four lists of up to 16 (the rest of each group -inf)."""
    s = np.full(64, NEG)
    for k, vals in enumerate(groups):
        s[16 * k:16 * k + len(vals)] = vals
    return s


# Row A, frame m = 0 (tile max 0 <= m + 4: the frame stays 0).
#   group 0, max 0:    2^0 / 6 = 0.16667 = 1.333 * 2^-3 -> UE4M3 1.375 * 2^-3 = 0.171875
#     s =  0: 1      / 0.171875 = 5.818 -> E2M1 6   -> 6   * 0.171875 = 1.03125
#     s = -1: 0.5    / 0.171875 = 2.909 -> 3        -> 0.515625
#     s = -2: 0.25   / 0.171875 = 1.455 -> 1.5      -> 0.2578125
#     s = -3: 0.125  / 0.171875 = 0.727 -> 0.5      -> 0.0859375
#     s = -4: 0.0625 / 0.171875 = 0.364 -> 0.5      -> 0.0859375
#     s = -5: 0.03125/ 0.171875 = 0.182 -> 0        -> 0
#   group 1, max -3:   2^-3 / 6 = 0.020833 = 1.333 * 2^-6 -> 1.375 * 2^-6 = 0.021484375 (>= 2^-6)
#     s = -3:   0.125    / 0.021484375 = 5.818 -> 6 -> 0.12890625
#     s = -3.5: 0.088388 / 0.021484375 = 4.114 -> 4 -> 0.0859375
#     s = -6:   0.015625 / 0.021484375 = 0.727 -> 0.5 -> 0.0107421875
#   group 2, max -5:   2^-5 / 6 = 0.0052083 < 2^-6: nearest UE4M3 is the subnormal
#                      3 * 2^-9, clamped up to 2^-6 = 0.015625
#     s = -5: 0.03125    / 0.015625 = 2    -> 2            -> 0.03125
#     s = -7: 0.0078125  / 0.015625 = 0.5  -> 0.5          -> 0.0078125
#     s = -8: 0.00390625 / 0.015625 = 0.25 -> tie of 0 and 0.5: the even code 0 -> 0
#   group 3, max -7.5: 2^-7.5 / 6 = 0.00092 -> nearest UE4M3 0, clamped to 2^-6
#     s = -7.5: 0.0055243 / 0.015625 = 0.354 -> 0.5 -> 0.0078125
#     s = -9:   0.0019531 / 0.015625 = 0.125 -> 0   -> 0
ROW_A = _row([[0, -1, -2, -3, -4, -5], [-3, -3.5, -6], [-5, -7, -8], [-7.5, -9]])
ROW_A_SC = [0.171875, 0.021484375, 0.015625, 0.015625]
ROW_A_P = _row([[1.03125, 0.515625, 0.2578125, 0.0859375, 0.0859375, 0.0],
                [0.12890625, 0.0859375, 0.0107421875], [0.03125, 0.0078125, 0.0], [0.0078125, 0.0]])
ROW_A_P[np.isinf(ROW_A_P)] = 0.0

# Row B, lazy maximum, frame m = 10:
#   max 13.9 <= 10 + 4: frame stays 10.  2^3.9 / 6 = 2.488 = 1.244 * 2 -> UE4M3 1.25 * 2 = 2.5
#     s = 13.9: 14.929 / 2.5 = 5.97 -> 6   -> 15
#     s = 10:   1      / 2.5 = 0.4  -> 0.5 -> 1.25
#   max 14 = 10 + 4 exactly: not more than tau above, the frame stays 10 (2^4/6 = 2.667
#     = 1.333 * 2 -> 1.375 * 2 = 2.75; 16 / 2.75 = 5.82 -> 6 -> 16.5)
#   max 14.1 > 14: the frame moves to 14.1.  Group scale 2^0 / 6 -> 0.171875
#     s = 14.1: 1 / 0.171875 = 5.818 -> 6 -> 1.03125
#     s = 10:   2^-4.1 / 0.171875 = 0.339 -> 0.5 -> 0.0859375
LAZY = [
    (13.9, 10.0, 2.5, [15.0, 1.25]),
    (14.0, 10.0, 2.75, [16.5, 1.375]),
    (14.1, 14.1, 0.171875, [1.03125, 0.0859375]),
]


def check_p_pins(p_tile):
    """Runs every hand-computed case through p_tile(s, m, tau) -> (c, mt, sc[4], p[64], ell);
    returns the list of the pins that failed (empty when all hold)."""
    bad = []
    c, mt, sc, p, ell = p_tile(ROW_A, 0.0, 4.0)
    if not (c == 0.0 and mt == 0.0):
        bad.append(f"row A frame: c={c} mt={mt}")
    if not np.array_equal(sc, ROW_A_SC):
        bad.append(f"row A group scales {sc}")
    if not np.array_equal(p, ROW_A_P):
        bad.append("row A P values")
    if ell != ROW_A_P.sum():
        bad.append(f"row A tile sum {ell} != {ROW_A_P.sum()}")
    for top, mt_want, sc_want, p_want in LAZY:
        s = _row([[top, 10.0]])
        c, mt, sc, p, ell = p_tile(s, 10.0, 4.0)
        if mt != mt_want:
            bad.append(f"lazy max: tile max {top} over m=10 gives frame {mt}, want {mt_want}")
        if sc[0] != sc_want or not np.array_equal(p[:2], p_want) or p[2:].any():
            bad.append(f"lazy max {top}: scale {sc[0]} P {p[:2]}")
    # first tile of a row (m = -inf): the frame is the tile maximum
    c, mt, sc, p, ell = p_tile(_row([[2.0]]), NEG, 4.0)
    if not (mt == 2.0 and p[0] == 1.03125 and ell == 1.03125):
        bad.append(f"first tile: frame {mt} P {p[0]}")
    # a tile the row does not see: no frame move, no mass
    c, mt, sc, p, ell = p_tile(np.full(64, NEG), 3.0, 4.0)
    if not (c == NEG and mt == 3.0 and ell == 0.0 and not p.any()):
        bad.append("empty tile")
    return bad


def _p_tile_of(lib):
    lib.oracle_p_tile.argtypes = [ctypes.c_void_p, ctypes.c_double, ctypes.c_double, ctypes.c_int] + \
        [ctypes.c_void_p] * 4
    lib.oracle_p_tile.restype = ctypes.c_double

    def f(s, m, tau):
        s = np.ascontiguousarray(s, np.float64)
        c, mt = ctypes.c_double(), ctypes.c_double()
        sc, p = np.empty(4), np.empty(64)
        ell = lib.oracle_p_tile(s.ctypes.data_as(ctypes.c_void_p), m, tau, 1, ctypes.byref(c), ctypes.byref(mt),
                                sc.ctypes.data_as(ctypes.c_void_p), p.ctypes.data_as(ctypes.c_void_p))
        if not (np.all(np.isfinite(p)) and np.all(np.isfinite(sc)) and math.isfinite(ell)):
            return c.value, mt.value, np.full(4, np.nan), np.full(64, np.nan), math.nan
        return c.value, mt.value, sc, p, ell
    return f


def test_p_encoding_hand_computed_rows():
    def f(s, m, tau):
        r = oracle.p_tile(s, m, tau)
        return r["c"], r["mt"], r["sc"], r["p"], r["ell"]
    assert check_p_pins(f) == []


def test_default_tau_and_offset_are_the_pages(golden):
    assert oracle.TAU == golden["lazy_max_tau_log2"]
    assert oracle.COLD_OFFSET == golden["cold_frame_offset"]


def _frame_violations(frame, hot, order_of_group):
    """Re-derives every (row, tile) frame of the emulation from the page's rules:
    m~ = c if c > m + 4 else m; after a hot tile m' = max(m, c - 32), after a cold one
    m' = m~.  Returns the number of violations and the number of checked (row, tile)."""
    bad = n = 0
    for grp in range(frame.shape[0]):
        for rr in range(frame.shape[1]):
            m = NEG
            for t in order_of_group(grp):
                c, mt, after = frame[grp, rr, t]
                if np.isnan(c):
                    continue
                n += 1
                want_mt = c if c > m + 4.0 else m
                want_after = max(m, c - 32.0) if hot[grp, t] else want_mt
                bad += (mt != want_mt) + (after != want_after)
                m = after
    return bad, n


def _small_case():
    w = synth.small(B=1, Hq=2, Hkv=1, Nq=32, Nkv=8192, d=64, sink_gain=8.0, n_outliers=2, seed=3)
    q, k, v = synth.generate(w)
    return w, q, k, v


def _order(w):
    G, off = w.Hq // w.Hkv, w.Nkv - w.Nq

    def order_of_group(grp):
        rows = oracle.group_rows(w.Hq, w.Hkv, w.Nq, 0, 0, grp)
        tmax = max(p + off for _, _, p in rows) // 64
        return [0] + list(range(tmax, 0, -1))
    return order_of_group


def _bits(mask, T):
    m = np.ascontiguousarray(mask, np.uint32)
    return np.unpackbits(m.view(np.uint8), bitorder="little").reshape(m.shape[:-1] + (-1,))[..., :T].astype(bool)


def test_frames_follow_lazy_max_and_cold_frame():
    w, q, k, v = _small_case()
    r = oracle.apa(q, k, v, eps=0.005, diag=True)
    T = w.Nkv // 64
    hot = _bits(r["hot_mask"][0, 0], T)
    bad, n = _frame_violations(r["frame"], hot, _order(w))
    assert n > 1000 and bad == 0
    # the case exercises both commit rules: frames moved by hot and by cold tiles
    moved_hot = moved_cold = 0
    for grp in range(hot.shape[0]):
        for t in range(T):
            f = r["frame"][grp, :, t]
            seen = ~np.isnan(f[:, 0])
            moved = seen & (f[:, 1] != f[:, 2])
            moved_hot += int(moved.sum()) if hot[grp, t] else 0
            moved_cold += int((seen & (f[:, 1] == f[:, 0])).sum()) if not hot[grp, t] else 0
    assert moved_hot > 0 and moved_cold > 0


# ----------------------------------------------------------------------------- planted mistakes
ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "apa_oracle.c")

_TRUNC_HELPERS = """
static int e2m1_code_truncated(double x) {  /* planted: rounds down instead of to nearest */
  double a = fabs(x); int c = 0;
  const double v[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  for (int i = 0; i < 8; ++i) if (a >= v[i]) c = i;
  return c;
}
static int ue4m3_code_truncated(double x) {  /* planted: rounds the scale down */
  int c = oracle_ue4m3_code(x);
  if (oracle_ue4m3_value(c) > x && c > 0) --c;
  return c;
}
double oracle_p_tile("""

MUTANTS = {
    # the group scale puts the maximum near 4 instead of 6
    "scale /4": [("exp2(g[kg] - mtl) / 6.0", "exp2(g[kg] - mtl) / 4.0")],
    # no clamp of the group scale: a far-below group gets scale 0
    "no clamp": [("      if (sck < P_SCALE_MIN) sck = P_SCALE_MIN;\n", "")],
    # the clamp at the smallest subnormal 2^-9 instead of 2^-6
    "clamp 2^-9": [("#define P_SCALE_MIN 0.015625", "#define P_SCALE_MIN 0.001953125")],
    # E2M1 of P rounded down instead of to nearest even
    "P truncated": [("double oracle_p_tile(", _TRUNC_HELPERS),
                    ("oracle_e2m1_value(oracle_e2m1_code(x / sck))", "oracle_e2m1_value(e2m1_code_truncated(x / sck))")],
    # UE4M3 group scale rounded down
    "scale truncated": [("double oracle_p_tile(", _TRUNC_HELPERS),
                        ("oracle_ue4m3_value(oracle_ue4m3_code(exp2(g[kg] - mtl) / 6.0))",
                         "oracle_ue4m3_value(ue4m3_code_truncated(exp2(g[kg] - mtl) / 6.0))")],
    # lazy maximum with tau = 2
    "tau 2": [("double mtl = (c > m + tau) ? c : m;", "double mtl = (c > m + 0.5 * tau) ? c : m;")],
    # a frame move at exactly tau above (>= instead of >)
    "tau inclusive": [("double mtl = (c > m + tau) ? c : m;", "double mtl = (c >= m + tau) ? c : m;")],
    # the tile sum taken over the unquantized P
    "sum unquantized": [("      p[jj] = pj;\n      sum += pj;", "      p[jj] = pj;\n      sum += s[jj] != -INFINITY ? exp2(s[jj] - mtl) : 0.0;")],
    # a hot tile lifts the frame to its maximum (the 0.2.0 frame)
    "hot lifts to c": [("mn = fmax(m[r], c - P->cold_offset);", "mn = fmax(m[r], c);")],
    # a cold tile keeps the old frame instead of the candidate one
    "cold keeps m": [("        mn = mt[r];\n", "        mn = m[r];\n")],
}


def _build_mutant(tmp_path, name, edits):
    src = open(ORACLE_SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new if old != "double oracle_p_tile(" else new)
    path = tmp_path / (name.replace(" ", "_").replace("/", "div").replace("^", "") + ".c")
    path.write_text(src)
    so = str(path)[:-2] + ".so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           str(path), "-o", so, "-lm"])
    return ctypes.CDLL(so)


def _apa_frames(lib, w, q, k, v, eps=0.005):
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_apa.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, f64, f64, f64, i32, P, i64,
                               P, P, P, P, P, P]
    lib.oracle_apa.restype = i32
    B, Hq, Nq, d = q.shape
    Hkv, Nkv = k.shape[1], k.shape[2]
    T = (Nkv + 63) // 64
    ng = oracle.n_groups(Hq, Hkv, Nq)
    out = np.full((B, Hq, Nq, d), np.nan)
    lse = np.full((B, Hq, Nq), np.nan)
    hot = np.zeros((B, Hkv, ng, (T + 31) // 32), np.uint32)
    frame = np.full((B * Hkv * ng, 16, T, 3), np.nan)
    qq, kk, vv = (np.ascontiguousarray(a, np.uint16) for a in (q, k, v))
    ptr = lambda a: a.ctypes.data_as(P)  # noqa: E731
    rc = lib.oracle_apa(ptr(qq), ptr(kk), ptr(vv), B, Hq, Hkv, Nq, Nkv, d, 1, eps, 4.0, 32.0, 15, None, 0,
                        ptr(out), ptr(lse), ptr(hot), None, None, ptr(frame))
    assert rc == 0
    return frame, _bits(hot[0, 0], T)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name, MUTANTS[name])
    failures = check_p_pins(_p_tile_of(lib))
    if not failures:
        # mistakes in the frame commit show up in the emulation's frames
        w, q, k, v = _small_case()
        frame, hot = _apa_frames(lib, w, q, k, v)
        bad, n = _frame_violations(frame, hot, _order(w))
        failures = [f"{bad} frame violations"] if bad else []
    assert failures, f"planted mistake '{name}' passed every pin"


def test_unmutated_copy_passes(tmp_path):
    # the mutation harness itself: an unmodified copy passes every pin
    lib = _build_mutant(tmp_path, "identity", [])
    assert check_p_pins(_p_tile_of(lib)) == []
    w, q, k, v = _small_case()
    frame, hot = _apa_frames(lib, w, q, k, v)
    assert _frame_violations(frame, hot, _order(w))[0] == 0
