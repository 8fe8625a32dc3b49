"""Pins of the oracle's FP4 (E2M1) weight format, on the CPU.

Format: "LLM Compressor 0.14: GPTQ's 15x speedup is one fused loop", section "Details worth
knowing": rounding onto {0, 0.5, 1, 1.5, 2, 3, 4, 6} through a ladder of thresholds whose
comparisons alternate so that ties go to the even code.  The checks below are independent of the
oracle's ladder: the E2M1 bit formula, nearest-value search in exact rational arithmetic, and a
hand-built fixture.
"""
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest

import oracle
from tests._exact import fl16, fl32

GOLDEN = Path(__file__).parent / "golden"


def _rows(name):
    out = []
    for line in (GOLDEN / name).read_text().splitlines():
        if line.startswith("#") or not line.strip():
            continue
        out.append([f.strip() for f in line.split("|")])
    return out


def _e2m1(code: int) -> Fraction:
    """E2M1 bit layout: sign bit 3, exponent bits 1-2 (bias 1), mantissa bit 0; exponent 0 is
    subnormal (m * 1/2)."""
    sgn = -1 if code & 8 else 1
    e, m = (code >> 1) & 3, code & 1
    mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return sgn * mag


def _nearest_even(r: Fraction) -> int:
    """Index of the grid value nearest to |r| by exhaustive search, a tie going to the even
    index; magnitudes past 6 give index 7."""
    grid = [_e2m1(i) for i in range(8)]
    m = abs(r)
    best = None
    for i, g in enumerate(grid):
        d = abs(m - g)
        if best is None or d < best[0] or (d == best[0] and i % 2 == 0):
            best = (d, i)
    return best[1]


def test_fp4_grid_is_e2m1():
    g = oracle.fp4_grid()
    assert [Fraction(float(v)) for v in g] == [_e2m1(i) for i in range(8)]
    codes = np.arange(16, dtype=np.uint8).reshape(1, 16)
    packed = oracle.pack(np.concatenate([codes, codes], axis=1))
    wh = oracle.dequantize_fp4(packed, np.ones((1, 1), np.float16), 32)[0, :16]
    for c in range(16):
        assert Fraction(float(wh[c])) == _e2m1(c), c
    assert np.signbit(wh[8]) and not np.signbit(wh[0])


def test_fp4_golden_on_grid():
    for e, chex in _rows("fp4_on_grid.txt"):
        codes = [int(ch, 16) for ch in chex]
        w = np.array([[float(_e2m1(c)) * 2.0 ** int(e) for c in codes]], np.float32)
        packed, scale = oracle.quantize_fp4(w, 32)
        assert packed.tobytes().hex() == chex
        assert scale.dtype == np.float16 and float(scale[0, 0]) == 2.0 ** int(e)
        assert np.array_equal(oracle.dequantize_fp4(packed, scale, 32), w)


def test_fp4_ties_go_to_even_code():
    """Every midpoint, written out: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2,
    3.5 -> 4, 5 -> 4 (grid values), with either sign."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    expect = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    w = np.zeros((1, 32), np.float32)
    w[0, :7] = mids
    w[0, 7:14] = [-m for m in mids]
    w[0, 31] = 6.0                                           # scale exactly 1
    packed, scale = oracle.quantize_fp4(w, 32)
    wh = oracle.dequantize_fp4(packed, scale, 32)[0]
    assert float(scale[0, 0]) == 1.0
    assert wh[:7].tolist() == expect
    assert wh[7:14].tolist() == [-v for v in expect]


def test_fp4_ladder_equals_nearest_search():
    """Magnitudes on, one FP32 step either side of, and between every midpoint, plus random ones
    and some past 6, at scale 1: the code equals the exhaustive nearest search."""
    vals = []
    g = [float(v) for v in oracle.fp4_grid()]
    for i in range(7):
        t = np.float32((g[i] + g[i + 1]) / 2)
        vals += [t, np.nextafter(t, np.float32(0)), np.nextafter(t, np.float32(10)), np.float32(g[i])]
    rng = np.random.default_rng(41)
    vals += list(rng.uniform(0, 6, 200).astype(np.float32))
    vals += [np.float32(6.0), np.float32(6.25), np.nextafter(np.float32(6), np.float32(7))]
    vals = np.array(vals, np.float32)
    n = len(vals)
    per = 31
    groups = (n + per - 1) // per
    w = np.zeros((groups, 32), np.float32)
    for gi in range(groups):
        chunk = vals[gi * per:(gi + 1) * per]
        w[gi, :len(chunk)] = chunk * (1 if gi % 2 == 0 else -1)
        w[gi, 31] = 6.0
    w = np.clip(w, -6.0, 6.0)                                 # keep absmax 6, scale 1
    w[-1, :3] = [6.0, 6.0, 6.0]
    packed, scale = oracle.quantize_fp4(w, 32)
    assert np.all(scale.astype(np.float64) == 1.0)
    q = oracle.unpack(packed)
    for gi in range(groups):
        for k in range(32):
            r = Fraction(float(w[gi, k]))
            exp = _nearest_even(r) | (8 if r < 0 else 0)
            assert int(q[gi, k]) == exp, (gi, k, float(w[gi, k]))


def test_fp4_past_six_clamps():
    """A group whose FP16 scale rounds below absmax / 6 holds |r| slightly above 6: index 7."""
    rng = np.random.default_rng(43)
    hits = 0
    for a in np.abs(rng.standard_normal(400) * 0.1).astype(np.float32):
        s = fl16(Fraction(float(a)) / 6)
        if s == 0 or fl32(Fraction(float(a)) / s) <= 6:
            continue
        w = np.zeros((1, 32), np.float32)
        w[0, 0] = a
        w[0, 1] = -a
        packed, scale = oracle.quantize_fp4(w, 32)
        q = oracle.unpack(packed)[0]
        assert q[0] == 7 and q[1] == 15
        hits += 1
    assert hits > 20


def test_fp4_scale_is_fp16_of_absmax_over_6():
    rng = np.random.default_rng(44)
    a = np.abs(rng.standard_normal(2000) * 0.05).astype(np.float32)
    a = np.concatenate([a, np.float32([6 * 2.0 ** -20, 6 * 2.0 ** -26, 1e-9, 0.0, 3.0e5])])
    w = np.zeros((len(a), 32), np.float32)
    w[:, 5] = -a
    _, scale = oracle.quantize_fp4(w, 32)
    for i, ai in enumerate(a):
        assert Fraction(float(scale[i, 0])) == fl16(Fraction(float(ai)) / 6), i


def test_fp4_rounding_brute_force_and_bound():
    """Every code by exact rational arithmetic (IEEE FP32 quotient, then nearest search), and the
    error bound: half the gap between the grid values around |r|, times s."""
    rng = np.random.default_rng(45)
    w = (rng.standard_normal((3, 128)) * 0.02).astype(np.float32)
    w[1, 32:64] = 0.0
    w[2, 5] = -0.0
    packed, scale = oracle.quantize_fp4(w, 32)
    q = oracle.unpack(packed).astype(int)
    wh = oracle.dequantize_fp4(packed, scale, 32)
    g = [_e2m1(i) for i in range(8)]
    for r_ in range(3):
        for k in range(128):
            s = Fraction(float(scale[r_, k // 32]))
            wk = Fraction(float(w[r_, k]))
            if s == 0:
                exp = 0
                assert wh[r_, k] == 0
            else:
                exp = _nearest_even(fl32(wk / s)) | (8 if w[r_, k] < 0 else 0)
            assert q[r_, k] == exp, (r_, k)
            if s != 0:
                m = abs(fl32(wk / s))
                i = max(j for j in range(8) if g[j] <= min(m, Fraction(6)))
                gap = (g[i + 1] - g[i]) if i < 7 else Fraction(0)
                bound = (gap / 2 + max(Fraction(0), m - 6) + m * Fraction(1, 2 ** 23)) * s
                assert abs(wk - Fraction(float(wh[r_, k]))) <= bound, (r_, k)
    assert q[1, 32:64].tolist() == [0] * 32 and float(scale[1, 1]) == 0.0
    assert q[2, 5] == 0


def test_fp4_requantize_is_identity():
    """Quantising the dequantised matrix again gives the same codes and scales."""
    rng = np.random.default_rng(46)
    w = (rng.standard_normal((6, 256)) * 0.02).astype(np.float32)
    packed, scale = oracle.quantize_fp4(w, 32)
    wh = oracle.dequantize_fp4(packed, scale, 32)
    wh[wh == 0] = 0.0                                         # -0 dequantises from code 8 only
    p2, s2 = oracle.quantize_fp4(wh, 32)
    assert np.array_equal(s2, scale)
    q1, q2 = oracle.unpack(packed), oracle.unpack(p2)
    assert np.array_equal(np.where(q1 == 8, 0, q1), q2)


@pytest.mark.parametrize("group", [32, 64, 128])
def test_fp4_gemv_brute_force_exact(group):
    rng = np.random.default_rng(47)
    w = (rng.standard_normal((3, 128)) * 0.02).astype(np.float32)
    x = rng.standard_normal((2, 128)).astype(np.float16)
    packed, scale = oracle.quantize_fp4(w, group)
    y = oracle.gemv_fp4(packed, scale, x, group)
    q = oracle.unpack(packed)
    for m in range(2):
        for n in range(3):
            acc = Fraction(0)
            for k in range(128):
                acc += _e2m1(int(q[n, k])) * Fraction(float(scale[n, k // group])) * Fraction(float(x[m, k]))
            assert abs(Fraction(float(y[m, n])) - acc) <= Fraction(1, 2 ** 45) * max(Fraction(1), abs(acc)), (m, n)
    rows = np.array([2, 0])
    assert np.array_equal(oracle.gemv_fp4(packed, scale, x, group, rows=rows), y[:, rows])
