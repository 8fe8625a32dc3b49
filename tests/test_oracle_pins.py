"""Pins for the CPU oracle: checks against what the pages and mathematics fix,
never against the oracle's own formulas retyped.

Each test names the mistake it would catch.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from weight_only_bit_gb300 import synth
from tests._exact import fl16, fl32, round_half_even

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        if line.startswith("#") or not line.strip():
            continue
        out.append([f.strip() for f in line.split("|")])
    return out


def _codes(hexdigits):
    return np.array([int(ch, 16) for ch in hexdigits], dtype=np.uint8)


# ----------------------------------------------------------------------------- codebook
def test_codebook_structure():
    """Normalised to [-1, 1] with an exact zero: c0 = -1, c7 = 0, c15 = 1, strictly
    increasing, 7 negative and 8 positive values (asymmetric NF4 with one zero)."""
    c = oracle.nf4_codebook()
    assert c.dtype == np.float32 and c.shape == (16,)
    assert c[0] == -1.0 and c[7] == 0.0 and c[15] == 1.0
    assert np.all(np.diff(c.astype(np.float64)) > 0)
    assert (c < 0).sum() == 7 and (c > 0).sum() == 8


def test_codebook_independent_quantile_routine():
    """The same construction through scipy's ndtri (a different inverse-normal
    routine, not the one the oracle calls) gives the same FP32 values."""
    from scipy.special import ndtri
    delta = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0))
    pos = ndtri(np.linspace(delta, 0.5, 9)[:-1])
    neg = -ndtri(np.linspace(delta, 0.5, 8)[:-1])
    v = np.sort(np.concatenate([pos, neg, [0.0]]))
    ref = (v / v.max()).astype(np.float32)
    c = oracle.nf4_codebook()
    ulps = np.abs(c.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1


def test_codebook_quantile_spacing():
    """Each positive code value is Phi^-1 at its probability divided by Phi^-1(delta):
    checked through the forward normal CDF (scipy ndtr), which inverts the quantile."""
    from scipy.special import ndtr, ndtri
    delta = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0))
    c = oracle.nf4_codebook().astype(np.float64)
    top = ndtri(delta)
    p_pos = ndtr(c[8:] * top)[::-1]          # descending values -> probabilities from delta down
    expect = delta + np.arange(8) * (0.5 - delta) / 8.0
    assert np.allclose(p_pos, expect, atol=1e-7)
    p_neg = ndtr(-c[:7] * top)               # c[0] = -1 ... c[6]
    expect_n = delta + np.arange(7) * (0.5 - delta) / 7.0
    assert np.allclose(p_neg, expect_n, atol=1e-7)


# ----------------------------------------------------------------------------- packing
def test_pack_unpack_all_bytes():
    b = np.arange(256, dtype=np.uint8).reshape(1, 256)
    assert np.array_equal(oracle.pack(oracle.unpack(b)), b)
    q = oracle.unpack(b)
    assert np.array_equal(q[0, 0::2], np.arange(256) >> 4)    # high nibble first
    assert np.array_equal(q[0, 1::2], np.arange(256) & 15)


def test_pack_literal_order():
    """Element 2j in the high nibble: codes (1,2,3,4) pack to bytes 0x12, 0x34."""
    assert oracle.pack(np.array([[1, 2, 3, 4]], np.uint8)).tolist() == [[0x12, 0x34]]


# ----------------------------------------------------------------------------- NF4
def test_nf4_golden_on_grid():
    """Hand-built fixture: weights placed on code points x a power of two quantise to
    the listed codes, pack to the same hex digits, keep absmax = a and dequantise exactly."""
    code = oracle.nf4_codebook()
    for a0, a1, qhex in _rows("nf4_on_grid.txt"):
        q = _codes(qhex).reshape(1, 128)
        a = np.array([[float.fromhex(a0), float.fromhex(a1)]], dtype=np.float32)
        w = (code[q] * np.repeat(a, 64, axis=1)).astype(np.float32)
        packed, absmax = oracle.quantize_nf4(w, code, 64)
        assert packed.tobytes().hex() == qhex
        assert np.array_equal(absmax, a)
        assert np.array_equal(oracle.dequantize_nf4(packed, absmax, code, 64), w)


def _nearest_code_exact(w, a, code):
    """Brute force: n = fl32(w / a) by exact rational rounding; nearest code by exact
    distances; a tie goes to the lower code."""
    if a == 0:
        n = Fraction(0)
    else:
        n = fl32(Fraction(float(w)) / Fraction(float(a)))
    best, best_d = None, None
    for i, c in enumerate(code):
        d = abs(n - Fraction(float(c)))
        if best is None or d < best_d:
            best, best_d = i, d
    return best


def test_nf4_rounding_brute_force():
    rng = np.random.default_rng(1)
    code = oracle.nf4_codebook()
    w = (rng.standard_normal((3, 128)) * 0.02).astype(np.float32)
    w[1, :64] = 0.0                                  # an all-zero block
    w[2, 5] = 0.3                                    # one large value in a block
    packed, absmax = oracle.quantize_nf4(w, code, 64)
    q = oracle.unpack(packed)
    for r in range(3):
        for k in range(128):
            assert q[r, k] == _nearest_code_exact(w[r, k], absmax[r, k // 64], code), (r, k)


def test_nf4_ties_go_to_lower_code():
    """A code book with FP32-exact midpoints: values exactly at a midpoint take the lower code."""
    code = (np.arange(16, dtype=np.float32) - 8) / 8       # -1 ... 0.875
    w = np.zeros((1, 64), np.float32)
    mids = (code[:-1].astype(np.float64) + code[1:]) / 2
    w[0, :15] = mids.astype(np.float32)                    # exact (multiples of 1/16)
    w[0, 15] = -1.0                                        # absmax = 1
    packed, absmax = oracle.quantize_nf4(w, code, 64)
    q = oracle.unpack(packed)[0]
    assert absmax[0, 0] == 1.0
    assert q[:15].tolist() == list(range(15))              # tie -> lower index i, not i+1
    assert q[15] == 0


def test_nf4_absmax_element_maps_to_end_code():
    rng = np.random.default_rng(2)
    code = oracle.nf4_codebook()
    w = (rng.standard_normal((4, 256)) * 0.02).astype(np.float32)
    packed, absmax = oracle.quantize_nf4(w, code, 64)
    q = oracle.unpack(packed).reshape(4, 4, 64)
    blocks = w.reshape(4, 4, 64)
    for r in range(4):
        for b in range(4):
            j = int(np.argmax(np.abs(blocks[r, b])))
            assert absmax[r, b] == np.abs(blocks[r, b]).max()
            assert q[r, b, j] == (15 if blocks[r, b, j] > 0 else 0)


def test_nf4_error_bound():
    """|w - w_hat| <= a * (largest half-gap of the code book) + rounding."""
    rng = np.random.default_rng(3)
    code = oracle.nf4_codebook()
    w = (rng.standard_normal((8, 512)) * 0.02).astype(np.float32)
    packed, absmax = oracle.quantize_nf4(w, code, 64)
    wh = oracle.dequantize_nf4(packed, absmax, code, 64)
    half_gap = np.max(np.diff(code.astype(np.float64))) / 2
    a = np.repeat(absmax, 64, axis=1).astype(np.float64)
    assert np.all(np.abs(w - wh) <= a * half_gap * (1 + 1e-6) + 1e-12)


# ----------------------------------------------------------------------------- INT4
def test_int4_golden_on_grid():
    for e, qhex in _rows("int4_on_grid.txt"):
        q = _codes(qhex).reshape(1, 128)
        w = ((q.astype(np.float32) - 8) * np.float32(2.0 ** int(e))).astype(np.float32)
        packed, scale = oracle.quantize_int4(w, 128)
        assert packed.tobytes().hex() == qhex
        assert scale.dtype == np.float16 and float(scale[0, 0]) == 2.0 ** int(e)
        assert np.array_equal(oracle.dequantize_int4(packed, scale, 128), w)


def test_int4_zero_point_keeps_sign():
    """The +8 zero point: positive weights stay positive, zero stays zero (q = 8)."""
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((4, 256)) * 0.02).astype(np.float32)
    w[0, 3] = 0.0
    packed, scale = oracle.quantize_int4(w, 128)
    q = oracle.unpack(packed)
    wh = oracle.dequantize_int4(packed, scale, 128)
    assert q[0, 3] == 8 and wh[0, 3] == 0.0
    big = np.abs(w) > np.repeat(scale.astype(np.float32), 128, axis=1) / 2
    assert np.all(q[(w > 0) & big] > 8) and np.all(wh[(w > 0) & big] > 0)
    assert np.all(q[(w < 0) & big] < 8) and np.all(wh[(w < 0) & big] < 0)


def test_int4_scale_is_fp16_of_absmax_over_7():
    """FP16 rounding of absmax / 7 checked by exact rational rounding (pins numpy's
    float16 conversion and the double rounding through float64)."""
    rng = np.random.default_rng(5)
    a = np.abs(rng.standard_normal(2000) * 0.05).astype(np.float32)
    a = np.concatenate([a, np.float32([7 * 2.0 ** -20, 7 * 2.0 ** -26, 1e-9, 0.0])])
    w = np.zeros((len(a), 128), np.float32)
    w[:, 0] = a
    _, scale = oracle.quantize_int4(w, 128)
    for i, ai in enumerate(a):
        assert Fraction(float(scale[i, 0])) == fl16(Fraction(float(ai)) / 7), i


def test_int4_rint_ties_to_even():
    """rint rounds halves to even ("LLM Compressor 0.14 ...", "Details worth knowing")."""
    t = np.array([2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5, 6.5, -6.5, 4.25, -4.75], np.float64)
    expect = [2, 4, -2, -4, 0, 0, 2, 6, -6, 4, -5]
    w = np.zeros((1, 128), np.float32)
    w[0, :len(t)] = (t * 2.0 ** -6).astype(np.float32)
    w[0, 127] = 7 * 2.0 ** -6                              # scale exactly 2^-6
    packed, scale = oracle.quantize_int4(w, 128)
    q = oracle.unpack(packed)[0].astype(int) - 8
    assert float(scale[0, 0]) == 2.0 ** -6
    assert q[:len(t)].tolist() == expect


def test_int4_rounding_brute_force_and_bound():
    rng = np.random.default_rng(6)
    w = (rng.standard_normal((2, 256)) * 0.02).astype(np.float32)
    w[1, 128:] = 0.0
    packed, scale = oracle.quantize_int4(w, 128)
    q = oracle.unpack(packed).astype(int) - 8
    wh = oracle.dequantize_int4(packed, scale, 128)
    for r in range(2):
        for k in range(256):
            s = Fraction(float(scale[r, k // 128]))
            if s == 0:
                exp = 0
            else:
                exp = max(-8, min(7, round_half_even(fl32(Fraction(float(w[r, k])) / s))))
            assert q[r, k] == exp, (r, k)
            assert abs(float(w[r, k]) - float(wh[r, k])) <= float(s) / 2 * (1 + 2 ** -20)
    assert np.all(np.abs(q) <= 8)


# ----------------------------------------------------------------------------- GEMV
def test_gemv_brute_force_exact():
    """Tiny matrices: exact rational dot products against the float64 oracle."""
    rng = np.random.default_rng(7)
    code = oracle.nf4_codebook()
    for n, k in [(1, 64), (3, 64), (4, 128)]:
        w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
        x = rng.standard_normal((2, k)).astype(np.float16)
        packed, absmax = oracle.quantize_nf4(w, code, 64)
        y = oracle.gemv_nf4(packed, absmax, code, x, 64)
        q = oracle.unpack(packed)
        for m in range(2):
            for r in range(n):
                exact = Fraction(0)
                for kk in range(k):
                    # w_hat = fl32(code * absmax), rounded exactly here
                    wh = fl32(Fraction(float(code[q[r, kk]])) * Fraction(float(absmax[r, kk // 64])))
                    exact += wh * Fraction(float(x[m, kk]))
                assert abs(y[m, r] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


def test_gemv_one_hot_selects_weight():
    """x = e_k returns column k of w_hat: pins orientation (y = x W^T, not x W)."""
    rng = np.random.default_rng(8)
    code = oracle.nf4_codebook()
    w = (rng.standard_normal((5, 128)) * 0.02).astype(np.float32)
    packed, absmax = oracle.quantize_nf4(w, code, 64)
    wh = oracle.dequantize_nf4(packed, absmax, code, 64)
    for k in (0, 1, 63, 64, 127):
        x = np.zeros((1, 128), np.float16)
        x[0, k] = 1.0
        assert np.array_equal(oracle.gemv_nf4(packed, absmax, code, x, 64)[0], wh[:, k].astype(np.float64))
    # square matrix: a transposed operand would still have the right shape
    w = (rng.standard_normal((128, 128)) * 0.02).astype(np.float32)
    packed, absmax = oracle.quantize_nf4(w, code, 64)
    wh = oracle.dequantize_nf4(packed, absmax, code, 64)
    x = np.zeros((1, 128), np.float16)
    x[0, 3] = 1.0
    assert np.array_equal(oracle.gemv_nf4(packed, absmax, code, x, 64)[0], wh[:, 3].astype(np.float64))


def test_gemv_zero_and_linearity():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((16, 256)) * 0.02).astype(np.float32)
    packed, scale = oracle.quantize_int4(w, 128)
    x = rng.standard_normal((3, 256)).astype(np.float16)
    y = oracle.gemv_int4(packed, scale, x, 128)
    assert np.all(oracle.gemv_int4(packed, scale, np.zeros_like(x), 128) == 0)
    assert np.array_equal(oracle.gemv_int4(packed, scale, (2 * x.astype(np.float32)).astype(np.float16), 128), 2 * y)
    x1 = rng.integers(-4, 5, (1, 256)).astype(np.float16)
    x2 = rng.integers(-4, 5, (1, 256)).astype(np.float16)
    y12 = oracle.gemv_int4(packed, scale, x1 + x2, 128)
    assert np.allclose(y12, oracle.gemv_int4(packed, scale, x1, 128) + oracle.gemv_int4(packed, scale, x2, 128),
                       rtol=1e-12, atol=1e-12)


def test_gemv_rows_matches_full():
    rng = np.random.default_rng(10)
    code = oracle.nf4_codebook()
    w = (rng.standard_normal((40, 192)) * 0.02).astype(np.float32)
    x = rng.standard_normal((2, 192)).astype(np.float16)
    packed, absmax = oracle.quantize_nf4(w, code, 64)
    rows = [0, 7, 39, 13]
    assert np.array_equal(oracle.gemv_nf4(packed, absmax, code, x, 64, rows=rows),
                          oracle.gemv_nf4(packed, absmax, code, x, 64)[:, rows])


# ----------------------------------------------------------------------------- workload
def test_step_matches_pages_numbers():
    vals = dict((ln.split()[0], float(ln.split()[1])) for ln in open(os.path.join(GOLDEN, "step_bytes.txt"))
                if ln.strip() and not ln.startswith("#"))
    assert synth.step_gemv_count() == vals["gemvs_per_step"]
    nw = synth.step_weight_count()
    assert nw == 1_543_569_408
    assert round(nw * 2 / 1e9, 3) == vals["bf16_weight_GB"]
    assert round(nw * 0.5 / 1e9, 3) == vals["int4_weight_GB"]
    assert round(100 * 151936 * 1536 / nw) == vals["lm_head_share_percent"]
    assert len(list(synth.decode_step_gemvs())) == 197


def test_synth_is_seeded_and_shaped():
    a = synth.weights(11, 8, 64)
    b = synth.weights(11, 8, 64)
    assert a.dtype == np.float32 and a.shape == (8, 64) and np.array_equal(a, b)
    o = synth.weights(12, 100, 100, outlier_frac=0.001)
    assert np.sum(np.abs(o) == np.float32(0.2)) == 10
    big = synth.weights(14, 2500, 64, outlier_frac=0.001)       # three row blocks
    rows = [0, 1023, 1024, 2499, 7]
    assert np.array_equal(synth.weights_rows(14, 2500, 64, rows, outlier_frac=0.001), big[rows])
    x = synth.activations(13, 2, 64)
    assert x.dtype == np.float16 and x.shape == (2, 64)
