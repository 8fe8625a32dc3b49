"""Plain CPU oracle for the fused 4-bit weight-only dequant-GEMV (W4A16).

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline / reference arm import this package.  The product package
(weight_only_bit_gb300) never imports it; it shares no code, table, constant or
helper with the CUDA path.  Its inputs come from weight_only_bit_gb300.synth
(random numbers and shapes only).

Everything here is written from the pages' definitions, in float64 where the
pages leave the precision open, in numpy, with no blocking or fusion:

  NF4 format -- "LLM Quantization on RTX 4060: Where 4-bit Decode Falls Behind
  FP16", section "Standard Expectation from Quantization": a 16-level normal
  float code book, blocks of 64 weights sharing one FP32 absmax, two 4-bit codes
  per uint8.  Same page, section "Kernel Implementation" (the fused kernel): the
  high nibble of packed byte j is element 2j, the low nibble element 2j+1, the
  block index is row * (K / blocksize) + col / blocksize, each weight is the
  FP32 product code[q] * absmax, the dot product accumulates in FP32 and the
  output is FP16.

  INT4 W4A16 -- "My Triton Kernel Ties bitsandbytes -- and Both Lose to Math",
  section "The kernels" (the +8 zero point stored in the nibble); group size 128
  from "LLM Compressor 0.14: GPTQ's 15x speedup is one fused loop", section
  "How the 15x and 30x were measured"; rounding with rint (ties to even) from
  the same page, "Details worth knowing".

Readings where the pages are silent (each is pinned by tests/test_oracle_pins.py):
  * NF4 code values: not printed on the pages.  The QLoRA construction
    (Dettmers et al. 2023, "4-bit NormalFloat"): 8 positive normal quantiles
    and 7 negative ones at probabilities evenly spaced from
    delta = ((1 - 1/32) + (1 - 1/30)) / 2 to 1/2, plus an exact zero, divided by
    the largest; computed in float64 and rounded to FP32.
  * NF4 rounding: the normalised weight n = fl32(w / absmax) (IEEE division);
    the code is the nearest code-book entry to n, exactly, a tie going to the
    lower code.  Equivalently: the number of exact midpoints
    (c[i] + c[i+1]) / 2 that lie strictly below n.  absmax == 0 gives n = 0.
  * INT4 scale: s = fl16(absmax / 7); q = clamp(rint(fl32(w / s)), -8, 7) + 8;
    s == 0 gives q = 8.
  * INT4 nibble order: the same as NF4 (element 2j in the high nibble).
  * Dequantised INT4 weight: (q - 8) * s, exact in FP32.
  * GEMV reference: y[m][n] = sum_k w_hat[n][k] * x[m][k] in float64.

  FP4 (E2M1) -- "LLM Compressor 0.14: GPTQ's 15x speedup is one fused loop",
  section "Details worth knowing": values rounded onto the grid
  {0, 0.5, 1, 1.5, 2, 3, 4, 6} through a ladder of thresholds, the comparison
  alternating between "<=" and "<" so that a value on a threshold goes to the
  even code.  Readings where the page is silent:
  * thresholds: the midpoints between consecutive grid values;
  * code: sign bit (bit 3) set iff w < 0, the grid index in bits 0-2 (the E2M1
    bit layout: exponent bits 1-2, mantissa bit 0); |value| above 6 stays at 6;
  * scale: one FP16 scale per group of `group` weights along a row (32 unless
    given), s = fl16(absmax / 6), the largest grid value; r = fl32(w / s);
    s == 0 gives code 0 for the whole group;
  * packing and dequantisation as for INT4: element 2j in the high nibble,
    w_hat = value * s, exact in FP32.
"""
from __future__ import annotations

import statistics

import numpy as np

__all__ = [
    "nf4_codebook", "pack", "unpack",
    "quantize_nf4", "dequantize_nf4", "quantize_int4", "dequantize_int4",
    "dequantize_nf4_rows", "dequantize_int4_rows", "gemv", "gemv_rows",
    "gemv_nf4", "gemv_int4",
    "fp4_grid", "quantize_fp4", "dequantize_fp4", "dequantize_fp4_rows", "gemv_fp4",
]


# --------------------------------------------------------------------------- codebook
def nf4_codebook() -> np.ndarray:
    """The 16 NF4 code values, ascending, FP32 (QLoRA "4-bit NormalFloat").

    Probabilities run evenly from delta down to 1/2: nine points for the positive
    half (the last, 1/2, dropped) and eight for the negative half (likewise),
    quantiles taken with the normal inverse CDF, zero added, everything divided
    by the largest value.  float64 throughout, one rounding to FP32 at the end.
    """
    delta = 0.5 * ((1.0 - 1.0 / 32.0) + (1.0 - 1.0 / 30.0))
    inv = statistics.NormalDist().inv_cdf
    pos = [inv(delta + i * ((0.5 - delta) / 8.0)) for i in range(8)]
    neg = [-inv(delta + i * ((0.5 - delta) / 7.0)) for i in range(7)]
    vals = sorted(pos + neg + [0.0])
    top = max(vals)
    return np.array([v / top for v in vals], dtype=np.float64).astype(np.float32)


# --------------------------------------------------------------------------- packing
def pack(codes: np.ndarray) -> np.ndarray:
    """Two 4-bit codes per byte: byte j = (code[2j] << 4) | code[2j+1]."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 2 == 0 and int(codes.max(initial=0)) < 16
    return ((codes[..., 0::2] << 4) | codes[..., 1::2]).astype(np.uint8)


def unpack(packed: np.ndarray) -> np.ndarray:
    """Inverse of pack: element 2j is the high nibble, 2j+1 the low nibble."""
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed >> 4
    out[..., 1::2] = packed & 0x0F
    return out


# --------------------------------------------------------------------------- NF4
def quantize_nf4(w: np.ndarray, code: np.ndarray, blocksize: int = 64):
    """Block-wise NF4 quantisation of an FP32 matrix w [N, K].

    Returns (packed uint8 [N, K/2], absmax float32 [N, K/blocksize]).
    Per block: a = max |w| (exact in FP32); n = fl32(w / a) (a == 0 -> 0);
    code = nearest entry of the ascending code book, a tie going to the lower.
    """
    w = np.asarray(w, dtype=np.float32)
    code = np.asarray(code, dtype=np.float32)
    n_rows, k = w.shape
    assert k % blocksize == 0
    blocks = w.reshape(n_rows, k // blocksize, blocksize)
    a = np.abs(blocks).max(axis=2)
    a64 = a.astype(np.float64)[..., None]
    with np.errstate(invalid="ignore", divide="ignore"):
        # float64 quotient rounded once more to FP32 == the IEEE FP32 quotient
        # (53 >= 2*24 + 2 makes the double rounding innocuous).
        n = np.where(a64 > 0.0, blocks.astype(np.float64) / a64, 0.0).astype(np.float32)
    c64 = code.astype(np.float64)
    mid = (c64[:-1] + c64[1:]) / 2.0            # exact in float64
    # searchsorted(side="left") = number of midpoints strictly below n
    q = np.searchsorted(mid, n.astype(np.float64).ravel(), side="left")
    q = q.astype(np.uint8).reshape(n_rows, k)
    return pack(q), a.astype(np.float32)


def dequantize_nf4(packed: np.ndarray, absmax: np.ndarray, code: np.ndarray,
                   blocksize: int = 64) -> np.ndarray:
    """w_hat = fl32(code[q] * absmax[block]) -- the FP32 product the fused kernel forms."""
    q = unpack(packed)
    code = np.asarray(code, dtype=np.float32)
    n_rows, k = q.shape
    scale = np.repeat(np.asarray(absmax, dtype=np.float32), blocksize, axis=1)
    assert scale.shape == (n_rows, k)
    return (code[q] * scale).astype(np.float32)


def dequantize_nf4_rows(packed, absmax, code, rows, blocksize: int = 64):
    rows = np.asarray(rows, dtype=np.int64)
    return dequantize_nf4(packed[rows], absmax[rows], code, blocksize)


# --------------------------------------------------------------------------- INT4
def quantize_int4(w: np.ndarray, group: int = 128):
    """Group-wise symmetric INT4 with a +8 zero point, FP16 scale per group.

    Returns (packed uint8 [N, K/2], scale float16 [N, K/group]).
    s = fl16(absmax / 7); q = clamp(rint(fl32(w / s)), -8, 7) + 8 (s == 0 -> q = 8).
    """
    w = np.asarray(w, dtype=np.float32)
    n_rows, k = w.shape
    assert k % group == 0
    blocks = w.reshape(n_rows, k // group, group)
    a = np.abs(blocks).max(axis=2).astype(np.float64)
    # float64 quotient then FP16: innocuous double rounding (53 >= 2*11 + 2)
    s16 = (a / 7.0).astype(np.float16)
    s = s16.astype(np.float64)[..., None]
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.where(s > 0.0, blocks.astype(np.float64) / s, 0.0).astype(np.float32)
    q = np.clip(np.rint(r), -8, 7).astype(np.int16) + 8
    return pack(q.reshape(n_rows, k).astype(np.uint8)), s16


def dequantize_int4(packed: np.ndarray, scale: np.ndarray, group: int = 128) -> np.ndarray:
    """w_hat = (q - 8) * s, exact in FP32."""
    q = unpack(packed).astype(np.int32) - 8
    n_rows, k = q.shape
    s = np.repeat(np.asarray(scale, dtype=np.float16).astype(np.float32), group, axis=1)
    assert s.shape == (n_rows, k)
    return (q.astype(np.float32) * s).astype(np.float32)


def dequantize_int4_rows(packed, scale, rows, group: int = 128):
    rows = np.asarray(rows, dtype=np.int64)
    return dequantize_int4(packed[rows], scale[rows], group)


# --------------------------------------------------------------------------- FP4 (E2M1)
def fp4_grid() -> np.ndarray:
    """The eight E2M1 magnitudes, index 0 ... 7 (float64, all exact)."""
    return np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _fp4_ladder(m: np.ndarray) -> np.ndarray:
    """Grid index of magnitudes m >= 0: one rung per midpoint t_i between grid
    values i and i + 1.  At an even i the value moves up only when m > t_i (a tie
    stays on i), at an odd i when m >= t_i (a tie moves on to i + 1): either way
    a tie lands on the even index.  Past the last rung the index stays 7."""
    g = fp4_grid()
    idx = np.zeros(m.shape, dtype=np.int64)
    for i in range(7):
        t = (g[i] + g[i + 1]) / 2.0
        idx += (m > t) if i % 2 == 0 else (m >= t)
    return idx


def quantize_fp4(w: np.ndarray, group: int = 32):
    """Group-wise FP4 (E2M1) with an FP16 scale per group.

    Returns (packed uint8 [N, K/2], scale float16 [N, K/group]).
    s = fl16(absmax / 6); r = fl32(w / s) (s == 0 -> r = 0); code =
    (w < 0) << 3 | ladder(|r|).
    """
    w = np.asarray(w, dtype=np.float32)
    n_rows, k = w.shape
    assert k % group == 0
    blocks = w.reshape(n_rows, k // group, group)
    a = np.abs(blocks).max(axis=2).astype(np.float64)
    # float64 quotient then FP16: innocuous double rounding (53 >= 2*11 + 2)
    s16 = (a / 6.0).astype(np.float16)
    s = s16.astype(np.float64)[..., None]
    with np.errstate(invalid="ignore", divide="ignore"):
        r = np.where(s > 0.0, blocks.astype(np.float64) / s, 0.0).astype(np.float32)
    mag = _fp4_ladder(np.abs(r.astype(np.float64)))
    sign = (blocks < 0).astype(np.int64)
    q = (sign << 3) | mag
    return pack(q.reshape(n_rows, k).astype(np.uint8)), s16


def dequantize_fp4(packed: np.ndarray, scale: np.ndarray, group: int = 32) -> np.ndarray:
    """w_hat = (-1)^(bit 3) * grid[q & 7] * s, exact in FP32."""
    q = unpack(packed).astype(np.int64)
    n_rows, k = q.shape
    v = fp4_grid()[q & 7] * np.where(q & 8, -1.0, 1.0)
    s = np.repeat(np.asarray(scale, dtype=np.float16).astype(np.float64), group, axis=1)
    assert s.shape == (n_rows, k)
    return (v * s).astype(np.float32)


def dequantize_fp4_rows(packed, scale, rows, group: int = 32):
    rows = np.asarray(rows, dtype=np.int64)
    return dequantize_fp4(packed[rows], scale[rows], group)


# --------------------------------------------------------------------------- GEMV
def gemv(w_hat: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y[m][n] = sum_k w_hat[n][k] * x[m][k], in float64 (inputs are exact in float64)."""
    w64 = np.asarray(w_hat, dtype=np.float32).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x, dtype=np.float16)).astype(np.float64)
    return x64 @ w64.T


def gemv_rows(w_hat_rows: np.ndarray, x: np.ndarray) -> np.ndarray:
    """Same as gemv for a subset of output rows (already dequantised)."""
    return gemv(w_hat_rows, x)


def gemv_nf4(packed, absmax, code, x, blocksize: int = 64, rows=None):
    if rows is None:
        return gemv(dequantize_nf4(packed, absmax, code, blocksize), x)
    return gemv(dequantize_nf4_rows(packed, absmax, code, rows, blocksize), x)


def gemv_int4(packed, scale, x, group: int = 128, rows=None):
    if rows is None:
        return gemv(dequantize_int4(packed, scale, group), x)
    return gemv(dequantize_int4_rows(packed, scale, rows, group), x)


def gemv_fp4(packed, scale, x, group: int = 32, rows=None):
    if rows is None:
        return gemv(dequantize_fp4(packed, scale, group), x)
    return gemv(dequantize_fp4_rows(packed, scale, rows, group), x)
