"""Low-precision read-copy formats, written from the format definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring for who may use it).

The pages keep a high-precision checkpoint for the recurrence and a low-precision
copy for reads. At flush the folded checkpoint is converted into both formats
independently ([RU] §06; [AR] "الحد من خطأ التكميم"; [ZH] 三项收益, item 3).
They name the formats only as "NVFP4" and "FP8". The layouts below are this
build's readings:

E4M3 rows (one fp32 scale per row of N elements):
    a = max|x|;  if a <= 2^-100 the row is all zero (codes 0, s = 0)
    inv = rn32(448 / a),  s = rn32(a / 448)
    code_n = E4M3(rn32(x_n * inv)),  x_hat_n = value(code_n) * s

E2M1 rows with 16-element blocks (NVFP4-style two-level scale, one fp32
scale per row and one E4M3 scale per block along N):
    a = max|x|;  if a <= 2^-100 the row is all zero
    s_r = rn32(a / 2688)            (2688 = 448 * 6)
    d6  = rn32(6 * s_r)
    per block: a_b = max|x| in block, sb = E4M3(rn32(a_b / d6))
               d = rn32(value(sb) * s_r),  r = rn32(1 / d) if d > 0 else 0
               code_n = E2M1(rn32(x_n * r))
    x_hat_n = value(code_n) * value(sb) * s_r

rn32 is IEEE round-to-nearest-even to binary32. A float64 operation on binary32
operands, rounded once to binary32, gives exactly the binary32 result for
+, -, * and / (the double precision is wide enough that double rounding
cannot occur). E4M3(.) and E2M1(.) round to nearest, ties to the even code.
They saturate to the largest finite magnitude and keep the sign, also for zero.
"""
from __future__ import annotations

import math

import numpy as np

from .recurrence import conventional_step

E4M3_MAX = 448.0
E2M1_MAX = 6.0
ZERO_ROW_AMAX = 2.0 ** -100
BLOCK = 16


def e4m3_value(code) -> np.ndarray:
    """Value of an E4M3 code (OCP FP8: 1 sign, 4 exponent bits with bias 7, 3
    mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN; no infinities)."""
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def e2m1_value(code) -> np.ndarray:
    """Value of an E2M1 code (OCP MX FP4: 1 sign, 2 exponent bits with bias 1,
    1 mantissa bit; exponent 0 is subnormal; no NaN or infinity)."""
    c = np.asarray(code, dtype=np.int64)
    s = (c >> 3) & 1
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return np.where(s == 1, -mag, mag)


_E4M3_MAG = e4m3_value(np.arange(0x7F))  # codes 0x00..0x7E, increasing magnitudes
_E2M1_MAG = e2m1_value(np.arange(0x8))  # codes 0x0..0x7


def _rne_to_grid(y, mags: np.ndarray, sign_bit: int) -> np.ndarray:
    """Round |y| to the nearest entry of the increasing grid ``mags`` (code = index).

    Ties go to the even code. Values at or above the top entry saturate to it.
    The sign bit is set from the sign of y, including -0.
    """
    y = np.asarray(y, dtype=np.float64)
    if np.any(np.isnan(y)):
        raise ValueError("NaN input to a quantizer")
    mag = np.abs(y)
    top = len(mags) - 1
    lo = np.clip(np.searchsorted(mags, mag, side="right") - 1, 0, top)
    hi = np.minimum(lo + 1, top)
    d_lo = mag - mags[lo]
    d_hi = mags[hi] - mag
    up = (hi != lo) & ((d_hi < d_lo) | ((d_hi == d_lo) & (lo % 2 == 1)))
    code = np.where(up, hi, lo)
    code = np.where(mag >= mags[top], top, code)
    neg = np.signbit(y)
    return (code | (neg.astype(np.int64) << sign_bit)).astype(np.uint8)


def e4m3_encode(y) -> np.ndarray:
    """binary32 values -> E4M3 codes, round to nearest even, saturating to +-448
    (OCP 8-bit floating point specification, E4M3 with saturating conversion)."""
    return _rne_to_grid(y, _E4M3_MAG, 7)


def e2m1_encode(y) -> np.ndarray:
    """binary32 values -> E2M1 codes (low nibble), round to nearest even, saturating to +-6
    (OCP Microscaling specification, FP4 E2M1 elements)."""
    return _rne_to_grid(y, _E2M1_MAG, 3)


def _rn32(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def quantize_rows_e4m3(X):
    """Rows of fp32 values [..., N] -> (codes uint8 [..., N], scale fp32 [...]).

    The E4M3 row recipe of the module docstring: this build's reading of the
    pages' FP8 read copy, refreshed from the checkpoint at each flush ([RU] §06)."""
    X = np.asarray(X, dtype=np.float32)
    a = np.abs(X).max(axis=-1)
    live = a > ZERO_ROW_AMAX
    a64 = a.astype(np.float64)
    safe = np.where(live, a64, 1.0)
    inv = np.where(live, _rn32(E4M3_MAX / safe), np.float32(0))
    s = np.where(live, _rn32(safe / E4M3_MAX), np.float32(0)).astype(np.float32)
    y = _rn32(X.astype(np.float64) * inv.astype(np.float64)[..., None])
    return e4m3_encode(y), s


def dequantize_rows_e4m3(codes, scale) -> np.ndarray:
    """x_hat = value(code) * s per row: what a non-flush step reads in place of the checkpoint ([RU] §06)."""
    return e4m3_value(codes) * np.asarray(scale, np.float64)[..., None]


def quantize_rows_e2m1(X):
    """Rows of fp32 values [..., N] (N a multiple of 16) ->
    (codes uint8 [..., N] one nibble each, block codes uint8 [..., N/16], row scale fp32 [...]).

    The E2M1 recipe of the module docstring: this build's NVFP4-style reading of
    the pages' 4-bit read copy ([RU] §06; [AR] "الحد من خطأ التكميم")."""
    X = np.asarray(X, dtype=np.float32)
    N = X.shape[-1]
    if N % BLOCK:
        raise ValueError("N must be a multiple of 16")
    a = np.abs(X).max(axis=-1)
    live = a > ZERO_ROW_AMAX
    a64 = np.where(live, a.astype(np.float64), 0.0)
    s_r = _rn32(a64 / (E4M3_MAX * E2M1_MAX))
    d6 = _rn32(6.0 * s_r.astype(np.float64))
    Xb = X.reshape(X.shape[:-1] + (N // BLOCK, BLOCK))
    a_b = np.abs(Xb).max(axis=-1).astype(np.float64)
    d6b = d6.astype(np.float64)[..., None]
    ratio = np.where(d6b > 0, _rn32(a_b / np.where(d6b > 0, d6b, 1.0)), np.float32(0))
    bcodes = e4m3_encode(ratio)
    sb = e4m3_value(bcodes)
    d = _rn32(sb * s_r.astype(np.float64)[..., None]).astype(np.float64)
    r = np.where(d > 0, _rn32(1.0 / np.where(d > 0, d, 1.0)), np.float32(0)).astype(np.float64)
    y = _rn32(Xb.astype(np.float64) * r[..., None])
    codes = e2m1_encode(y).reshape(X.shape)
    return codes, bcodes, s_r.astype(np.float32)


def dequantize_rows_e2m1(codes, bcodes, rscale) -> np.ndarray:
    """x_hat = value(code) * value(block code) * s_r: the 4-bit read copy as a non-flush step reads it ([RU] §06)."""
    codes = np.asarray(codes)
    N = codes.shape[-1]
    vb = e2m1_value(codes).reshape(codes.shape[:-1] + (N // BLOCK, BLOCK))
    sb = e4m3_value(bcodes)[..., None]
    out = vb * sb * np.asarray(rscale, np.float64)[..., None, None]
    return out.reshape(codes.shape)


def element_error_bound(fmt: str, X) -> np.ndarray:
    """Per-element bound on |x_hat - x| for the read-copy formats.

    The pages ask that the read copy's error stay that of one quantization
    ([RU] §06; [AR] "الحد من خطأ التكميم") but state no bound; this one is
    derived here from the format definitions.

    E4M3: round to nearest gives relative error <= 2^-4 for normal codes and an
    absolute error <= 2^-10 (in units of the row scale s) for subnormal codes.
    Three binary32 roundings (inv, s, y) add a few ulps:
        |x_hat - x| <= (2^-4 + 2^-20)|x| + (2^-10 + 2^-20) s.
    E2M1: on the grid {0,.5,1,1.5,2,3,4,6} the rounding error is at most
    0.25*max(1,|y|) in block units d = value(sb)*s_r. When the block scale
    rounds down, values beyond 6 saturate. That adds at most the E4M3 error
    of the block scale, max(2^-4 a_b, 6*2^-10 s_r) in absolute terms. A zero
    block scale is the limiting case of the same term:
        |x_hat - x| <= 0.25 max(d, |x|) + max(2^-4 a_b, 6*2^-10 s_r) + 2^-20 (|x| + d).
    """
    X = np.asarray(X, dtype=np.float32).astype(np.float64)
    ax = np.abs(X)
    a = ax.max(axis=-1, keepdims=True)
    if fmt == "e4m3":
        s = a / E4M3_MAX
        return (2.0 ** -4 + 2.0 ** -20) * ax + (2.0 ** -10 + 2.0 ** -20) * s
    if fmt == "e2m1":
        N = X.shape[-1]
        _, bcodes, s_r = quantize_rows_e2m1(X.astype(np.float32))
        d = (e4m3_value(bcodes) * s_r.astype(np.float64)[..., None])  # [..., N/16]
        d_el = np.repeat(d, BLOCK, axis=-1)
        a_b = np.repeat(ax.reshape(ax.shape[:-1] + (N // BLOCK, BLOCK)).max(axis=-1), BLOCK, axis=-1)
        sr_el = s_r.astype(np.float64)[..., None]
        return (0.25 * np.maximum(d_el, ax) + np.maximum(2.0 ** -4 * a_b, 6.0 * 2.0 ** -10 * sr_el)
                + 2.0 ** -20 * (ax + d_el))
    raise ValueError(fmt)


class FullyQuantizedState:
    """Comparator in which the state itself is stored quantized and fed back each step.

    Rounding error then re-enters the recurrence at every step, which is the
    failure mode the split-precision design avoids ([RU] §02 item 3; [AR]
    "الحد من خطأ التكميم"). Each step computes S_pre = alpha * deQ(S_q) + v k^T,
    outputs o = S_pre q (the fresh update, as a conventional kernel with
    quantized storage would), and stores S_q = Q(rn32(S_pre)).
    """

    def __init__(self, S0, fmt: str):
        self.fmt = fmt
        self.S = self._roundtrip(np.asarray(S0, np.float64))

    def _roundtrip(self, X):
        X32 = X.astype(np.float32)
        if self.fmt == "e4m3":
            return dequantize_rows_e4m3(*quantize_rows_e4m3(X32))
        if self.fmt == "e2m1":
            return dequantize_rows_e2m1(*quantize_rows_e2m1(X32))
        raise ValueError(self.fmt)

    def step(self, alpha, v, k, q):
        """One step of the quantized-state recurrence ([RU] §02 item 3); returns o."""
        S_pre, o = conventional_step(self.S, alpha, v, k, q)
        self.S = self._roundtrip(S_pre)
        return o


assert math.isclose(float(_E4M3_MAG[-1]), E4M3_MAX) and float(_E2M1_MAG[-1]) == E2M1_MAX
