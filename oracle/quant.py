"""FP8 E4M3 key/value quantisation (oracle; test infrastructure only).

The pages say only that quantised KV (INT8/FP8) reduces bytes per token at a
precision cost ("PagedAttention and KV Memory", "Alternatives and
ecosystem"), and that exactness of paging is judged at the same KV precision
("PagedAttention in vLLM: scattered memory, exact attention", sections 8 and
11).  This restates the plainest FP8 scheme:

  * E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
    bits; exponent 0 is subnormal (m * 2^-9), codes S.1111.111 are NaN, there
    is no infinity; the largest finite magnitude is 448.
  * A cache holds code = E4M3(x / scale) with one float32 scale per layer for
    K and one for V; x / scale is a float32 division (round to nearest), then
    rounded to the nearest E4M3 value, ties to the even code, magnitudes above
    448 saturating to 448 and NaN staying NaN.
  * Reading a cache gives E4M3(code) * scale, exactly (in float64).

Decode over a quantised cache is then the ordinary paged attention of
attention.py over the dequantised keys and values.
"""
import numpy as np

E4M3_MAX = 448.0
NAN_CODE = 0x7F


def e4m3_to_f64(codes):
    """Value of each E4M3 code (uint8), from the format definition."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


_CODES = np.arange(256, dtype=np.uint8)
_VALUES = e4m3_to_f64(_CODES)
_FINITE = ~np.isnan(_VALUES)
_POS = _CODES[_FINITE & (_VALUES >= 0) & ((_CODES & 0x80) == 0)]      # 0x00 .. 0x7E
_POS_VALUES = _VALUES[_POS]                                            # increasing


def f64_to_e4m3(x):
    """Round each value to the nearest E4M3 value (ties to the even code),
    saturating at +-448; NaN gives the NaN code with the input's sign bit.
    Input float values (any float dtype); returns uint8 codes.

    For every magnitude a = min(|x|, 448): the neighbours are the largest
    grid value <= a and the smallest >= a; the nearer wins, and on a tie the
    one whose code is even."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")              # first grid value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.where(_POS_VALUES[hi] == a, hi, np.maximum(hi - 1, 0))
    d_lo = a - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - a
    code_lo, code_hi = _POS[lo].astype(np.int64), _POS[hi].astype(np.int64)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (code_hi % 2 == 0) & (code_lo % 2 != 0))
    code = np.where(pick_hi, code_hi, code_lo)
    code = np.where(nan, NAN_CODE, code)
    sign = np.signbit(x).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def quantize(x, scale):
    """Codes of x (float values, e.g. decoded bf16) for one float32 scale:
    E4M3(float32(x) / float32(scale)) with a float32 division."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return f64_to_e4m3(q.astype(np.float64))


def dequantize(codes, scale):
    """float64 values of codes at one float32 scale."""
    return e4m3_to_f64(codes) * float(np.float32(scale))
