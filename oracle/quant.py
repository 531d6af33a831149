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
    Input float values (any float dtype); returns uint8 codes."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    flat_x, flat_o = x.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat_x):
        if np.isnan(v):
            flat_o[i] = NAN_CODE | (0x80 if np.signbit(v) else 0)
            continue
        a = min(abs(v), E4M3_MAX)
        j = int(np.searchsorted(_POS_VALUES, a))          # first value >= a
        if j < len(_POS_VALUES) and _POS_VALUES[j] == a:
            code = int(_POS[j])
        else:
            lo, hi = j - 1, j                               # a lies strictly between
            dlo, dhi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
            if dlo < dhi:
                code = int(_POS[lo])
            elif dhi < dlo:
                code = int(_POS[hi])
            else:                                           # tie: the even code
                code = int(_POS[lo]) if int(_POS[lo]) % 2 == 0 else int(_POS[hi])
        flat_o[i] = code | (0x80 if np.signbit(v) else 0)
    return out


def quantize(x, scale):
    """Codes of x (float values, e.g. decoded bf16) for one float32 scale:
    E4M3(float32(x) / float32(scale)) with a float32 division."""
    q = np.asarray(x, dtype=np.float32) / np.float32(scale)
    return f64_to_e4m3(q.astype(np.float64))


def dequantize(codes, scale):
    """float64 values of codes at one float32 scale."""
    return e4m3_to_f64(codes) * float(np.float32(scale))
