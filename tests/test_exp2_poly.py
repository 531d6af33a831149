"""The cubic the prefill kernel uses for part of its exp2 evaluations: its
coefficients in the CUDA source are the Remez fit of exp2_poly_fit.py, and
its error (float32 Horner evaluation, range reduction included) stays below
the bound the prefill tolerance assumes.  CPU only."""
import os
import re

import numpy as np

from paged_kv_cache_124_gb300 import exp2_poly_fit as F

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "paged_kv_cache_124_gb300", "csrc",
                   "pa_prefill.cu")


def _kernel_coefficients():
    text = open(SRC).read()
    return [float(re.search(r"kExp2C%d = ([0-9.eE+-]+)f;" % i, text).group(1)) for i in range(4)]


def test_kernel_coefficients_are_the_fit():
    c, err = F.fit()
    assert err < 7.5e-5
    np.testing.assert_allclose(_kernel_coefficients(), c, rtol=1e-8)


def _emulate(x):
    """The kernel's evaluation in float32: round-to-integer by adding
    1.5 * 2^23, cubic in the remainder, exponent add."""
    c = np.array(_kernel_coefficients(), dtype=np.float32)
    x = np.maximum(x.astype(np.float32), np.float32(-125.0))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    f = (x - (t - np.float32(12582912.0))).astype(np.float32)
    p = (((c[3] * f + c[2]) * f + c[1]) * f + c[0]).astype(np.float32)
    bits = p.view(np.int32) + (t.view(np.int32) << 23)
    return bits.view(np.float32)


def test_whole_range_relative_error():
    x = np.linspace(-125.0, 8.0, 2_000_003).astype(np.float32)
    got = _emulate(x).astype(np.float64)
    want = 2.0 ** x.astype(np.float64)
    assert np.abs(got / want - 1).max() < 7.6e-5
    # below the clamp every input gives (about) 2^-125, a normal float
    low = float(_emulate(np.array([-np.inf, -1000.0], dtype=np.float32)).max())
    assert abs(low / 2.0 ** -125 - 1) < 7.6e-5
