"""Seeded sweeps over the supported shape space (decode and prefill, bf16 and
FP8 caches), GPU against the oracle.

Each case draws d_head, block size, KV heads, group size, batch, context
lengths (a mix of the lengths around block, 16-position tile, partition and
128-key tile boundaries, and uniform ones), new-token counts, partition size
and output type from a generator seeded by the case number, builds the paged
problem (random physical placement, NaN in every slot past a context) and
compares the kernel with the oracle under the same tolerances as the
per-kernel tests.  The draws depend only on the seed, so a failing case is
reproducible by its id."""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A
from oracle import quant as Q
from _gpu_util import assert_attention_close, out_to_f64

pytestmark = pytest.mark.gpu

api = pytest.importorskip("paged_kv_cache_124_gb300.api")
from test_gpu_fp8 import _decode_fp8, _fp8_problem  # noqa: E402
from test_gpu_kernels import _paged_problem, _run_decode  # noqa: E402
from test_gpu_prefill import _problem as _prefill_problem, _run as _run_prefill  # noqa: E402

EDGE = [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 512, 513]


def _lengths(rng, S, hi):
    return [int(rng.choice(EDGE)) if rng.random() < 0.5 else int(rng.integers(1, hi + 1)) for _ in range(S)]


def _decode_case(i):
    rng = np.random.default_rng(1000 + i)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([8, 16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    S = int(rng.integers(1, 9))
    lens = _lengths(rng, S, 2500)
    P = int(rng.choice([0, 0, 64, 128, 192, 256, 512, 1024]))
    out_dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    return D, B, Hkv, G, lens, P, out_dtype


@pytest.mark.parametrize("i", range(24))
def test_decode_random_config(i):
    D, B, Hkv, G, lens, P, out_dtype = _decode_case(i)
    Hq = G * Hkv
    rng = np.random.default_rng(2000 + i)
    q, kc, vc, tables, ctx = _paged_problem(rng, lens, Hq, Hkv, D, B)
    scale = 1.0 / math.sqrt(D)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _run_decode(q, kc, vc, tables, ctx, B, scale, Hq, Hkv, D, out_dtype, P, status=st)
    ref = A.paged_decode(q, kc, vc, tables, ctx, scale, B)
    what = "decode case %d: D %d B %d Hkv %d G %d lens %s P %d %s" % (i, D, B, Hkv, G, lens, P, out_dtype)
    assert_attention_close(out_to_f64(out), ref, out_dtype == torch.float32, what)
    assert st.item() == 0, what


@pytest.mark.parametrize("i", range(12))
def test_decode_fp8_random_config(i):
    rng = np.random.default_rng(3000 + i)
    B = int(rng.choice([8, 16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    S = int(rng.integers(1, 7))
    lens = _lengths(rng, S, 3000)
    P = int(rng.choice([0, 0, 64, 256, 512]))
    ks, vs = float(rng.choice([4.0 / 448, 0.01, 0.05])), float(rng.choice([3.0 / 448, 0.02]))
    out_dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    Hq = G * Hkv
    qb, kc, vc, tab, ctx = _fp8_problem(40 + i, Hq, Hkv, B, lens, ks, vs)
    want = A.paged_decode(qb, Q.dequantize(kc, ks), Q.dequantize(vc, vs), tab, ctx, 1 / math.sqrt(128), B)
    got, st = _decode_fp8(qb, kc, vc, tab, ctx, B, Hq, Hkv, ks, vs, out_dtype, P)
    what = "fp8 decode case %d: B %d Hkv %d G %d lens %s P %d scales %g %g %s" % (
        i, B, Hkv, G, lens, P, ks, vs, out_dtype)
    assert st == 0, what
    assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, what)


def _prefill_case(i):
    rng = np.random.default_rng(4000 + i)
    D = int(rng.choice([64, 128]))
    B = int(rng.choice([8, 16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16, 32]))
    while G * Hkv > 64:                      # keep the oracle's work small
        G //= 2
    S = int(rng.integers(1, 6))
    ctxs = _lengths(rng, S, 700)
    news = []
    for c in ctxs:
        u = rng.random()
        news.append(c if u < 0.4 else (1 if u < 0.55 else (0 if u < 0.6 else int(rng.integers(1, c + 1)))))
    out_dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    return D, B, Hkv, G, ctxs, news, out_dtype


@pytest.mark.parametrize("i", range(16))
def test_prefill_random_config(i):
    D, B, Hkv, G, ctxs, news, out_dtype = _prefill_case(i)
    Hq = G * Hkv
    qb, kb, vb, tab, qs, ctx = _prefill_problem(50 + i, Hq, Hkv, D, B, ctxs, news)
    what = "prefill case %d: D %d B %d Hkv %d G %d ctxs %s news %s %s" % (i, D, B, Hkv, G, ctxs, news, out_dtype)
    if sum(news) == 0:
        pytest.skip("no new tokens drawn")
    want = A.paged_prefill(qb, kb, vb, tab, qs, ctx, 1.0 / math.sqrt(D), B)
    got, status = _run_prefill(qb, kb, vb, tab, qs, ctx, B, Hq, Hkv, D, out_dtype)
    assert status == 0, what
    assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, what)


@pytest.mark.parametrize("i", range(12))
def test_prefill_fp8_random_config(i):
    from test_gpu_prefill_fp8 import _problem as _fp8_prefill_problem, _run as _run_fp8_prefill
    rng = np.random.default_rng(5000 + i)
    B = int(rng.choice([8, 16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 4, 8, 16]))
    while G * Hkv > 64:                      # keep the oracle's work small
        G //= 2
    S = int(rng.integers(1, 5))
    ctxs = _lengths(rng, S, 700)
    news = []
    for c in ctxs:
        u = rng.random()
        news.append(c if u < 0.4 else (1 if u < 0.55 else int(rng.integers(1, c + 1))))
    ks, vs = float(rng.choice([4.0 / 448, 0.01, 0.05])), float(rng.choice([3.0 / 448, 0.02]))
    out_dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    Hq = G * Hkv
    qb, kc, vc, tab, qs, ctx = _fp8_prefill_problem(70 + i, Hq, Hkv, B, ctxs, news, ks, vs)
    want = A.paged_prefill(qb, Q.dequantize(kc, ks), Q.dequantize(vc, vs), tab, qs, ctx, 1 / math.sqrt(128), B)
    got, st = _run_fp8_prefill(qb, kc, vc, tab, qs, ctx, B, Hq, Hkv, ks, vs, out_dtype)
    what = "fp8 prefill case %d: B %d Hkv %d G %d ctxs %s news %s scales %g %g %s" % (
        i, B, Hkv, G, ctxs, news, ks, vs, out_dtype)
    assert st == 0, what
    assert_attention_close(out_to_f64(got), want, out_dtype == torch.float32, what)
