"""Host-side argument checks of the C ABI (include/pa.h: host-detected errors
are returned before anything is enqueued), called through the raw entry
points with stand-in device addresses that are never dereferenced: every
case here is rejected before the library makes its first CUDA call, so no
GPU is needed.  Plus the binding's refusal of host tensors.  CPU only."""

import ctypes

import pytest
import torch

from paged_kv_cache_124_gb300 import api

L = api._lib
A = 0x100000            # a 256-byte-aligned stand-in address (never dereferenced)


def decode(**kw):
    a = dict(out=A, out_dtype=api.PA_DTYPE_BF16, q=A, k=A, v=A, tables=A, ctx=A, block_size=16, scale=0.088,
             hq=32, hkv=8, d=128, num_seqs=4, max_blocks=8, num_blocks=64, max_ctx=128, partition=0, ws=None,
             ws_bytes=0, status=None)
    a.update(kw)
    return L.pa_decode(a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["tables"], a["ctx"], a["block_size"],
                       a["scale"], a["hq"], a["hkv"], a["d"], a["num_seqs"], a["max_blocks"], a["num_blocks"],
                       a["max_ctx"], a["partition"], a["ws"], a["ws_bytes"], a["status"], None)


def decode_fp8(**kw):
    a = dict(out=A, out_dtype=api.PA_DTYPE_F32, q=A, k=A, v=A, tables=A, ctx=A, block_size=16, scale=0.088,
             k_scale=0.01, v_scale=0.01, hq=32, hkv=8, d=128, num_seqs=4, max_blocks=8, num_blocks=64, max_ctx=128,
             partition=0)
    a.update(kw)
    return L.pa_decode_fp8(a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["tables"], a["ctx"],
                           a["block_size"], a["scale"], a["k_scale"], a["v_scale"], a["hq"], a["hkv"], a["d"],
                           a["num_seqs"], a["max_blocks"], a["num_blocks"], a["max_ctx"], a["partition"], None, 0,
                           None, None)


def prefill(**kw):
    a = dict(out=A, out_dtype=api.PA_DTYPE_BF16, q=A, k=A, v=A, tables=A, max_blocks=8, qs=A, ctx=A, num_seqs=2,
             num_tokens=100, max_q=64, num_blocks=64, block_size=16, scale=0.088, hq=32, hkv=8, d=128, ws=A,
             ws_bytes=1 << 30, sched=None)
    a.update(kw)
    return L.pa_prefill(a["out"], a["out_dtype"], a["q"], a["k"], a["v"], a["tables"], a["max_blocks"], a["qs"],
                        a["ctx"], a["num_seqs"], a["num_tokens"], a["max_q"], a["num_blocks"], a["block_size"],
                        a["scale"], a["hq"], a["hkv"], a["d"], a["ws"], a["ws_bytes"], a["sched"], None, None)


def reshape(**kw):
    a = dict(k_cache=A, v_cache=A, k=A, v=A, slots=A, num_tokens=4, hkv=8, d=128, block_size=16, num_blocks=64)
    a.update(kw)
    return L.pa_reshape_and_cache(a["k_cache"], a["v_cache"], a["k"], a["v"], a["slots"], a["num_tokens"], a["hkv"],
                                  a["d"], a["block_size"], a["num_blocks"], None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(num_seqs=0), api.PA_OK),                                    # nothing to do, nothing read
    (dict(num_seqs=-1), api.PA_ERR_INVALID_ARG),
    (dict(out_dtype=7), api.PA_ERR_INVALID_ARG),
    (dict(out=None), api.PA_ERR_INVALID_ARG),
    (dict(ctx=None), api.PA_ERR_INVALID_ARG),
    (dict(block_size=12), api.PA_ERR_UNSUPPORTED),
    (dict(d=96), api.PA_ERR_UNSUPPORTED),
    (dict(hq=12, hkv=8), api.PA_ERR_UNSUPPORTED),                     # not a whole group per KV head
    (dict(hq=32, hkv=1), api.PA_ERR_UNSUPPORTED),                     # G = 32 > 16
    (dict(q=A + 8), api.PA_ERR_MISALIGNED),
    (dict(partition=100), api.PA_ERR_INVALID_ARG),                    # not a multiple of 64
    (dict(partition=16384), api.PA_ERR_INVALID_ARG),                  # above 8192
    (dict(ws=A + 16, ws_bytes=1 << 20), api.PA_ERR_WORKSPACE),        # workspace not 256-byte aligned
    (dict(scale=float("nan")), api.PA_ERR_INVALID_ARG),
])
def test_decode_host_checks(kw, want):
    assert decode(**kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(k_scale=0.0), api.PA_ERR_INVALID_ARG),
    (dict(v_scale=float("inf")), api.PA_ERR_INVALID_ARG),
    (dict(d=64), api.PA_ERR_UNSUPPORTED),                             # E4M3 caches: d_head 128 only
    (dict(num_seqs=0), api.PA_OK),
])
def test_decode_fp8_host_checks(kw, want):
    assert decode_fp8(**kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(num_seqs=0), api.PA_OK),
    (dict(num_tokens=0), api.PA_OK),
    (dict(hq=12, hkv=8), api.PA_ERR_UNSUPPORTED),                     # not a whole group per KV head, as decode
    (dict(hq=24, hkv=8), api.PA_ERR_UNSUPPORTED),                     # G = 3 does not divide a 128-row tile
    (dict(out_dtype=9), api.PA_ERR_INVALID_ARG),
    (dict(block_size=64), api.PA_ERR_UNSUPPORTED),
    (dict(qs=None), api.PA_ERR_INVALID_ARG),
    (dict(max_blocks=0), api.PA_ERR_INVALID_ARG),
    (dict(num_seqs=70000), api.PA_ERR_UNSUPPORTED),
    (dict(ws=None), api.PA_ERR_WORKSPACE),
    (dict(ws_bytes=16), api.PA_ERR_WORKSPACE),
    (dict(out=A + 8), api.PA_ERR_MISALIGNED),
    (dict(sched=A + 2), api.PA_ERR_MISALIGNED),
])
def test_prefill_host_checks(kw, want):
    assert prefill(**kw) == want


@pytest.mark.parametrize("kw,want", [
    (dict(num_tokens=0), api.PA_OK),
    (dict(num_tokens=-1), api.PA_ERR_INVALID_ARG),
    (dict(block_size=12), api.PA_ERR_UNSUPPORTED),
    (dict(slots=None), api.PA_ERR_INVALID_ARG),
    (dict(k=A + 4), api.PA_ERR_MISALIGNED),
])
def test_reshape_and_cache_host_checks(kw, want):
    assert reshape(**kw) == want


def test_binding_refuses_host_tensors():
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    kc = torch.zeros(4, 2, 16, 64, dtype=torch.bfloat16)
    tables = torch.zeros(2, 2, dtype=torch.int32)
    ctx = torch.ones(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        api.pa_decode(torch.empty_like(q), q, kc, kc, tables, ctx, 16, 0.125, 4, 2, 64, 16)
    with pytest.raises(ValueError, match="CUDA"):
        api.pa_reshape_and_cache(kc, kc, q[:, :2], q[:, :2], torch.zeros(2, dtype=torch.int64))


def copy_blocks(layers_k, layers_v, pairs=A, num_pairs=3, block_size=16, d=128, hkv=8, num_blocks=64):
    arr = lambda xs: (ctypes.c_void_p * max(1, len(xs)))(*xs)
    return L.pa_copy_blocks(arr(layers_k), arr(layers_v), len(layers_k), pairs, num_pairs, hkv, d, block_size,
                            num_blocks, None, None)


@pytest.mark.parametrize("args,want", [
    (dict(layers_k=[], layers_v=[]), api.PA_OK),                     # no layers: nothing to do
    (dict(layers_k=[A], layers_v=[A], num_pairs=0), api.PA_OK),
    (dict(layers_k=[A], layers_v=[A], num_pairs=-1), api.PA_ERR_INVALID_ARG),
    (dict(layers_k=[A], layers_v=[A], block_size=4), api.PA_ERR_UNSUPPORTED),
    (dict(layers_k=[A, None], layers_v=[A, A]), api.PA_ERR_INVALID_ARG),
    (dict(layers_k=[A, A + 8], layers_v=[A, A]), api.PA_ERR_MISALIGNED),
    (dict(layers_k=[A], layers_v=[A], pairs=A + 2), api.PA_ERR_MISALIGNED),
    (dict(layers_k=[A], layers_v=[A], pairs=None), api.PA_ERR_INVALID_ARG),
])
def test_copy_blocks_host_checks(args, want):
    assert copy_blocks(**args) == want


@pytest.mark.parametrize("kw,want", [
    (dict(num_seqs=0), api.PA_OK),
    (dict(max_parts=0), api.PA_ERR_INVALID_ARG),
    (dict(partition=0), api.PA_ERR_INVALID_ARG),
    (dict(out_dtype=3), api.PA_ERR_INVALID_ARG),
    (dict(pm=None), api.PA_ERR_INVALID_ARG),
    (dict(d=2048), api.PA_ERR_UNSUPPORTED),
    (dict(ps=A + 2), api.PA_ERR_MISALIGNED),
])
def test_lse_merge_host_checks(kw, want):
    a = dict(out=A, out_dtype=api.PA_DTYPE_F32, pm=A, ps=A, pacc=A, ctx=A, partition=512, max_parts=4, num_seqs=2,
             hq=8, d=128)
    a.update(kw)
    assert L.pa_lse_merge(a["out"], a["out_dtype"], a["pm"], a["ps"], a["pacc"], a["ctx"], a["partition"],
                          a["max_parts"], a["num_seqs"], a["hq"], a["d"], None) == want


def test_append_and_fp8_host_checks():
    # the fused append needs both new-row arrays, 16-byte aligned
    common = (A, api.PA_DTYPE_BF16, A, A, A)
    rest = (A, A, 16, 0.088, 32, 8, 128, 4, 8, 64, 128, 0, None, 0, None, None)
    assert L.pa_decode_append(*common, None, A, *rest) == api.PA_ERR_INVALID_ARG
    assert L.pa_decode_append(*common, A + 8, A + 8, *rest) == api.PA_ERR_MISALIGNED
    # E4M3 cache write: scales finite and > 0
    assert L.pa_reshape_and_cache_fp8(A, A, A, A, A, 4, 8, 128, 16, 64, 0.0, 1.0, None, None) == api.PA_ERR_INVALID_ARG
    assert L.pa_reshape_and_cache_fp8(A, A, A, A, A, 0, 8, 128, 16, 64, 1.0, 1.0, None, None) == api.PA_OK
    # E4M3 prefill: scales, d_head 128 only
    pf = lambda ks, d: L.pa_prefill_fp8(A, api.PA_DTYPE_BF16, A, A, A, A, 8, A, A, 2, 100, 64, 64, 16, 0.088, ks, 0.01,
                                        32, 8, d, A, 1 << 30, None, None, None)
    assert pf(-1.0, 128) == api.PA_ERR_INVALID_ARG
    assert pf(0.01, 64) == api.PA_ERR_UNSUPPORTED


def swap_blocks(**kw):
    arr = lambda xs: (ctypes.c_void_p * max(1, len(xs)))(*xs)
    a = dict(dst_k=[A], dst_v=[A], src_k=[A], src_v=[A], layers=1, pairs=A, num_pairs=2, hkv=8, d=128, block_size=16,
             src_nb=64, dst_nb=64)
    a.update(kw)
    conv = lambda xs: None if xs is None else arr(xs)
    return L.pa_swap_blocks(conv(a["dst_k"]), conv(a["dst_v"]), conv(a["src_k"]), conv(a["src_v"]), a["layers"],
                            a["pairs"], a["num_pairs"], a["hkv"], a["d"], a["block_size"], a["src_nb"], a["dst_nb"],
                            None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(layers=0), api.PA_OK),                                      # nothing to move
    (dict(num_pairs=0), api.PA_OK),
    (dict(num_pairs=-1), api.PA_ERR_INVALID_ARG),
    (dict(src_nb=0), api.PA_ERR_INVALID_ARG),
    (dict(block_size=12), api.PA_ERR_UNSUPPORTED),
    (dict(d=96), api.PA_ERR_UNSUPPORTED),
    (dict(dst_k=None), api.PA_ERR_INVALID_ARG),
    (dict(pairs=None), api.PA_ERR_INVALID_ARG),
])
def test_swap_blocks_host_checks(kw, want):
    assert swap_blocks(**kw) == want


def test_remaining_entry_points_host_checks():
    """The FP8 copy and swap, the FP8 fused append, the static-scratch decode
    and the bounded-wait self-test reject bad arguments on the host too."""
    arr = lambda xs: (ctypes.c_void_p * max(1, len(xs)))(*xs)
    # FP8 block copies: the same checks as their bf16 forms
    cp8 = lambda ks, bs=16: L.pa_copy_blocks_fp8(arr(ks), arr(ks), len(ks), A, 3, 8, 128, bs, 64, None, None)
    assert cp8([]) == api.PA_OK
    assert cp8([A], bs=4) == api.PA_ERR_UNSUPPORTED
    assert cp8([A + 8]) == api.PA_ERR_MISALIGNED
    sw8 = lambda layers, bs=16: L.pa_swap_blocks_fp8(arr([A]), arr([A]), arr([A]), arr([A]), layers, A, 2, 8, 128,
                                                     bs, 64, 64, None, None)
    assert sw8(0) == api.PA_OK
    assert sw8(1, bs=12) == api.PA_ERR_UNSUPPORTED
    # FP8 fused append: both new-row arrays, finite positive scales
    app8 = lambda kn, ks: L.pa_decode_append_fp8(A, api.PA_DTYPE_F32, A, A, A, kn, A, A, A, 16, 0.088, ks, 0.01, 32, 8,
                                                 128, 4, 8, 64, 128, 0, None, 0, None, None)
    assert app8(None, 0.01) == api.PA_ERR_INVALID_ARG
    assert app8(A, 0.0) == api.PA_ERR_INVALID_ARG
    assert app8(A, float("nan")) == api.PA_ERR_INVALID_ARG
    # static scratch: a problem whose partition statistics exceed the array is refused up front
    ss = lambda S, hq, max_ctx, P: L.pa_decode_static_scratch(A, api.PA_DTYPE_BF16, A, A, A, A, A, 16, 0.088, hq, 8,
                                                              128, S, 8, 64, max_ctx, P, None, None)
    assert ss(1024, 64, 1 << 20, 256) == api.PA_ERR_WORKSPACE
    assert ss(0, 32, 128, 512) == api.PA_OK
    # the bounded-wait self-test: probe limit in [1, 10^7] and a status word
    assert L.pa_check_bounded_wait(0, A, None) == api.PA_ERR_INVALID_ARG
    assert L.pa_check_bounded_wait(10 ** 7 + 1, A, None) == api.PA_ERR_INVALID_ARG
    assert L.pa_check_bounded_wait(100, None, None) == api.PA_ERR_INVALID_ARG
