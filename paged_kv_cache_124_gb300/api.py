"""Python binding of the C ABI in include/pa.h (ctypes; marshalling only).

Every function here checks tensor placement, dtype and shape, turns tensors
into raw pointers and sizes, and calls the library entry point of the same
name.  All computation happens in libpa_gb300.so; if the library is missing
this module raises at import time rather than computing anything itself.
"""

import ctypes
import os
import re

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa_gb300.so")
_HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")

PA_OK = 0
PA_FAIL_NO_BLOCKS = 1
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_MISALIGNED = -3
PA_ERR_CUDA = -4
PA_ERR_WORKSPACE = -5
PA_ERR_UNKNOWN_SEQ = -6
PA_ERR_DUPLICATE_SEQ = -7
PA_ERR_SWAPPED = -8

PA_DEV_BAD_BLOCK_ID = 1
PA_DEV_BAD_SLOT = 2
PA_DEV_BAD_CONTEXT = 4
PA_DEV_WAIT_TIMEOUT = 8

PA_DTYPE_BF16 = 0
PA_DTYPE_F32 = 1


class PAError(RuntimeError):
    def __init__(self, status, where):
        super().__init__("%s failed: %s (%d)" % (where, status_string(status), status))
        self.status = status


if not os.path.exists(_LIB_PATH):
    raise ImportError("libpa_gb300.so has not been built (python -m paged_kv_cache_124_gb300.build); "
                      "there is no fallback implementation")

_lib = ctypes.CDLL(_LIB_PATH)

_c_int, _c_size, _c_float = ctypes.c_int, ctypes.c_size_t, ctypes.c_float
_vp, _i32p, _i64p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
_f32p = ctypes.POINTER(ctypes.c_float)


class AllocStats(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("num_free", ctypes.c_int32), ("num_used", ctypes.c_int32),
                ("num_seqs", ctypes.c_int32), ("num_cow_copies", ctypes.c_int64), ("num_cached", ctypes.c_int32),
                ("num_swapped", ctypes.c_int32), ("num_prompt_tokens", ctypes.c_int64),
                ("num_cached_tokens", ctypes.c_int64), ("num_swap_outs", ctypes.c_int64),
                ("num_context_tokens", ctypes.c_int64)]


_SIGS = {
    "pa_version": (ctypes.c_char_p, []),
    "pa_status_string": (ctypes.c_char_p, [_c_int]),
    "pa_decode_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_decode": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_float, _c_int, _c_int, _c_int,
                           _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp, _vp]),
    "pa_decode_static_scratch": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_float, _c_int, _c_int,
                                          _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp]),
    "pa_decode_fp8": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _vp, _c_int, _c_float, _c_float, _c_float, _c_int,
                               _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp, _vp]),
    "pa_decode_append": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_float, _c_int, _c_int,
                                  _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp, _vp]),
    "pa_decode_append_fp8": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _c_int, _c_float, _c_float,
                                      _c_float, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                      _c_size, _vp, _vp]),
    "pa_reshape_and_cache_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_float,
                                          _c_float, _vp, _vp]),
    "pa_prefill": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                            _c_int, _c_float, _c_int, _c_int, _c_int, _vp, _c_size, _vp, _vp, _vp]),
    "pa_prefill_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_prefill_fp8": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _c_int, _vp, _vp, _c_int, _c_int, _c_int, _c_int,
                                _c_int, _c_float, _c_float, _c_float, _c_int, _c_int, _c_int, _vp, _c_size, _vp, _vp,
                                _vp]),
    "pa_prefill_fp8_workspace_size": (_c_size, [_c_int, _c_int, _c_int, _c_int, _c_int]),
    "pa_check_bounded_wait": (_c_int, [_c_int, _vp, _vp]),
    "pa_lse_merge": (_c_int, [_vp, _c_int, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp]),
    "pa_reshape_and_cache": (_c_int, [_vp, _vp, _vp, _vp, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                      _vp]),
    "pa_copy_blocks": (_c_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _c_int, _vp, _c_int, _c_int, _c_int,
                                _c_int, _c_int, _vp, _vp]),
    "pa_copy_blocks_fp8": (_c_int, [ctypes.POINTER(_vp), ctypes.POINTER(_vp), _c_int, _vp, _c_int, _c_int, _c_int,
                                    _c_int, _c_int, _vp, _vp]),
    "pa_alloc_create": (_vp, [_c_int, _c_int]),
    "pa_alloc_destroy": (None, [_vp]),
    "pa_alloc_set_free_order": (_c_int, [_vp, _i32p, _c_int]),
    "pa_alloc_sequence": (_c_int, [_vp, ctypes.c_int64, _c_int]),
    "pa_alloc_fork": (_c_int, [_vp, ctypes.c_int64, ctypes.c_int64]),
    "pa_alloc_append_slot": (_c_int, [_vp, ctypes.c_int64, _i64p, _i32p, _i32p]),
    "pa_alloc_append_slots": (_c_int, [_vp, _i64p, _c_int, _i64p, _i32p, _c_int, ctypes.POINTER(_c_int),
                                       ctypes.POINTER(_c_int)]),
    "pa_alloc_free": (_c_int, [_vp, ctypes.c_int64]),
    "pa_alloc_block_table": (_c_int, [_vp, ctypes.c_int64, _i32p, _c_int, ctypes.POINTER(_c_int)]),
    "pa_alloc_build_tables": (_c_int, [_vp, _i64p, _c_int, _i32p, _c_int, _i32p]),
    "pa_alloc_slot_mapping": (_c_int, [_vp, ctypes.c_int64, _c_int, _c_int, _i64p]),
    "pa_alloc_seq_len": (_c_int, [_vp, ctypes.c_int64]),
    "pa_alloc_ref_count": (_c_int, [_vp, ctypes.c_int32]),
    "pa_alloc_num_free": (_c_int, [_vp]),
    "pa_alloc_free_list": (_c_int, [_vp, _i32p, _c_int]),
    "pa_alloc_get_stats": (_c_int, [_vp, ctypes.POINTER(AllocStats)]),
    "pa_alloc_enable_prefix_caching": (_c_int, [_vp, _c_int]),
    "pa_alloc_set_key_mask": (_c_int, [_vp, ctypes.c_uint64]),
    "pa_alloc_num_prefix_nodes": (_c_int, [_vp]),
    "pa_alloc_sequence_tokens": (_c_int, [_vp, ctypes.c_int64, _i32p, _c_int, ctypes.POINTER(_c_int)]),
    "pa_alloc_append_token": (_c_int, [_vp, ctypes.c_int64, ctypes.c_int32, _i64p, _i32p, _i32p]),
    "pa_alloc_num_cached": (_c_int, [_vp]),
    "pa_alloc_enable_swap": (_c_int, [_vp, _c_int]),
    "pa_alloc_swap_out": (_c_int, [_vp, _i64p, _c_int, _i32p, _c_int, ctypes.POINTER(_c_int)]),
    "pa_alloc_swap_in": (_c_int, [_vp, _i64p, _c_int, _i32p, _c_int, ctypes.POINTER(_c_int)]),
    "pa_alloc_num_free_host": (_c_int, [_vp]),
    "pa_alloc_is_swapped": (_c_int, [_vp, ctypes.c_int64]),
    "pa_swap_blocks": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp,
                                _vp]),
    "pa_swap_blocks_fp8": (_c_int, [_vp, _vp, _vp, _vp, _c_int, _vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int,
                                    _vp, _vp]),
    "pa_alloc_cached_list": (_c_int, [_vp, _i32p, _c_int]),
}

for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


def library_path():
    return _LIB_PATH


def header_functions():
    """Names of the functions include/pa.h declares."""
    text = open(_HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def version():
    return _lib.pa_version().decode()


def status_string(status):
    return _lib.pa_status_string(int(status)).decode()


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _check(status, where):
    if status < 0:
        raise PAError(status, where)
    return status


def _dev(t, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _opt_dev(t, dtype, name):
    return ctypes.c_void_p(0) if t is None else _dev(t, dtype, name)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


# ----------------------------------------------------------------------------
# kernels
# ----------------------------------------------------------------------------

def pa_decode_workspace_size(num_seqs, n_q_heads, d_head, max_context_len, partition_size=0):
    return int(_lib.pa_decode_workspace_size(num_seqs, n_q_heads, d_head, max_context_len, partition_size))


def decode_workspace(num_seqs, n_q_heads, d_head, max_context_len, partition_size=0, device=None):
    """A caller-owned workspace tensor (uint8) of the size pa_decode needs,
    or None when no workspace is needed."""
    n = pa_decode_workspace_size(num_seqs, n_q_heads, d_head, max_context_len, partition_size)
    if n == 0:
        return None
    # zeroed: the header's claim counters must be zero before the first call
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, n_q_heads,
              n_kv_heads, d_head, max_context_len, partition_size=0, workspace=None, status=None,
              stream=None):
    """out [S, Hq, D] (bf16 or f32) <- paged decode attention; see pa.h."""
    if out.dtype == torch.bfloat16:
        out_dtype = PA_DTYPE_BF16
    elif out.dtype == torch.float32:
        out_dtype = PA_DTYPE_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    num_seqs = q.shape[0]
    if tuple(q.shape) != (num_seqs, n_q_heads, d_head) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [num_seqs, n_q_heads, d_head]")
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (n_kv_heads, block_size, d_head) or \
            k_cache.shape != v_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, n_kv_heads, block_size, d_head]")
    if block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or context_lens.shape != (num_seqs,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], context_lens [num_seqs]")
    ws_ptr = ctypes.c_void_p(0)
    ws_bytes = 0
    if workspace is not None:
        ws_ptr = _dev(workspace, torch.uint8, "workspace")
        ws_bytes = workspace.numel()
    st = _lib.pa_decode(_opt_dev(out, out.dtype, "out"), out_dtype, _dev(q, torch.bfloat16, "q"),
                        _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
                        _dev(block_tables, torch.int32, "block_tables"),
                        _dev(context_lens, torch.int32, "context_lens"), int(block_size), float(scale),
                        int(n_q_heads), int(n_kv_heads), int(d_head), int(num_seqs), int(block_tables.shape[1]),
                        int(k_cache.shape[0]), int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
                        _opt_dev(status, torch.int32, "status"), _stream(stream))
    return _check(st, "pa_decode")


def pa_decode_append(out, q, k_cache, v_cache, k_new, v_new, block_tables, context_lens, block_size, scale,
                     n_q_heads, n_kv_heads, d_head, max_context_len, partition_size=0, workspace=None, status=None,
                     stream=None, k_scale=None, v_scale=None):
    """The step's cache write and decode in one call: k_new / v_new [S, Hkv, D]
    bf16 are the keys and values of position context_lens[s] - 1, written at
    its slot and attended to (bit-equal to pa_reshape_and_cache + pa_decode);
    with k_scale / v_scale, the E4M3 form (uint8 caches); see pa.h."""
    f8 = k_scale is not None
    if out.dtype == torch.bfloat16:
        out_dtype = PA_DTYPE_BF16
    elif out.dtype == torch.float32:
        out_dtype = PA_DTYPE_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    num_seqs = q.shape[0]
    if tuple(q.shape) != (num_seqs, n_q_heads, d_head) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [num_seqs, n_q_heads, d_head]")
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (n_kv_heads, block_size, d_head) or \
            k_cache.shape != v_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, n_kv_heads, block_size, d_head]")
    if tuple(k_new.shape) != (num_seqs, n_kv_heads, d_head) or k_new.shape != v_new.shape:
        raise ValueError("k_new/v_new must be [num_seqs, n_kv_heads, d_head]")
    if block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or context_lens.shape != (num_seqs,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], context_lens [num_seqs]")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, torch.uint8, "workspace")
        ws_bytes = workspace.numel()
    cache_dtype = torch.uint8 if f8 else torch.bfloat16
    args = [_opt_dev(out, out.dtype, "out"), out_dtype, _dev(q, torch.bfloat16, "q"),
            _dev(k_cache, cache_dtype, "k_cache"), _dev(v_cache, cache_dtype, "v_cache"),
            _dev(k_new, torch.bfloat16, "k_new"), _dev(v_new, torch.bfloat16, "v_new"),
            _dev(block_tables, torch.int32, "block_tables"), _dev(context_lens, torch.int32, "context_lens"),
            int(block_size), float(scale)]
    if f8:
        args += [float(k_scale), float(v_scale)]
    args += [int(n_q_heads), int(n_kv_heads), int(d_head), int(num_seqs), int(block_tables.shape[1]),
             int(k_cache.shape[0]), int(max_context_len), int(partition_size), ws_ptr, ws_bytes,
             _opt_dev(status, torch.int32, "status"), _stream(stream)]
    name = "pa_decode_append_fp8" if f8 else "pa_decode_append"
    return _check(getattr(_lib, name)(*args), name)


_prefill_counters = {}


def prefill_counters(device, stream=None):
    """The two zeroed int32 work-claim counters pa_prefill uses on this device
    and stream (each call leaves them zero again); one pair per stream, since
    calls sharing a pair must not overlap."""
    dev = torch.device(device)
    handle = _stream(stream).value or 0
    key = (dev.index if dev.index is not None else torch.cuda.current_device(), handle)
    t = _prefill_counters.get(key)
    if t is None:
        t = torch.zeros(2, dtype=torch.int32, device=dev)
        _prefill_counters[key] = t
    return t


def pa_prefill_workspace_size(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head):
    return int(_lib.pa_prefill_workspace_size(int(num_seqs), int(max_blocks_per_seq), int(block_size),
                                              int(n_kv_heads), int(d_head)))


def prefill_workspace(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head, device=None):
    """A caller-owned workspace tensor (uint8) of the size pa_prefill needs."""
    n = pa_prefill_workspace_size(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")


def pa_prefill(out, q, k_cache, v_cache, block_tables, query_start, context_lens, max_query_len, block_size,
               scale, n_q_heads, n_kv_heads, d_head, status=None, stream=None, counters=None, workspace=None):
    """out [T, Hq, D] (bf16 or f32) <- causal paged prefill attention of the
    new positions of each sequence; see pa.h.  `counters`: the int32 [2]
    work-claim pair (default: this stream's, from prefill_counters; False:
    none, a fixed round-robin assignment of work).  `workspace`: a uint8
    device tensor of at least pa_prefill_workspace_size bytes (default: one
    allocated for this call through PyTorch's caching allocator)."""
    if out.dtype == torch.bfloat16:
        out_dtype = PA_DTYPE_BF16
    elif out.dtype == torch.float32:
        out_dtype = PA_DTYPE_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    num_tokens = q.shape[0]
    if tuple(q.shape) != (num_tokens, n_q_heads, d_head) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [num_tokens, n_q_heads, d_head]")
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (n_kv_heads, block_size, d_head) or \
            k_cache.shape != v_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, n_kv_heads, block_size, d_head]")
    if counters is None:
        counters = prefill_counters(q.device, stream)
    if counters is not False and counters.numel() < 2:
        raise ValueError("counters must hold 2 int32")
    num_seqs = block_tables.shape[0]
    if block_tables.dim() != 2 or context_lens.shape != (num_seqs,) or query_start.shape != (num_seqs + 1,):
        raise ValueError("block_tables [S, max_blocks], query_start [S + 1], context_lens [S]")
    if workspace is None:
        workspace = prefill_workspace(num_seqs, block_tables.shape[1], block_size, n_kv_heads, d_head, q.device)
    st = _lib.pa_prefill(_opt_dev(out, out.dtype, "out"), out_dtype, _dev(q, torch.bfloat16, "q"),
                         _dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
                         _dev(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
                         _dev(query_start, torch.int32, "query_start"), _dev(context_lens, torch.int32, "context_lens"),
                         int(num_seqs), int(num_tokens), int(max_query_len), int(k_cache.shape[0]), int(block_size),
                         float(scale), int(n_q_heads), int(n_kv_heads), int(d_head),
                         _dev(workspace, torch.uint8, "workspace"), int(workspace.numel()),
                         _opt_dev(None if counters is False else counters, torch.int32, "counters"),
                         _opt_dev(status, torch.int32, "status"),
                         _stream(stream))
    return _check(st, "pa_prefill")


def pa_prefill_fp8_workspace_size(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head):
    return int(_lib.pa_prefill_fp8_workspace_size(int(num_seqs), int(max_blocks_per_seq), int(block_size),
                                                  int(n_kv_heads), int(d_head)))


def prefill_fp8_workspace(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head, device=None):
    """A caller-owned workspace tensor (uint8) of the size pa_prefill_fp8 needs."""
    n = pa_prefill_fp8_workspace_size(num_seqs, max_blocks_per_seq, block_size, n_kv_heads, d_head)
    return torch.empty(max(n, 1), dtype=torch.uint8, device=device or "cuda")


def pa_prefill_fp8(out, q, k_cache, v_cache, block_tables, query_start, context_lens, max_query_len, block_size,
                   scale, k_scale, v_scale, n_q_heads, n_kv_heads, d_head, status=None, stream=None, counters=None,
                   workspace=None):
    """pa_prefill over E4M3 caches (uint8 [num_blocks, Hkv, B, D]) with per-cache scales; see pa.h."""
    if out.dtype == torch.bfloat16:
        out_dtype = PA_DTYPE_BF16
    elif out.dtype == torch.float32:
        out_dtype = PA_DTYPE_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    num_tokens = q.shape[0]
    if tuple(q.shape) != (num_tokens, n_q_heads, d_head) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [num_tokens, n_q_heads, d_head]")
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (n_kv_heads, block_size, d_head) or \
            k_cache.shape != v_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, n_kv_heads, block_size, d_head]")
    if counters is None:
        counters = prefill_counters(q.device, stream)
    if counters is not False and counters.numel() < 2:
        raise ValueError("counters must hold 2 int32")
    num_seqs = block_tables.shape[0]
    if block_tables.dim() != 2 or context_lens.shape != (num_seqs,) or query_start.shape != (num_seqs + 1,):
        raise ValueError("block_tables [S, max_blocks], query_start [S + 1], context_lens [S]")
    if workspace is None:
        workspace = prefill_fp8_workspace(num_seqs, block_tables.shape[1], block_size, n_kv_heads, d_head, q.device)
    st = _lib.pa_prefill_fp8(_opt_dev(out, out.dtype, "out"), out_dtype, _dev(q, torch.bfloat16, "q"),
                             _dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"),
                             _dev(block_tables, torch.int32, "block_tables"), int(block_tables.shape[1]),
                             _dev(query_start, torch.int32, "query_start"),
                             _dev(context_lens, torch.int32, "context_lens"), int(num_seqs), int(num_tokens),
                             int(max_query_len), int(k_cache.shape[0]), int(block_size), float(scale), float(k_scale),
                             float(v_scale), int(n_q_heads), int(n_kv_heads), int(d_head),
                             _dev(workspace, torch.uint8, "workspace"), int(workspace.numel()),
                             _opt_dev(None if counters is False else counters, torch.int32, "counters"),
                             _opt_dev(status, torch.int32, "status"), _stream(stream))
    return _check(st, "pa_prefill_fp8")


def pa_decode_fp8(out, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, k_scale, v_scale,
                  n_q_heads, n_kv_heads, d_head, max_context_len, partition_size=0, workspace=None, status=None,
                  stream=None):
    """pa_decode over E4M3 caches (uint8 [num_blocks, Hkv, B, D]) with per-cache scales; see pa.h."""
    if out.dtype == torch.bfloat16:
        out_dtype = PA_DTYPE_BF16
    elif out.dtype == torch.float32:
        out_dtype = PA_DTYPE_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    num_seqs = q.shape[0]
    if tuple(q.shape) != (num_seqs, n_q_heads, d_head) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [num_seqs, n_q_heads, d_head]")
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (n_kv_heads, block_size, d_head) or \
            k_cache.shape != v_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, n_kv_heads, block_size, d_head]")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr = _dev(workspace, torch.uint8, "workspace")
        ws_bytes = workspace.numel()
    st = _lib.pa_decode_fp8(_opt_dev(out, out.dtype, "out"), out_dtype, _dev(q, torch.bfloat16, "q"),
                            _dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"),
                            _dev(block_tables, torch.int32, "block_tables"),
                            _dev(context_lens, torch.int32, "context_lens"), int(block_size), float(scale),
                            float(k_scale), float(v_scale), int(n_q_heads), int(n_kv_heads), int(d_head),
                            int(num_seqs), int(block_tables.shape[1]), int(k_cache.shape[0]), int(max_context_len),
                            int(partition_size), ws_ptr, ws_bytes, _opt_dev(status, torch.int32, "status"),
                            _stream(stream))
    return _check(st, "pa_decode_fp8")


def pa_reshape_and_cache_fp8(k_cache, v_cache, k, v, slot_mapping, k_scale, v_scale, status=None, stream=None):
    """Quantise k[t], v[t] ([T, Hkv, D] bf16) to E4M3 codes in the slots slot_mapping[t] of uint8 caches."""
    NB, Hkv, B, D = k_cache.shape
    T = slot_mapping.shape[0]
    if tuple(k.shape) != (T, Hkv, D) or k.shape != v.shape:
        raise ValueError("k/v must be [num_tokens, n_kv_heads, d_head]")
    st = _lib.pa_reshape_and_cache_fp8(_dev(k_cache, torch.uint8, "k_cache"), _dev(v_cache, torch.uint8, "v_cache"),
                                       _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                                       _dev(slot_mapping, torch.int64, "slot_mapping"), int(T), int(Hkv), int(D),
                                       int(B), int(NB), float(k_scale), float(v_scale),
                                       _opt_dev(status, torch.int32, "status"), _stream(stream))
    return _check(st, "pa_reshape_and_cache_fp8")


PA_STATIC_SCRATCH_BYTES = 16 << 20


def pa_decode_static_scratch(out, q, k_cache, v_cache, block_tables, context_lens, block_size, scale, n_q_heads,
                             n_kv_heads, d_head, max_context_len, partition_size=0, status=None, stream=None):
    """pa_decode for callers that cannot supply device scratch memory: the
    library keeps the split path's partition statistics in its own static
    device array (PA_STATIC_SCRATCH_BYTES) and allocates nothing.  Larger
    problems raise PAError(PA_ERR_WORKSPACE).  Calls share that array, so
    calls running at the same time on the GPU must not overlap."""
    if out.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("out must be bfloat16 or float32")
    num_seqs = q.shape[0]
    if tuple(q.shape) != (num_seqs, n_q_heads, d_head) or tuple(out.shape) != tuple(q.shape):
        raise ValueError("q/out must be [num_seqs, n_q_heads, d_head]")
    if k_cache.dim() != 4 or tuple(k_cache.shape[1:]) != (n_kv_heads, block_size, d_head) or \
            k_cache.shape != v_cache.shape:
        raise ValueError("k_cache/v_cache must be [num_blocks, n_kv_heads, block_size, d_head]")
    if block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or context_lens.shape != (num_seqs,):
        raise ValueError("block_tables must be [num_seqs, max_blocks], context_lens [num_seqs]")
    out_dtype = PA_DTYPE_F32 if out.dtype == torch.float32 else PA_DTYPE_BF16
    st = _lib.pa_decode_static_scratch(
        _dev(out, out.dtype, "out"), out_dtype, _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        _dev(context_lens, torch.int32, "context_lens"), int(block_size), float(scale), int(n_q_heads),
        int(n_kv_heads), int(d_head), int(num_seqs), int(block_tables.shape[1]), int(k_cache.shape[0]),
        int(max_context_len), int(partition_size), _opt_dev(status, torch.int32, "status"), _stream(stream))
    return _check(st, "pa_decode_static_scratch")


def pa_lse_merge(out, part_max, part_sum, part_acc, context_lens, partition_size, stream=None):
    """out [S, Hq, D] <- exact merge of partition statistics
    part_max/part_sum [S, Hq, NP], part_acc [S, Hq, NP, D] (f32)."""
    S, Hq, NP, D = part_acc.shape
    if tuple(part_max.shape) != (S, Hq, NP) or tuple(part_sum.shape) != (S, Hq, NP):
        raise ValueError("part_max/part_sum must be [S, Hq, NP]")
    out_dtype = PA_DTYPE_F32 if out.dtype == torch.float32 else PA_DTYPE_BF16
    st = _lib.pa_lse_merge(_dev(out, out.dtype, "out"), out_dtype, _dev(part_max, torch.float32, "part_max"),
                           _dev(part_sum, torch.float32, "part_sum"), _dev(part_acc, torch.float32, "part_acc"),
                           _dev(context_lens, torch.int32, "context_lens"), int(partition_size), int(NP), int(S),
                           int(Hq), int(D), _stream(stream))
    return _check(st, "pa_lse_merge")


def pa_reshape_and_cache(k_cache, v_cache, k, v, slot_mapping, status=None, stream=None):
    """Write k[t], v[t] ([T, Hkv, D] bf16) into the slots slot_mapping[t] (int64)."""
    NB, Hkv, B, D = k_cache.shape
    T = slot_mapping.shape[0]
    if tuple(k.shape) != (T, Hkv, D) or k.shape != v.shape:
        raise ValueError("k/v must be [num_tokens, n_kv_heads, d_head]")
    st = _lib.pa_reshape_and_cache(_dev(k_cache, torch.bfloat16, "k_cache"), _dev(v_cache, torch.bfloat16, "v_cache"),
                                   _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                                   _dev(slot_mapping, torch.int64, "slot_mapping"), int(T), int(Hkv), int(D), int(B),
                                   int(NB), _opt_dev(status, torch.int32, "status"), _stream(stream))
    return _check(st, "pa_reshape_and_cache")


def pa_copy_blocks(k_caches, v_caches, block_pairs, status=None, stream=None):
    """For every (src, dst) row of block_pairs (int32 [P, 2], device) copy
    block src onto block dst in every layer's caches (bf16, or uint8 E4M3
    codes: pa_copy_blocks_fp8)."""
    L = len(k_caches)
    if len(v_caches) != L:
        raise ValueError("k_caches and v_caches must have the same length")
    P = block_pairs.shape[0] if block_pairs is not None else 0
    if L == 0 or P == 0:
        return PA_OK
    NB, Hkv, B, D = k_caches[0].shape
    for t in list(k_caches) + list(v_caches):
        if tuple(t.shape) != (NB, Hkv, B, D):
            raise ValueError("all caches must share one shape")
    fp8 = k_caches[0].dtype == torch.uint8
    dt = torch.uint8 if fp8 else torch.bfloat16
    fn = _lib.pa_copy_blocks_fp8 if fp8 else _lib.pa_copy_blocks
    kp = (ctypes.c_void_p * L)(*[_dev(t, dt, "k_caches[i]").value for t in k_caches])
    vp = (ctypes.c_void_p * L)(*[_dev(t, dt, "v_caches[i]").value for t in v_caches])
    st = fn(kp, vp, L, _dev(block_pairs, torch.int32, "block_pairs"), int(P), int(Hkv), int(D),
            int(B), int(NB), _opt_dev(status, torch.int32, "status"), _stream(stream))
    return _check(st, "pa_copy_blocks_fp8" if fp8 else "pa_copy_blocks")


def _dev_or_pinned(t, dtype, name):
    """Pointer of a CUDA tensor or of a page-locked host tensor."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("%s must be a CUDA tensor or a page-locked (pinned) host tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def pa_check_bounded_wait(status, max_probes=20000, stream=None):
    """Run the kernels' bounded-wait failure path on a barrier nothing arrives
    on: status (device int32) receives PA_DEV_WAIT_TIMEOUT; see pa.h."""
    return _check(_lib.pa_check_bounded_wait(int(max_probes), _dev(status, torch.int32, "status"), _stream(stream)),
                  "pa_check_bounded_wait")


def pa_swap_blocks(dst_k, dst_v, src_k, src_v, block_pairs, status=None, stream=None):
    """For every (src, dst) row of block_pairs (int32 [P, 2]) copy block src
    of every src pool onto block dst of the matching dst pool.  Pools are
    lists (one per layer) of CUDA or pinned host tensors [num_blocks, Hkv, B,
    D], bf16 or uint8 E4M3 codes (pa_swap_blocks_fp8); source and destination
    may differ in num_blocks."""
    L = len(src_k)
    if not (len(src_v) == len(dst_k) == len(dst_v) == L):
        raise ValueError("the four pool lists must have the same length")
    P = block_pairs.shape[0] if block_pairs is not None else 0
    if L == 0 or P == 0:
        return PA_OK
    SNB, Hkv, B, D = src_k[0].shape
    DNB = dst_k[0].shape[0]
    for t in list(src_k) + list(src_v):
        if tuple(t.shape) != (SNB, Hkv, B, D):
            raise ValueError("source pools must share one shape")
    for t in list(dst_k) + list(dst_v):
        if tuple(t.shape) != (DNB, Hkv, B, D):
            raise ValueError("destination pools must share one shape")
    fp8 = src_k[0].dtype == torch.uint8
    dt = torch.uint8 if fp8 else torch.bfloat16
    fn = _lib.pa_swap_blocks_fp8 if fp8 else _lib.pa_swap_blocks
    arr = lambda ts, nm: (ctypes.c_void_p * L)(*[_dev_or_pinned(t, dt, nm).value for t in ts])
    st = fn(arr(dst_k, "dst_k"), arr(dst_v, "dst_v"), arr(src_k, "src_k"), arr(src_v, "src_v"), L,
            _dev_or_pinned(block_pairs, torch.int32, "block_pairs"), int(P), int(Hkv), int(D), int(B),
            int(SNB), int(DNB), _opt_dev(status, torch.int32, "status"), _stream(stream))
    return _check(st, "pa_swap_blocks_fp8" if fp8 else "pa_swap_blocks")


# ----------------------------------------------------------------------------
# host block manager
# ----------------------------------------------------------------------------

def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_i32p)


def _i64(a):
    a = np.ascontiguousarray(a, dtype=np.int64)
    return a, a.ctypes.data_as(_i64p)


class BlockAllocator:
    """The C++ block manager (pa_alloc_*).  Methods return the library's
    status codes; PA_FAIL_NO_BLOCKS is a normal outcome, not an exception."""

    def __init__(self, num_blocks, block_size):
        self._h = _lib.pa_alloc_create(int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("pa_alloc_create(%r, %r) failed" % (num_blocks, block_size))
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            _lib.pa_alloc_destroy(h)

    def set_free_order(self, order):
        arr, p = _i32(order)
        return _lib.pa_alloc_set_free_order(self._h, p, len(arr))

    def allocate(self, seq, num_tokens):
        return _lib.pa_alloc_sequence(self._h, int(seq), int(num_tokens))

    def fork(self, parent, child):
        return _lib.pa_alloc_fork(self._h, int(parent), int(child))

    def enable_prefix_caching(self, enable=True):
        return _lib.pa_alloc_enable_prefix_caching(self._h, 1 if enable else 0)

    def set_key_mask(self, mask):
        """Testing hook: bucket the interned prefixes by hash & mask (0: one
        bucket, every lookup meets colliding candidates)."""
        return _lib.pa_alloc_set_key_mask(self._h, int(mask) & 0xFFFFFFFFFFFFFFFF)

    def num_prefix_nodes(self):
        return _lib.pa_alloc_num_prefix_nodes(self._h)

    def allocate_tokens(self, seq, tokens):
        """New sequence with known prompt token ids.  Returns (status,
        num_cached_tokens): the leading positions found in the prefix cache,
        whose KV is already in the pool."""
        arr, p = _i32(tokens)
        hit = ctypes.c_int(0)
        st = _lib.pa_alloc_sequence_tokens(self._h, int(seq), p, len(arr), ctypes.byref(hit))
        return st, hit.value

    def append_token(self, seq, token):
        slot, src, dst = ctypes.c_int64(-1), ctypes.c_int32(-1), ctypes.c_int32(-1)
        st = _lib.pa_alloc_append_token(self._h, int(seq), int(token), ctypes.byref(slot), ctypes.byref(src),
                                        ctypes.byref(dst))
        return st, slot.value, src.value, dst.value

    def num_cached(self):
        return _lib.pa_alloc_num_cached(self._h)

    def enable_swap(self, num_host_blocks):
        return _lib.pa_alloc_enable_swap(self._h, int(num_host_blocks))

    def _swap(self, fn, seqs):
        seqs, sp = _i64(seqs)
        cap = max(1, sum(len(self.block_table(int(q))) for q in seqs if self.seq_len(int(q)) >= 0))
        pairs = np.zeros((cap, 2), dtype=np.int32)
        n = ctypes.c_int(0)
        st = fn(self._h, sp, len(seqs), pairs.ctypes.data_as(_i32p), cap, ctypes.byref(n))
        return st, (pairs[:n.value].copy() if st == 0 else np.zeros((0, 2), dtype=np.int32))

    def swap_out(self, seqs):
        """Returns (status, pairs [k, 2] int32 of (device block, host block))."""
        return self._swap(_lib.pa_alloc_swap_out, seqs)

    def swap_in(self, seqs):
        """Returns (status, pairs [k, 2] int32 of (host block, device block))."""
        return self._swap(_lib.pa_alloc_swap_in, seqs)

    def num_free_host(self):
        return _lib.pa_alloc_num_free_host(self._h)

    def is_swapped(self, seq):
        return _lib.pa_alloc_is_swapped(self._h, int(seq))

    def cached_list(self):
        """Zero-count cached blocks, next to be evicted first."""
        n = _lib.pa_alloc_cached_list(self._h, None, 0)
        out = np.zeros(max(n, 1), dtype=np.int32)
        _lib.pa_alloc_cached_list(self._h, out.ctypes.data_as(_i32p), n)
        return out[:n].tolist()

    def append_slot(self, seq):
        slot, src, dst = ctypes.c_int64(-1), ctypes.c_int32(-1), ctypes.c_int32(-1)
        st = _lib.pa_alloc_append_slot(self._h, int(seq), ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst))
        return st, slot.value, src.value, dst.value

    def append_slots(self, seqs):
        """Plan one position for each sequence.  Returns (status, slots[n]
        int64, cow_pairs[k, 2] int32, num_done)."""
        seqs, sp = _i64(seqs)
        n = len(seqs)
        slots = np.full(n, -1, dtype=np.int64)
        pairs = np.zeros((max(n, 1), 2), dtype=np.int32)
        ncow, ndone = ctypes.c_int(0), ctypes.c_int(0)
        st = _lib.pa_alloc_append_slots(self._h, sp, n, slots.ctypes.data_as(_i64p),
                                        pairs.ctypes.data_as(_i32p), max(n, 1), ctypes.byref(ncow),
                                        ctypes.byref(ndone))
        return st, slots, pairs[:ncow.value].copy(), ndone.value

    def free(self, seq):
        return _lib.pa_alloc_free(self._h, int(seq))

    def block_table(self, seq):
        n = ctypes.c_int(0)
        st = _lib.pa_alloc_block_table(self._h, int(seq), None, 0, ctypes.byref(n))
        if st == PA_ERR_UNKNOWN_SEQ:
            raise KeyError(seq)
        out = np.zeros(max(n.value, 1), dtype=np.int32)
        _check(_lib.pa_alloc_block_table(self._h, int(seq), out.ctypes.data_as(_i32p), len(out), ctypes.byref(n)),
               "pa_alloc_block_table")
        return out[:n.value].tolist()

    def build_tables(self, seqs, max_blocks):
        seqs, sp = _i64(seqs)
        tables = np.zeros((len(seqs), max_blocks), dtype=np.int32)
        ctx = np.zeros(len(seqs), dtype=np.int32)
        _check(_lib.pa_alloc_build_tables(self._h, sp, len(seqs), tables.ctypes.data_as(_i32p), int(max_blocks),
                                          ctx.ctypes.data_as(_i32p)), "pa_alloc_build_tables")
        return tables, ctx

    def slot_mapping(self, seq, start, n):
        out = np.zeros(max(n, 1), dtype=np.int64)
        _check(_lib.pa_alloc_slot_mapping(self._h, int(seq), int(start), int(n), out.ctypes.data_as(_i64p)),
               "pa_alloc_slot_mapping")
        return out[:n]

    def seq_len(self, seq):
        return _lib.pa_alloc_seq_len(self._h, int(seq))

    def ref_count(self, block):
        return _lib.pa_alloc_ref_count(self._h, int(block))

    def num_free(self):
        return _lib.pa_alloc_num_free(self._h)

    def free_list(self):
        n = _lib.pa_alloc_free_list(self._h, None, 0)
        out = np.zeros(max(n, 1), dtype=np.int32)
        _lib.pa_alloc_free_list(self._h, out.ctypes.data_as(_i32p), n)
        return out[:n].tolist()

    def stats(self):
        s = AllocStats()
        _check(_lib.pa_alloc_get_stats(self._h, ctypes.byref(s)), "pa_alloc_get_stats")
        d = {f: getattr(s, f) for f, _ in AllocStats._fields_}
        d["prefix_cache_hit_rate"] = d["num_cached_tokens"] / d["num_prompt_tokens"] if d["num_prompt_tokens"] else 0.0
        return d

    def metrics(self):
        """The pool's operational metrics: the share of blocks held by
        sequences (percent; zero-count cached blocks are reclaimable and not
        counted), sequences swapped out to host memory since creation (each
        swap-out is a preemption), the share of admitted prompt positions
        found in the prefix cache, and the mean length of the live
        sequences."""
        st = self.stats()
        return {"gpu_cache_usage_perc": 100.0 * st["num_used"] / st["num_blocks"],
                "num_preemption": st["num_swap_outs"],
                "prefix_cache_hit_rate": st["prefix_cache_hit_rate"],
                "avg_sequence_length": st["num_context_tokens"] / st["num_seqs"] if st["num_seqs"] else 0.0}
