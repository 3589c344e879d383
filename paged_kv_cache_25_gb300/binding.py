"""Thin ctypes binding over libpa.so, with the C ABI's names.

Argument marshalling only: tensors become pointers and shapes, and a non-OK
status becomes a PAError.  Every step of the path runs in the library's CUDA
kernels; there is no Python or CPU fallback, and importing this module on a
machine where libpa.so has not been built raises at first use.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import numpy as np
import torch

from . import build as _build

__all__ = [
    "PAError", "lib", "pa_reshape_and_cache", "pa_reshape_and_cache_quant", "pa_decode",
    "pa_decode_workspace_size", "pa_decode_verify", "pa_decode_verify_workspace_size",
    "pa_decode_no_alloc", "PA_DECODE_NO_ALLOC_SCRATCH_BYTES",
    "pa_prefill_chunk", "pa_prefill_workspace_size", "pa_get_device_error", "pa_status_string",
    "pa_set_profile_events", "pa_copy_blocks", "pa_swap_blocks", "Allocator", "PrefixCache", "pa_prefix_block_hash", "pa_slot_mapping", "pa_kv_bytes_per_token",
    "pa_pool_blocks", "EXPORTED", "dtype_code",
]

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_OUT_OF_RANGE = 0, 1, 2, 3
PA_ERR_WORKSPACE, PA_ERR_TIMEOUT, PA_ERR_CUDA = 4, 5, 6
_DT = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2, torch.float8_e4m3fn: 3}
PA_F32, PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2, 3


class _Desc(C.Structure):
    _fields_ = [("num_blocks", C.c_int), ("block_size", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("dtype", C.c_int), ("k_scale", C.c_float),
                ("v_scale", C.c_float), ("act_dtype", C.c_int)]


P, I, L, F, SZ, U8P = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_size_t, C.c_void_p
_SIGS = {
    "pa_reshape_and_cache": (I, [P, P, P, P, P, I, C.POINTER(_Desc), P]),
    "pa_decode": (I, [P, I, P, P, P, C.POINTER(_Desc), P, I, P, I, I, F, I, P, SZ, P]),
    "pa_decode_workspace_size": (SZ, [I, I, I, I, I, I]),
    "pa_decode_no_alloc": (I, [P, I, P, P, P, C.POINTER(_Desc), P, I, P, I, I, F, I, P]),
    "pa_decode_verify": (I, [P, I, P, P, P, C.POINTER(_Desc), P, I, P, I, I, I, F, I, P, SZ, P]),
    "pa_decode_verify_workspace_size": (SZ, [I, I, I, I, I, I, I]),
    "pa_reshape_and_cache_quant": (I, [P, P, I, P, P, P, I, C.POINTER(_Desc), P]),
    "pa_prefill_chunk": (I, [P, I, P, P, P, C.POINTER(_Desc), P, I, P, P, I, I, I, F, I, P, SZ, P]),
    "pa_prefill_workspace_size": (SZ, [I, I, I, I]),
    "pa_copy_blocks": (I, [P, P, C.POINTER(_Desc), P, I, P]),
    "pa_swap_blocks": (I, [P, P, I, P, P, I, C.POINTER(_Desc), P, I, P]),
    "pa_get_device_error": (I, [P]),
    "pa_selftest_bounded_wait": (I, [C.c_uint, P, P]),
    "pa_status_string": (C.c_char_p, [I]),
    "pa_last_error_message": (C.c_char_p, []),
    "pa_set_profile_events": (None, [P, P]),
    "pa_alloc_create": (P, [I, P]),
    "pa_alloc_blocks": (I, [P, I, P]),
    "pa_alloc_share": (None, [P, P, I]),
    "pa_alloc_free": (None, [P, P, I]),
    "pa_alloc_num_free": (I, [P]),
    "pa_alloc_refcount": (I, [P, I]),
    "pa_alloc_destroy": (None, [P]),
    "pa_alloc_build_tables": (I, [P, I, P, P, I, I, I, P]),
    "pa_slot_mapping": (I, [P, I, I, P, P, I, P]),
    "pa_prefix_create": (P, [I, I, P]),
    "pa_prefix_destroy": (None, [P]),
    "pa_prefix_block_hash": (C.c_uint64, [C.c_uint64, P, I]),
    "pa_prefix_lookup": (I, [P, P, I]),
    "pa_prefix_acquire": (I, [P, P, I, P, I]),
    "pa_prefix_alloc": (I, [P, I, P]),
    "pa_prefix_commit": (I, [P, P, I, P]),
    "pa_prefix_release": (I, [P, P, I]),
    "pa_prefix_num_free": (I, [P]),
    "pa_prefix_num_evictable": (I, [P]),
    "pa_prefix_num_cached": (I, [P]),
    "pa_prefix_refcount": (I, [P, I]),
    "pa_kv_bytes_per_token": (L, [I, I, I, I]),
    "pa_pool_blocks": (L, [L, I, L]),
}
EXPORTED = tuple(_SIGS)

_lock = threading.Lock()
_lib = None


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(what)


def lib(path: str | None = None):
    """Loads libpa.so (built in-tree by build.build()); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"libpa.so not found at {p}: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            h = C.CDLL(p)
            for name, (res, args) in _SIGS.items():
                f = getattr(h, name)
                f.restype, f.argtypes = res, args
            _lib = h
    return _lib


def dtype_code(dt: torch.dtype) -> int:
    if dt not in _DT:
        raise TypeError(f"unsupported dtype {dt}")
    return _DT[dt]


def _check(st: int, what: str):
    if st != PA_OK:
        msg = lib().pa_last_error_message().decode()
        name = lib().pa_status_string(st).decode()
        raise PAError(st, f"{what}: {name}: {msg}")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr() if t.numel() else None
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    raise TypeError(type(t))


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return stream


def _desc(k_cache: torch.Tensor, k_scale=None, v_scale=None, act_dtype=None) -> _Desc:
    """Cache descriptor; FP8 pools (torch.float8_e4m3fn) need the two scales and
    the activation dtype (of q and of the rows written into the pool)."""
    nb, n_kv, bs, d = k_cache.shape
    dt = dtype_code(k_cache.dtype)
    if dt == PA_FP8_E4M3:   # missing scales reach the library as 0 and are refused there
        return _Desc(nb, bs, n_kv, d, dt, float(k_scale or 0.0), float(v_scale or 0.0),
                     dtype_code(act_dtype) if act_dtype is not None else -1)
    return _Desc(nb, bs, n_kv, d, dt, 1.0, 1.0, dt)


def pa_status_string(st: int) -> str:
    return lib().pa_status_string(st).decode()


def pa_reshape_and_cache(k, v, k_cache, v_cache, slot_mapping, stream=None, k_scale=None,
                         v_scale=None):
    """k, v [T][n_kv][d] -> pools [NB][n_kv][bs][d] at slot_mapping (int64 [T]).
    FP8 pools take rows of E4M3 codes (copied as they are) and their scales."""
    assert k.is_contiguous() and v.is_contiguous() and slot_mapping.dtype == torch.int64
    d = _desc(k_cache, k_scale, v_scale)
    _check(lib().pa_reshape_and_cache(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache),
                                      _ptr(slot_mapping), int(k.shape[0]), C.byref(d),
                                      _stream(stream)), "pa_reshape_and_cache")


def pa_decode_workspace_size(num_seqs, n_q_heads, n_kv_heads, head_dim, block_size,
                             max_context_len) -> int:
    return int(lib().pa_decode_workspace_size(num_seqs, n_q_heads, n_kv_heads, head_dim,
                                              block_size, max_context_len))


def pa_decode_verify_workspace_size(num_seqs, q_per_seq, n_q_heads, n_kv_heads, head_dim,
                                    block_size, max_context_len) -> int:
    return int(lib().pa_decode_verify_workspace_size(num_seqs, q_per_seq, n_q_heads, n_kv_heads,
                                                     head_dim, block_size, max_context_len))


def pa_decode_verify(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                     block_size: int, workspace=None, stream=None, k_scale=None, v_scale=None):
    """out, q [B][q_per_seq][n_q][d]: query i of sequence s sits at position
    context_lens[s] - q_per_seq + i and sees keys up to it."""
    B, nq, n_q, _ = q.shape
    d = _desc(k_cache, k_scale, v_scale, q.dtype)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_decode_verify(_ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache),
                                  _ptr(v_cache), C.byref(d), _ptr(block_tables),
                                  int(block_tables.shape[1]), _ptr(context_lens), int(B), int(nq),
                                  int(n_q), float(scale), int(block_size), _ptr(workspace),
                                  ws_bytes, _stream(stream)), "pa_decode_verify")


def pa_reshape_and_cache_quant(k, v, k_cache, v_cache, slot_mapping, k_scale=None, v_scale=None,
                               stream=None):
    """k, v [T][n_kv][d] (fp32/fp16/bf16) -> pools, quantized to E4M3 codes of
    x / scale when the pools are torch.float8_e4m3fn."""
    assert k.is_contiguous() and v.is_contiguous() and slot_mapping.dtype == torch.int64
    d = _desc(k_cache, k_scale, v_scale, k.dtype)
    _check(lib().pa_reshape_and_cache_quant(_ptr(k), _ptr(v), dtype_code(k.dtype), _ptr(k_cache),
                                            _ptr(v_cache), _ptr(slot_mapping), int(k.shape[0]),
                                            C.byref(d), _stream(stream)),
           "pa_reshape_and_cache_quant")


def pa_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
              block_size: int, workspace=None, stream=None, k_scale=None, v_scale=None):
    """out [B][n_q][d] (fp32/fp16/bf16) = paged decode attention of q [B][n_q][d].
    FP8 pools also take k_scale and v_scale."""
    B, n_q, _ = q.shape
    d = _desc(k_cache, k_scale, v_scale, q.dtype)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_decode(_ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache),
                           _ptr(v_cache), C.byref(d), _ptr(block_tables),
                           int(block_tables.shape[1]), _ptr(context_lens), int(B), int(n_q),
                           float(scale), int(block_size), _ptr(workspace), ws_bytes,
                           _stream(stream)), "pa_decode")


def pa_decode_no_alloc(out, q, k_cache, v_cache, block_tables, context_lens, scale: float,
                       block_size: int, stream=None):
    """pa_decode with the library's fixed internal scratch: the caller passes
    only inputs and outputs and nothing is allocated.  Batches that need more
    than PA_DECODE_NO_ALLOC_SCRATCH_BYTES of scratch raise PAError."""
    B, n_q, _ = q.shape
    d = _desc(k_cache)
    _check(lib().pa_decode_no_alloc(_ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache),
                                    _ptr(v_cache), C.byref(d), _ptr(block_tables),
                                    int(block_tables.shape[1]), _ptr(context_lens), int(B),
                                    int(n_q), float(scale), int(block_size), _stream(stream)),
           "pa_decode_no_alloc")


PA_DECODE_NO_ALLOC_SCRATCH_BYTES = 16 << 20


def pa_prefill_workspace_size(num_reqs, n_q_heads, head_dim, total_q) -> int:
    return int(lib().pa_prefill_workspace_size(num_reqs, n_q_heads, head_dim, total_q))


def pa_prefill_chunk(out, q, k_cache, v_cache, block_tables, query_start_loc, context_lens,
                     max_query_len: int, scale: float, block_size: int, workspace=None,
                     stream=None, k_scale=None, v_scale=None):
    """Chunked prefill: out/q [sum C][n_q][d]; query_start_loc int32 [R+1].
    FP8 pools also take k_scale and v_scale."""
    R = int(context_lens.shape[0])
    n_q = int(q.shape[1])
    d = _desc(k_cache, k_scale, v_scale, q.dtype)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().pa_prefill_chunk(_ptr(out), dtype_code(out.dtype), _ptr(q), _ptr(k_cache),
                                  _ptr(v_cache), C.byref(d), _ptr(block_tables),
                                  int(block_tables.shape[1]), _ptr(query_start_loc),
                                  _ptr(context_lens), R, int(max_query_len), n_q, float(scale),
                                  int(block_size), _ptr(workspace), ws_bytes, _stream(stream)),
           "pa_prefill_chunk")


def pa_copy_blocks(k_cache, v_cache, block_mapping, stream=None):
    """Copy whole blocks mapping[i][0] -> mapping[i][1] within the pools."""
    d = _desc(k_cache)
    _check(lib().pa_copy_blocks(_ptr(k_cache), _ptr(v_cache), C.byref(d), _ptr(block_mapping),
                                int(block_mapping.shape[0]), _stream(stream)), "pa_copy_blocks")


def pa_swap_blocks(src_k, src_v, dst_k, dst_v, block_mapping, stream=None):
    """Copy whole blocks between two pools of one layout; either side may be a
    pinned host tensor (torch pin_memory) or a device tensor."""
    d = _desc(src_k)
    _check(lib().pa_swap_blocks(_ptr(src_k), _ptr(src_v), int(src_k.shape[0]), _ptr(dst_k),
                                _ptr(dst_v), int(dst_k.shape[0]), C.byref(d), _ptr(block_mapping),
                                int(block_mapping.shape[0]), _stream(stream)), "pa_swap_blocks")


def pa_get_device_error(stream=None) -> int:
    """Synchronizes the stream, returns and clears the device error word."""
    return int(lib().pa_get_device_error(_stream(stream)))


def pa_selftest_bounded_wait(limit_us: int, scratch, stream=None):
    """Run the bounded-wait self-test (a wait nothing completes) on `stream`."""
    _check(lib().pa_selftest_bounded_wait(int(limit_us), _ptr(scratch), _stream(stream)),
           "pa_selftest_bounded_wait")


def pa_set_profile_events(start=None, stop=None):
    """Record torch.cuda.Event pair around pa_decode's main kernel (None: off)."""
    s = start.cuda_event if start is not None else None
    e = stop.cuda_event if stop is not None else None
    lib().pa_set_profile_events(s, e)


# ------------------------------------------------------------------ host allocator

class Allocator:
    """The library's FIFO free-block queue with reference counts (host memory)."""

    def __init__(self, num_blocks: int, initial_order=None):
        self._l = lib()
        order = None if initial_order is None else np.ascontiguousarray(initial_order, np.int32)
        self._h = self._l.pa_alloc_create(num_blocks, _ptr(order))
        if not self._h:
            raise PAError(PA_ERR_INVALID_ARG, "pa_alloc_create: bad size or order")

    def blocks(self, n: int):
        out = np.empty(max(n, 1), np.int32)
        return out[:n] if self._l.pa_alloc_blocks(self._h, n, _ptr(out)) == 0 else None

    def share(self, ids):
        ids = np.ascontiguousarray(ids, np.int32)
        self._l.pa_alloc_share(self._h, _ptr(ids), len(ids))

    def free(self, ids):
        ids = np.ascontiguousarray(ids, np.int32)
        self._l.pa_alloc_free(self._h, _ptr(ids), len(ids))

    def num_free(self) -> int:
        return int(self._l.pa_alloc_num_free(self._h))

    def refcount(self, block_id: int) -> int:
        return int(self._l.pa_alloc_refcount(self._h, block_id))

    def build_tables(self, lens, max_blocks: int, block_size: int, sharer=None,
                     prefix_tokens: int = 0) -> np.ndarray:
        lens = np.ascontiguousarray(lens, np.int32)
        sh = None if sharer is None else np.ascontiguousarray(sharer, np.uint8)
        tables = np.empty((len(lens), max_blocks), np.int32)
        st = self._l.pa_alloc_build_tables(self._h, len(lens), _ptr(lens), _ptr(sh),
                                           prefix_tokens, block_size, max_blocks, _ptr(tables))
        _check(st, "pa_alloc_build_tables")
        return tables

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._l.pa_alloc_destroy(h)


class PrefixCache:
    """The library's host prefix cache: fingerprinted full blocks reused across
    requests, unused cached blocks evicted least recently released first."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self._l = lib()
        order = None if free_order is None else np.ascontiguousarray(free_order, np.int32)
        self._h = self._l.pa_prefix_create(num_blocks, block_size, _ptr(order))
        if not self._h:
            raise PAError(PA_ERR_INVALID_ARG, "pa_prefix_create: bad size or order")
        self.block_size = block_size

    @staticmethod
    def _toks(tokens):
        return np.ascontiguousarray(tokens, np.int32)

    def lookup(self, tokens) -> int:
        t = self._toks(tokens)
        return int(self._l.pa_prefix_lookup(self._h, _ptr(t), len(t)))

    def acquire(self, tokens, table_len: int):
        """(hit blocks, table) or None when the pool cannot supply the rest."""
        t = self._toks(tokens)
        table = np.empty(max(table_len, 1), np.int32)
        r = self._l.pa_prefix_acquire(self._h, _ptr(t), len(t), _ptr(table), table_len)
        if r == -2:
            raise PAError(PA_ERR_INVALID_ARG, "pa_prefix_acquire: bad arguments")
        return None if r < 0 else (int(r), table[:table_len])

    def alloc(self, n: int):
        out = np.empty(max(n, 1), np.int32)
        r = self._l.pa_prefix_alloc(self._h, n, _ptr(out))
        if r == -2:
            raise PAError(PA_ERR_INVALID_ARG, "pa_prefix_alloc: bad arguments")
        return None if r < 0 else out[:n]

    def commit(self, tokens, table) -> int:
        t = self._toks(tokens)
        tb = np.ascontiguousarray(table, np.int32)
        r = self._l.pa_prefix_commit(self._h, _ptr(t), len(t), _ptr(tb))
        if r < 0:
            raise PAError(PA_ERR_INVALID_ARG, "pa_prefix_commit: bad table")
        return int(r)

    def release(self, table):
        tb = np.ascontiguousarray(table, np.int32)
        if self._l.pa_prefix_release(self._h, _ptr(tb), len(tb)) != 0:
            raise PAError(PA_ERR_INVALID_ARG, "pa_prefix_release: bad ids or counts")

    def num_free(self) -> int:
        return int(self._l.pa_prefix_num_free(self._h))

    def num_evictable(self) -> int:
        return int(self._l.pa_prefix_num_evictable(self._h))

    def num_cached(self) -> int:
        return int(self._l.pa_prefix_num_cached(self._h))

    def refcount(self, block_id: int) -> int:
        return int(self._l.pa_prefix_refcount(self._h, block_id))

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._l.pa_prefix_destroy(h)


def pa_prefix_block_hash(parent: int, tokens) -> int:
    t = np.ascontiguousarray(tokens, np.int32)
    return int(lib().pa_prefix_block_hash(parent, _ptr(t), len(t)))


def pa_slot_mapping(tables, block_size: int, seq, pos) -> np.ndarray:
    tables = np.ascontiguousarray(tables, np.int32)
    seq = np.ascontiguousarray(seq, np.int32)
    pos = np.ascontiguousarray(pos, np.int32)
    out = np.empty(max(len(seq), 1), np.int64)
    _check(lib().pa_slot_mapping(_ptr(tables), tables.shape[1], block_size, _ptr(seq), _ptr(pos),
                                 len(seq), _ptr(out)), "pa_slot_mapping")
    return out[:len(seq)]


def pa_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, elem_bytes) -> int:
    return int(lib().pa_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, elem_bytes))


def pa_pool_blocks(pool_bytes, block_size, bytes_per_token) -> int:
    return int(lib().pa_pool_blocks(int(pool_bytes), block_size, bytes_per_token))
