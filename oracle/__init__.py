"""CPU fp64 oracle for the paged-attention path (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The product library never does, and this
package imports nothing from the product package.

The arithmetic lives in ``pa_oracle.c`` (plain C, fp64, compiled with gcc,
``-ffp-contract=off``); this module only marshals numpy/torch arrays into it.
Inputs are converted exactly to float64 from their stored dtype.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(the pages' worked figures, closed forms, library routines on special cases,
invariants, and brute force on tiny inputs).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_HDR = os.path.join(_HERE, "pa_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libpa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH) or
             max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)) > os.path.getmtime(_LIB_PATH))
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build())
            P, I, L, D = C.c_void_p, C.c_int, C.c_int64, C.c_double
            sig = {
                "orc_kv_bytes_per_token": (L, [I, I, I, I]),
                "orc_blocks_for_tokens": (L, [L, I]),
                "orc_pool_blocks": (L, [L, I, L]),
                "orc_alloc_create": (P, [I, P]),
                "orc_alloc_take": (I, [P, I, P]),
                "orc_alloc_share": (None, [P, P, I]),
                "orc_alloc_release": (None, [P, P, I]),
                "orc_alloc_num_free": (I, [P]),
                "orc_alloc_refcount": (I, [P, I]),
                "orc_alloc_destroy": (None, [P]),
                "orc_build_tables": (I, [P, I, P, P, I, I, I, P]),
                "orc_slot_mapping": (None, [P, I, I, P, P, I, P]),
                "orc_cache_write": (None, [P, P, P, P, P, I, I, I, I, I, I]),
                "orc_gather": (None, [P, P, I, I, I, I, I, P]),
                "orc_cache_write_vt": (None, [P, P, P, I, I, I, I, I, I, I]),
                "orc_copy_blocks": (None, [P, P, P, P, P, I, L]),
                "orc_fp8_e4m3_encode": (C.c_uint8, [C.c_float]),
                "orc_fp8_e4m3_decode": (D, [C.c_uint8]),
                "orc_quantize_fp8": (None, [P, L, C.c_float, P]),
                "orc_dequantize_fp8": (None, [P, L, D, P]),
                "orc_decode": (None, [P, P, P, P, P, P, I, I, I, I, D, I]),
                "orc_prefill": (None, [P, P, P, P, P, P, P, P, I, I, I, I, D, I]),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype, f.argtypes = res, args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def _f64(t) -> np.ndarray:
    """Exact conversion of a stored tensor/array to float64."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return np.ascontiguousarray(t.detach().cpu().to(torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(t, dtype=np.float64))


def _bytes(t) -> np.ndarray:
    """Raw bytes of a stored tensor (any dtype) as a uint8 array."""
    import torch
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        return t.view(torch.uint8).numpy().reshape(-1).copy()
    return np.ascontiguousarray(np.asarray(t)).view(np.uint8).reshape(-1).copy()


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


# ----------------------------------------------------------------- sizes

def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    return int(_load().orc_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, elem_bytes))


def blocks_for_tokens(tokens: int, block_size: int) -> int:
    return int(_load().orc_blocks_for_tokens(tokens, block_size))


def pool_blocks(pool_bytes: int, block_size: int, bytes_per_token: int) -> int:
    return int(_load().orc_pool_blocks(int(pool_bytes), block_size, bytes_per_token))


# ------------------------------------------------------------- allocator

class Allocator:
    """FIFO free-block queue with reference counts."""

    def __init__(self, num_blocks: int, initial_order=None):
        self._lib = _load()
        self._order = None if initial_order is None else _c(initial_order, np.int32)
        self._h = self._lib.orc_alloc_create(num_blocks,
                                             None if self._order is None else _ptr(self._order))

    def take(self, n: int) -> np.ndarray | None:
        out = np.empty(max(n, 1), np.int32)
        if self._lib.orc_alloc_take(self._h, n, _ptr(out)) != 0:
            return None
        return out[:n]

    def share(self, ids):
        ids = _c(ids, np.int32)
        self._lib.orc_alloc_share(self._h, _ptr(ids), len(ids))

    def release(self, ids):
        ids = _c(ids, np.int32)
        self._lib.orc_alloc_release(self._h, _ptr(ids), len(ids))

    def num_free(self) -> int:
        return int(self._lib.orc_alloc_num_free(self._h))

    def refcount(self, block_id: int) -> int:
        return int(self._lib.orc_alloc_refcount(self._h, block_id))

    def build_tables(self, lens, max_blocks: int, block_size: int, sharer=None,
                     prefix_tokens: int = 0) -> np.ndarray:
        lens = _c(lens, np.int32)
        B = len(lens)
        sh = None if sharer is None else _c(sharer, np.uint8)
        tables = np.empty((B, max_blocks), np.int32)
        rc = self._lib.orc_build_tables(self._h, B, _ptr(lens), None if sh is None else _ptr(sh),
                                        prefix_tokens, block_size, max_blocks, _ptr(tables))
        if rc != 0:
            raise RuntimeError("oracle allocator: pool exhausted or table too small")
        return tables

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.orc_alloc_destroy(h)


def slot_mapping(tables, block_size: int, seq, pos) -> np.ndarray:
    tables = _c(tables, np.int32)
    seq, pos = _c(seq, np.int32), _c(pos, np.int32)
    out = np.empty(len(seq), np.int64)
    _load().orc_slot_mapping(_ptr(tables), tables.shape[1], block_size, _ptr(seq), _ptr(pos),
                             len(seq), _ptr(out))
    return out


# ------------------------------------------------------ cache write, gather

def cache_write(k_cache, v_cache, k, v, slots, block_size: int):
    """Returns new (k_cache, v_cache) byte arrays after writing rows of k, v.

    k_cache, v_cache: tensors [NB][n_kv][bs][d]; k, v: tensors [T][n_kv][d]."""
    NB, n_kv, bs, d = k_cache.shape
    assert bs == block_size
    eb = k_cache.element_size()
    kc, vc = _bytes(k_cache), _bytes(v_cache)
    kb, vb = _bytes(k), _bytes(v)
    slots = _c(slots, np.int64)
    _load().orc_cache_write(_ptr(kc), _ptr(vc), _ptr(kb), _ptr(vb), _ptr(slots), len(slots),
                            NB, n_kv, bs, d, eb)
    return kc, vc


def cache_write_vt(v_cache, v, slots, block_size: int):
    """Returns the new byte array of a V pool stored transposed per piece of
    P tokens of each (block, head), [NB][n_kv][bs / P][d][P] (the shape of
    v_cache gives P), after writing rows of v [T][n_kv][d]."""
    NB, n_kv, n_pieces, d, piece = v_cache.shape
    assert n_pieces * piece == block_size
    eb = v_cache.element_size()
    vc, vb = _bytes(v_cache), _bytes(v)
    slots = _c(slots, np.int64)
    _load().orc_cache_write_vt(_ptr(vc), _ptr(vb), _ptr(slots), len(slots), NB, n_kv, block_size,
                               d, eb, piece)
    return vc


def copy_blocks(src_k, src_v, dst_k, dst_v, mapping):
    """Returns new (dst_k, dst_v) byte arrays: whole blocks mapping[i][0] of
    the source pools copied over blocks mapping[i][1] of the destination."""
    NB, n_kv, bs, d = src_k.shape
    bb = n_kv * bs * d * src_k.element_size()
    sk, sv = _bytes(src_k), _bytes(src_v)
    dk, dv = _bytes(dst_k), _bytes(dst_v)
    m = _c(mapping, np.int32).reshape(-1, 2)
    _load().orc_copy_blocks(_ptr(sk), _ptr(sv), _ptr(dk), _ptr(dv), _ptr(m), len(m), bb)
    return dk, dv


def gather(cache, table, L: int) -> np.ndarray:
    """Contiguous [L][n_kv][d] bytes of one sequence read through its table."""
    NB, n_kv, bs, d = cache.shape
    eb = cache.element_size()
    cb = _bytes(cache)
    table = _c(table, np.int32)
    out = np.empty(L * n_kv * d * eb, np.uint8)
    _load().orc_gather(_ptr(cb), _ptr(table), L, n_kv, bs, d, eb, _ptr(out))
    return out


# ---------------------------------------------------------------- fp8 e4m3

def fp8_encode(x: float) -> int:
    return int(_load().orc_fp8_e4m3_encode(float(x)))


def fp8_decode(code: int) -> float:
    return float(_load().orc_fp8_e4m3_decode(int(code)))


def quantize_fp8(x, scale: float) -> np.ndarray:
    """uint8 codes of encode(fp32(x) / fp32(scale)), same shape as x."""
    import torch
    xf = x.detach().cpu().to(torch.float32).numpy() if isinstance(x, torch.Tensor) else np.asarray(x, np.float32)
    xf = np.ascontiguousarray(xf, np.float32)
    out = np.empty(xf.shape, np.uint8)
    _load().orc_quantize_fp8(_ptr(xf), xf.size, float(scale), _ptr(out))
    return out


def dequantize_fp8(codes, scale: float) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes), np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().orc_dequantize_fp8(_ptr(c), c.size, float(np.float32(scale)), _ptr(out))
    return out


# ---------------------------------------------------------------- attention

def _pack(seqs):
    lens = np.array([s.shape[0] for s in seqs], np.int32)
    start = np.zeros(len(seqs), np.int64)
    if len(seqs) > 1:
        start[1:] = np.cumsum(lens[:-1])
    return np.concatenate([_f64(s) for s in seqs]) if len(seqs) else np.zeros((0,)), start, lens


def decode(q, ks, vs, scale: float, threads: int | None = None) -> np.ndarray:
    """out[s][h] = softmax(scale q K_s^T) V_s; ks/vs: per-sequence [L][n_kv][d]."""
    qd = _f64(q)
    B, n_q, d = qd.shape
    K, start, lens = _pack(ks)
    V, _, _ = _pack(vs)
    n_kv = ks[0].shape[1]
    out = np.zeros((B, n_q, d), np.float64)
    _load().orc_decode(_ptr(out), _ptr(qd), _ptr(K), _ptr(V), _ptr(start), _ptr(lens),
                       B, n_q, n_kv, d, float(scale), threads or default_threads())
    return out


def prefill(qs, ks, vs, scale: float, threads: int | None = None) -> list[np.ndarray]:
    """Chunked prefill: qs[r] is [C_r][n_q][d], ks/vs[r] are [L_r][n_kv][d]
    (all tokens of request r, chunk included); row i of the chunk is at
    position L_r - C_r + i.  Returns per-request [C_r][n_q][d]."""
    Q, q_start, chunk = _pack(qs)
    K, kv_start, lens = _pack(ks)
    V, _, _ = _pack(vs)
    R = len(qs)
    n_q, d = qs[0].shape[1], qs[0].shape[2]
    n_kv = ks[0].shape[1]
    out = np.zeros(Q.shape, np.float64)
    _load().orc_prefill(_ptr(out), _ptr(Q), _ptr(q_start), _ptr(chunk), _ptr(K), _ptr(V),
                        _ptr(kv_start), _ptr(lens), R, n_q, n_kv, d, float(scale),
                        threads or default_threads())
    return [out[q_start[r]:q_start[r] + chunk[r]] for r in range(R)]
