"""Device state and one step of the paged-attention hot path for a workload.

Setting up (off the timed path): the library's host allocator hands out
physical blocks from a seeded free-queue order and builds every sequence's
block table; the pools are filled with NaN so that any read of a slot the
method must not read shows up; every cached context row is appended through
pa_reshape_and_cache exactly as a serving loop would have appended it.

One step (the timed hot path): append the new tokens' K/V
(pa_reshape_and_cache), decode one token for every decode sequence
(pa_decode, split-K plus reduce; pa_decode_verify when a sequence brings
several query rows), and run the chunked-prefill requests, if any
(pa_prefill_chunk).  All of it runs in the library's CUDA kernels.
"""
from __future__ import annotations

import collections
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

from . import binding as pa
from .inputs import Draws, Workload


def _ceil_div(a, b):
    return -(-a // b)


def _draw_threads() -> int:
    return max(1, min(16, len(os.sched_getaffinity(0))))


def _ordered_window(ex, fn, items, window):
    """fn(item) for every item, in order, at most `window` results ahead."""
    items = list(items)
    pending = collections.deque()
    for i, it in enumerate(items):
        pending.append(ex.submit(fn, it))
        if len(pending) > window:
            yield pending.popleft().result()
    while pending:
        yield pending.popleft().result()


class PagedStep:
    def __init__(self, wl: Workload, seed: int | None = None, device="cuda",
                 out_dtype: torch.dtype | None = None, upload_chunk_tokens: int = 1 << 18,
                 prefill_out_dtype: torch.dtype | None = None):
        self.wl = wl
        self.draws = dr = Draws(wl, seed)
        self.device = torch.device(device)
        bs, n_kv, d = wl.block_size, wl.n_kv_heads, wl.head_dim
        self.lens = dr.decode_lens()
        self.sharers = dr.sharers()
        self.prefix = wl.shared_prefix_tokens if self.sharers.any() else 0
        self.p_ctx = dr.prefill_ctx()
        self.p_chunk = dr.prefill_chunks()
        self.p_lens = (self.p_ctx + self.p_chunk).astype(np.int32)
        self.R = len(self.p_lens)

        # ---- pool size and block tables (library allocator) ----------------
        per_tok = pa.pa_kv_bytes_per_token(1, n_kv, d, wl.pool_elem_bytes)
        self.fp8 = wl.pool_dtype == torch.float8_e4m3fn
        self.kv_scales = dict(k_scale=wl.kv_scale, v_scale=wl.kv_scale) if self.fp8 else {}
        need = int(sum(_ceil_div(int(L), bs) for L in self.lens))
        if self.prefix:
            need -= (int(self.sharers.sum()) - 1) * (self.prefix // bs)
        need += int(sum(_ceil_div(int(L), bs) for L in self.p_lens))
        if wl.pool == "fixed":
            nb = int(wl.pool_arg)
        elif wl.pool == "scale":
            nb = int(math.ceil(wl.pool_arg * need))
        else:
            nb = pa.pa_pool_blocks(int(wl.pool_arg), bs, per_tok)
        self.num_blocks = nb
        all_lens = np.concatenate([self.lens, self.p_lens]) if self.R else self.lens
        self.max_blocks = _ceil_div(int(all_lens.max()), bs)
        self.alloc = pa.Allocator(nb, dr.free_order(nb))
        self.tables = self.alloc.build_tables(self.lens, self.max_blocks, bs, self.sharers,
                                              self.prefix)
        self.p_tables = (self.alloc.build_tables(self.p_lens, self.max_blocks, bs)
                         if self.R else np.zeros((0, self.max_blocks), np.int32))

        dev = self.device
        # unwritten slots hold NaN (E4M3 NaN code 0x7F for FP8 pools)
        if self.fp8:
            self.k_cache = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8,
                                      device=dev).view(torch.float8_e4m3fn)
            # FP8 V codes are stored transposed per 16-token piece of a
            # (block, head): [block_size / 16][d][16]
            self.v_cache = torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8,
                                      device=dev).view(torch.float8_e4m3fn)
        else:
            self.k_cache = torch.full((nb, n_kv, bs, d), float("nan"), dtype=wl.dtype, device=dev)
            self.v_cache = torch.full((nb, n_kv, bs, d), float("nan"), dtype=wl.dtype, device=dev)

        # ---- pre-fill the cached context through the cache-write kernel ------
        self._prefill_context(upload_chunk_tokens)

        # ---- per-step inputs ------------------------------------------------
        B, nq = wl.batch, wl.q_per_seq
        self.q = dr.q().to(dev)
        # the newest row(s) of every decode sequence, kept aside by the pre-fill
        new_k = torch.cat([k for k, _ in self._newest])
        new_v = torch.cat([v for _, v in self._newest])
        del self._newest
        seq = np.repeat(np.arange(B, dtype=np.int32), nq)
        pos = (self.lens[:, None] - nq + np.arange(nq)[None, :]).reshape(-1).astype(np.int32)
        slots = pa.pa_slot_mapping(self.tables, bs, seq, pos)
        ks, vs, ss = [new_k], [new_v], [slots]
        self.p_q = []
        for r in range(self.R):
            k, v = dr.prefill_kv(r, int(self.p_lens[r]))
            c0 = int(self.p_ctx[r])
            ks.append(k[c0:]); vs.append(v[c0:])
            ss.append(pa.pa_slot_mapping(self.p_tables, bs, np.full(len(k) - c0, r, np.int32),
                                         np.arange(c0, len(k), dtype=np.int32)))
            self.p_q.append(dr.prefill_q(r))
        self.new_k = torch.cat(ks).to(dev).contiguous()
        self.new_v = torch.cat(vs).to(dev).contiguous()
        self.new_slots = torch.from_numpy(np.concatenate(ss)).to(dev)
        self.block_tables = torch.from_numpy(self.tables).to(dev)
        self.context_lens = torch.from_numpy(self.lens.astype(np.int32)).to(dev)
        od = out_dtype or wl.dtype
        self.out = torch.empty(tuple(self.q.shape), dtype=od, device=dev)
        ws = pa.pa_decode_verify_workspace_size(B, nq, wl.n_q_heads, n_kv, d, bs,
                                                self.max_blocks * bs)
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev) if ws else None
        if self.R:
            self.p_q_dev = torch.cat(self.p_q).to(dev).contiguous()
            qsl = np.zeros(self.R + 1, np.int32)
            qsl[1:] = np.cumsum(self.p_chunk)
            self.query_start_loc = torch.from_numpy(qsl).to(dev)
            self.p_block_tables = torch.from_numpy(self.p_tables).to(dev)
            self.p_context_lens = torch.from_numpy(self.p_lens).to(dev)
            self.p_out = torch.empty((int(qsl[-1]), wl.n_q_heads, d),
                                     dtype=prefill_out_dtype or od, device=dev)

    # ------------------------------------------------------------------
    def _prefill_context(self, chunk_tokens: int):
        """Appends every cached row (all rows but the step's new ones)."""
        wl, dr, bs = self.wl, self.draws, self.wl.block_size
        prefix = dr.prefix_kv() if self.prefix else None
        pending_k, pending_v, pending_s, n = [], [], [], 0
        first_sharer_done = False
        self._newest = []

        def flush():
            nonlocal pending_k, pending_v, pending_s, n
            if not n:
                return
            k = torch.cat(pending_k).to(self.device, non_blocking=False).contiguous()
            v = torch.cat(pending_v).to(self.device, non_blocking=False).contiguous()
            s = torch.from_numpy(np.concatenate(pending_s)).to(self.device)
            self._write(k, v, s)
            torch.cuda.synchronize(self.device)
            pending_k, pending_v, pending_s, n = [], [], [], 0

        def add(k, v, table_set, row, p0, p1):
            nonlocal n
            if p1 <= p0:
                return
            pending_k.append(k[p0:p1]); pending_v.append(v[p0:p1])
            pending_s.append(pa.pa_slot_mapping(table_set, bs, np.full(p1 - p0, row, np.int32),
                                                np.arange(p0, p1, dtype=np.int32)))
            n += p1 - p0
            if n >= chunk_tokens:
                flush()

        # the draws are keyed per sequence, so worker threads produce them (numpy
        # and torch release the GIL while filling) in order, a window ahead
        draw = lambda s: dr.seq_kv(s, int(self.lens[s]), bool(self.sharers[s]), prefix)
        with ThreadPoolExecutor(_draw_threads()) as ex:
            for s, (k, v) in enumerate(_ordered_window(ex, draw, range(wl.batch), 32)):
                L = int(self.lens[s])
                start = 0
                if self.sharers[s]:
                    if first_sharer_done:
                        start = self.prefix       # the shared blocks are written once
                    first_sharer_done = True
                add(k, v, self.tables, s, start, L - wl.q_per_seq)
                self._newest.append((k[L - wl.q_per_seq:].clone(), v[L - wl.q_per_seq:].clone()))
            pdraw = lambda r: dr.prefill_kv(r, int(self.p_lens[r]))
            for r, (k, v) in enumerate(_ordered_window(ex, pdraw, range(self.R), 4)):
                add(k, v, self.p_tables, r, 0, int(self.p_ctx[r]))
        flush()

    def _write(self, k, v, slots, stream=None):
        if self.fp8:
            pa.pa_reshape_and_cache_quant(k, v, self.k_cache, self.v_cache, slots, stream=stream,
                                          **self.kv_scales)
        else:
            pa.pa_reshape_and_cache(k, v, self.k_cache, self.v_cache, slots, stream=stream)

    # ------------------------------------------------------------------
    # per-step inputs and outputs, replaceable by another set (see io_set)
    IO_NAMES = ("q", "new_k", "new_v", "new_slots", "block_tables", "context_lens", "out",
                "p_q_dev", "query_start_loc", "p_block_tables", "p_context_lens", "p_out")

    def io_set(self, clone: bool = False) -> dict:
        """The step's per-step device tensors by name (this object's own, or
        fresh copies of them, e.g. to double-buffer host uploads)."""
        io = {n: getattr(self, n) for n in self.IO_NAMES if hasattr(self, n)}
        return {n: t.clone() for n, t in io.items()} if clone else io

    def step(self, stream=None, prefill_events=None, io=None):
        """One pass of the hot path on `stream` (default: the current stream).
        prefill_events: optional (start, stop) torch.cuda.Event pair recorded
        around the chunked-prefill kernel.  io: per-step tensors to use instead
        of this object's own (same names and shapes as io_set()).

        With prefill requests the chunked prefill is launched first, on a side
        stream, and the decode after it on `stream`: the prefill grid's last
        wave leaves SMs idle, and the persistent decode's CTAs start on them
        while it drains.  Both wait for the cache write; `stream` waits for
        the prefill before the step ends."""
        wl = self.wl
        t = self.io_set() if io is None else io
        main = stream or torch.cuda.current_stream(self.device)
        self._write(t["new_k"], t["new_v"], t["new_slots"], stream=main)
        if self.R:
            side = self._side_stream()
            side.wait_stream(main)                    # after the cache write
            if prefill_events is not None:
                prefill_events[0].record(side)
            pa.pa_prefill_chunk(t["p_out"], t["p_q_dev"], self.k_cache, self.v_cache,
                                t["p_block_tables"], t["query_start_loc"], t["p_context_lens"],
                                int(self.p_chunk.max()), wl.scale, wl.block_size, stream=side,
                                **self.kv_scales)
            if prefill_events is not None:
                prefill_events[1].record(side)
        decode = pa.pa_decode if wl.q_per_seq == 1 else pa.pa_decode_verify
        decode(t["out"], t["q"], self.k_cache, self.v_cache, t["block_tables"],
               t["context_lens"], wl.scale, wl.block_size, self.workspace, stream=main,
               **self.kv_scales)
        if self.R:
            main.wait_stream(side)

    def _side_stream(self):
        if getattr(self, "_side", None) is None:
            self._side = torch.cuda.Stream(device=self.device)
        return self._side

    # ------------------------------------------------------------------ accounting
    def kv_bytes_unique(self) -> int:
        """K+V bytes the decode must read: valid rows of distinct physical blocks."""
        wl, bs = self.wl, self.wl.block_size
        row = 2 * wl.n_kv_heads * wl.head_dim * wl.pool_elem_bytes
        seen = {}
        for s, L in enumerate(self.lens):
            for i in range(_ceil_div(int(L), bs)):
                b = int(self.tables[s, i])
                seen[b] = max(seen.get(b, 0), min(bs, int(L) - i * bs))
        return sum(seen.values()) * row

    def kv_bytes_block_granular(self) -> int:
        """K+V bytes of whole blocks: every distinct physical block the decode
        touches counted with all block_size rows (masked tail rows included)."""
        wl, bs = self.wl, self.wl.block_size
        row = 2 * wl.n_kv_heads * wl.head_dim * wl.pool_elem_bytes
        blocks = set()
        for s, L in enumerate(self.lens):
            blocks.update(int(b) for b in self.tables[s, :_ceil_div(int(L), bs)])
        return len(blocks) * bs * row

    def kv_bytes_logical(self) -> int:
        wl = self.wl
        return int(self.lens.sum()) * 2 * wl.n_kv_heads * wl.head_dim * wl.pool_elem_bytes

    def prefill_flops(self) -> int:
        """2 matmuls x 2 flops per MAC over the causal (query, key) pairs."""
        wl = self.wl
        pairs = 0
        for r in range(self.R):
            c, ctx = int(self.p_chunk[r]), int(self.p_ctx[r])
            pairs += c * ctx + c * (c + 1) // 2
        return 4 * pairs * wl.n_q_heads * wl.head_dim
