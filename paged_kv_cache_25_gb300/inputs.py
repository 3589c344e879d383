"""Seeded synthetic workloads for the paged-attention path.

This module only draws random numbers and states workload sizes.  It holds
none of the method's arithmetic: no block arithmetic, no slot arithmetic and no
attention.  Both the CUDA path and the CPU oracle are fed from it, and neither
one's results ever flow back into it.

Every draw is keyed by ``(seed, tag, index)`` through numpy's SeedSequence, so a
single sequence's K/V can be regenerated on its own (the oracle only ever needs
a sample of the sequences at full size) and the draws for many sequences can be
produced in parallel threads with identical results.

Workloads (the KV shapes are single transformer layers):

* ``tiny-fp32``      4 sequences, context lengths {7, 16, 33, 50}, 4 query heads,
                     2 KV heads, head_dim 64, block_size 16, fp32, a pool of 32
                     physical blocks handed out in a seeded random order.
* ``tinyllama-bf16`` 64 sequences, lengths U[128, 2048], 32/4 heads, d 64,
                     bs 16, bf16, pool 1.5x the blocks needed.
* ``llama3-8b-bf16`` 256 sequences, lengths U[512, 4096], 32/8 heads, d 128,
                     bs 16, bf16, pool 1.5x the blocks needed.
* ``opt13b-fp16``    128 sequences, every length 2048, 40/40 heads, d 128, bs 16,
                     fp16, values N(0, 0.5) (standard deviation 0.5).
* ``llama3-8b-bf16-verify4``  the Llama-3-8B decode batch (same lengths and K/V)
                     where each sequence brings 4 query rows (3 drafted tokens to
                     verify plus one), the last 4 rows of its context.
* ``llama3-8b-fp8``  the Llama-3-8B decode batch (same draws) stored in an FP8
                     E4M3 pool with K and V scale 1/64.
* ``mixed-llama3-8b-bf16``  one continuous-batching step on Llama-3-8B shapes with
                     bs 32: 192 decode sequences with lengths lognormal(7, 1)
                     clipped to [16, 32768], a quarter of them sharing one
                     1024-token prefix (their length is 1024 plus the draw,
                     clipped), and 4 chunked-prefill requests, each a 512-token
                     chunk on top of U[1024, 8192] cached tokens; the pool is
                     sized to 60e9 bytes of K plus V.
* ``mixed-llama3-8b-fp8``  the same step (same draws) over an FP8 E4M3 pool with
                     K and V scale 1/64 (60e9 bytes hold twice the blocks).

Context lengths include the token being decoded: its K/V row is the last row of
the sequence's logical K/V and is appended by the cache write of the step.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np
import torch

__all__ = ["Workload", "WORKLOADS", "get", "Draws"]

_TAGS = {"lens": 1, "kv": 2, "q": 3, "order": 4, "share": 5, "prefix": 6,
         "pq": 7, "pkv": 8, "plens": 9, "newkv": 10, "toks": 11, "tokkv": 12}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int                 # decode sequences
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    std: float = 1.0
    lens_kind: str = "list"    # list | uniform | const | lognormal
    lens_args: tuple = ()
    pool: str = "scale"        # scale: factor x blocks needed; fixed: that many blocks; bytes: K+V bytes
    pool_arg: float = 1.5
    shared_prefix_tokens: int = 0
    shared_fraction: float = 0.0
    prefill_requests: int = 0
    prefill_chunk: int = 0
    prefill_ctx_range: tuple = (0, 0)
    cache_dtype: torch.dtype | None = None   # pool dtype when it differs (FP8 pools)
    kv_scale: float = 1.0                     # FP8 pools: per-tensor scale of K and V
    q_per_seq: int = 1                        # query rows per decode sequence (k+1 to verify k drafts)

    @property
    def pool_dtype(self) -> torch.dtype:
        return self.cache_dtype or self.dtype

    @property
    def pool_elem_bytes(self) -> int:
        return torch.empty((), dtype=self.pool_dtype).element_size()

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def elem_bytes(self) -> int:
        return torch.empty((), dtype=self.dtype).element_size()

    @property
    def scale(self) -> float:
        # the usual 1/sqrt(head_dim), as an fp32 value (the value the kernels receive)
        return float(np.float32(1.0 / np.sqrt(self.head_dim)))


WORKLOADS = {
    "tiny-fp32": Workload("tiny-fp32", 1001, 4, 4, 2, 64, 16, torch.float32,
                          lens_kind="list", lens_args=(7, 16, 33, 50),
                          pool="fixed", pool_arg=32),
    "tinyllama-bf16": Workload("tinyllama-bf16", 1002, 64, 32, 4, 64, 16, torch.bfloat16,
                               lens_kind="uniform", lens_args=(128, 2048)),
    "llama3-8b-bf16": Workload("llama3-8b-bf16", 1003, 256, 32, 8, 128, 16, torch.bfloat16,
                               lens_kind="uniform", lens_args=(512, 4096)),
    "opt13b-fp16": Workload("opt13b-fp16", 1004, 128, 40, 40, 128, 16, torch.float16, std=0.5,
                            lens_kind="const", lens_args=(2048,)),
    # the Llama-3-8B decode batch verifying 3 drafted tokens per sequence (4 query rows)
    "llama3-8b-bf16-verify4": Workload("llama3-8b-bf16-verify4", 1003, 256, 32, 8, 128, 16,
                                       torch.bfloat16, lens_kind="uniform",
                                       lens_args=(512, 4096), q_per_seq=4),
    # the Llama-3-8B decode batch with an FP8 E4M3 pool (K and V scale 1/64)
    "llama3-8b-fp8": Workload("llama3-8b-fp8", 1003, 256, 32, 8, 128, 16, torch.bfloat16,
                              lens_kind="uniform", lens_args=(512, 4096),
                              cache_dtype=torch.float8_e4m3fn, kv_scale=1.0 / 64),
    "mixed-llama3-8b-bf16": Workload("mixed-llama3-8b-bf16", 1005, 192, 32, 8, 128, 32,
                                     torch.bfloat16, lens_kind="lognormal",
                                     lens_args=(7.0, 1.0, 16, 32768),
                                     pool="bytes", pool_arg=60e9,
                                     shared_prefix_tokens=1024, shared_fraction=0.25,
                                     prefill_requests=4, prefill_chunk=512,
                                     prefill_ctx_range=(1024, 8192)),
    "mixed-llama3-8b-fp8": Workload("mixed-llama3-8b-fp8", 1005, 192, 32, 8, 128, 32,
                                    torch.bfloat16, lens_kind="lognormal",
                                    lens_args=(7.0, 1.0, 16, 32768),
                                    pool="bytes", pool_arg=60e9,
                                    shared_prefix_tokens=1024, shared_fraction=0.25,
                                    prefill_requests=4, prefill_chunk=512,
                                    prefill_ctx_range=(1024, 8192),
                                    cache_dtype=torch.float8_e4m3fn, kv_scale=1.0 / 64),
}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _rng(seed: int, tag: str, *idx: int) -> np.random.Generator:
    return np.random.default_rng([seed, _TAGS[tag], *idx])


def _normal(rng: np.random.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    # round-to-nearest-even into the storage dtype
    return torch.from_numpy(x).to(dtype)


def _threads() -> int:
    return max(1, min(32, len(os.sched_getaffinity(0))))


class Draws:
    """All random draws of one workload, replaceable by a different seed."""

    def __init__(self, wl: Workload, seed: int | None = None):
        self.wl = wl
        self.seed = wl.seed if seed is None else seed

    # ---- lengths --------------------------------------------------------
    def decode_lens(self) -> np.ndarray:
        """Context length of every decode sequence (new token included)."""
        wl, rng = self.wl, _rng(self.seed, "lens")
        if wl.lens_kind == "list":
            lens = np.array(wl.lens_args, dtype=np.int64)
            assert len(lens) == wl.batch
        elif wl.lens_kind == "uniform":
            lo, hi = wl.lens_args
            lens = rng.integers(lo, hi, size=wl.batch, endpoint=True)
        elif wl.lens_kind == "const":
            lens = np.full(wl.batch, wl.lens_args[0], dtype=np.int64)
        elif wl.lens_kind == "lognormal":
            mu, sigma, lo, hi = wl.lens_args
            draw = rng.lognormal(mu, sigma, size=wl.batch)
            lens = np.rint(draw).astype(np.int64)
            sh = self.sharers()
            lens = np.where(sh, lens + wl.shared_prefix_tokens, lens)
            lens = np.clip(lens, lo, hi)
        else:
            raise ValueError(wl.lens_kind)
        return lens.astype(np.int32)

    def sharers(self) -> np.ndarray:
        """Boolean mask: which decode sequences start with the shared prefix."""
        wl = self.wl
        mask = np.zeros(wl.batch, dtype=bool)
        n = int(round(wl.batch * wl.shared_fraction))
        if n:
            idx = _rng(self.seed, "share").choice(wl.batch, size=n, replace=False)
            mask[idx] = True
        return mask

    def prefill_ctx(self) -> np.ndarray:
        """Tokens already cached for each chunked-prefill request."""
        wl = self.wl
        if wl.prefill_requests == 0:
            return np.zeros(0, dtype=np.int32)
        lo, hi = wl.prefill_ctx_range
        return _rng(self.seed, "plens").integers(lo, hi, size=wl.prefill_requests,
                                                 endpoint=True).astype(np.int32)

    def prefill_chunks(self) -> np.ndarray:
        return np.full(self.wl.prefill_requests, self.wl.prefill_chunk, dtype=np.int32)

    # ---- pool order -----------------------------------------------------
    def free_order(self, num_blocks: int) -> np.ndarray:
        """Initial order of the free-block queue: a seeded permutation."""
        return _rng(self.seed, "order").permutation(num_blocks).astype(np.int32)

    # ---- tensors ----------------------------------------------------------
    def q(self) -> torch.Tensor:
        """[B][n_q][d], or [B][q_per_seq][n_q][d] when a sequence has several rows."""
        wl = self.wl
        shape = ((wl.batch, wl.n_q_heads, wl.head_dim) if wl.q_per_seq == 1 else
                 (wl.batch, wl.q_per_seq, wl.n_q_heads, wl.head_dim))
        return _normal(_rng(self.seed, "q"), shape, wl.std, wl.dtype)

    def prefix_kv(self):
        wl = self.wl
        shape = (wl.shared_prefix_tokens, wl.n_kv_heads, wl.head_dim)
        r = _rng(self.seed, "prefix")
        return _normal(r, shape, wl.std, wl.dtype), _normal(r, shape, wl.std, wl.dtype)

    def seq_kv(self, s: int, length: int, shared: bool = False, prefix=None):
        """Logical K and V of decode sequence s: [length][n_kv][d] each."""
        wl = self.wl
        r = _rng(self.seed, "kv", s)
        p = wl.shared_prefix_tokens if shared else 0
        shape = (length - p, wl.n_kv_heads, wl.head_dim)
        k, v = _normal(r, shape, wl.std, wl.dtype), _normal(r, shape, wl.std, wl.dtype)
        if p:
            pk, pv = prefix if prefix is not None else self.prefix_kv()
            k, v = torch.cat([pk, k]), torch.cat([pv, v])
        return k, v

    def all_seq_kv(self, lens, sharers=None, threads: int | None = None):
        """Logical K/V of every decode sequence (drawn in parallel)."""
        sharers = np.zeros(len(lens), bool) if sharers is None else sharers
        prefix = self.prefix_kv() if sharers.any() else None
        with ThreadPoolExecutor(threads or _threads()) as ex:
            return list(ex.map(lambda s: self.seq_kv(s, int(lens[s]), bool(sharers[s]), prefix),
                               range(len(lens))))

    def prefill_q(self, r: int) -> torch.Tensor:
        wl = self.wl
        return _normal(_rng(self.seed, "pq", r), (wl.prefill_chunk, wl.n_q_heads, wl.head_dim),
                       wl.std, wl.dtype)

    def prefill_kv(self, r: int, length: int):
        """Logical K/V of prefill request r over all its tokens (context + chunk)."""
        wl = self.wl
        rr = _rng(self.seed, "pkv", r)
        shape = (length, wl.n_kv_heads, wl.head_dim)
        return _normal(rr, shape, wl.std, wl.dtype), _normal(rr, shape, wl.std, wl.dtype)


def random_case(seed: int, batch: int, n_q: int, n_kv: int, d: int, bs: int, dtype, lens,
                std: float = 1.0, cache_dtype=None, kv_scale: float = 1.0) -> Workload:
    """An ad-hoc workload for property tests (explicit lengths, 1.5x pool)."""
    return Workload(f"case-{seed}", seed, batch, n_q, n_kv, d, bs, dtype, std=std,
                    lens_kind="list", lens_args=tuple(int(x) for x in lens),
                    cache_dtype=cache_dtype, kv_scale=kv_scale)


def token_stream(seed: int, index: int, length: int, vocab: int) -> np.ndarray:
    """Token ids of one synthetic request (uniform over the vocabulary)."""
    return _rng(seed, "toks", index).integers(0, vocab, size=length).astype(np.int32)


def token_keyed_kv(seed: int, tokens, n_kv: int, head_dim: int, dtype, std: float = 1.0):
    """K and V rows [len][n_kv][d] for a token sequence where the row at
    position p is drawn from a generator keyed by tokens[0..p] only: requests
    that share a prefix of tokens get identical rows over that prefix."""
    ks, vs = [], []
    toks = [int(t) for t in tokens]
    for p in range(len(toks)):
        r = np.random.default_rng([seed, _TAGS["tokkv"], p, *toks[:p + 1]])
        ks.append(_normal(r, (n_kv, head_dim), std, dtype))
        vs.append(_normal(r, (n_kv, head_dim), std, dtype))
    return torch.stack(ks), torch.stack(vs)
