"""Shared test helpers: expected values come from the oracle fed by the seeded
generator only (never from the CUDA path)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_25_gb300 import inputs

# max |error| bars: fp32 inputs 1e-5; bf16/fp16 inputs 2e-3 (fp32 accumulation)
TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3, torch.float16: 2e-3}


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Half a unit in the last place of |x| in dtype: the rounding of the store."""
    mant = {torch.bfloat16: 8, torch.float16: 11, torch.float32: 24}[dtype]
    ax = np.maximum(np.abs(x), {torch.float16: 6.1e-5, torch.bfloat16: 1e-30,
                                torch.float32: 1e-30}[dtype])
    e = np.floor(np.log2(ax))
    return 0.5 * np.exp2(e - (mant - 1))


def stored_kv(wl, k, v):
    """The K/V values a pool of the workload holds for rows k, v: the rows
    themselves, or for FP8 pools the oracle's E4M3 codes times the scale."""
    if wl.pool_dtype != torch.float8_e4m3fn:
        return k, v
    kq = oracle.dequantize_fp8(oracle.quantize_fp8(k, wl.kv_scale), wl.kv_scale)
    vq = oracle.dequantize_fp8(oracle.quantize_fp8(v, wl.kv_scale), wl.kv_scale)
    return kq, vq


def oracle_decode(step, seqs=None, threads=None) -> np.ndarray:
    """fp64 decode for the given decode sequences of a PagedStep's workload."""
    dr, wl = step.draws, step.wl
    seqs = list(range(wl.batch)) if seqs is None else list(seqs)
    prefix = dr.prefix_kv() if step.prefix else None
    ks, vs = [], []
    for s in seqs:
        k, v = dr.seq_kv(s, int(step.lens[s]), bool(step.sharers[s]), prefix)
        k, v = stored_kv(wl, k, v)
        ks.append(k); vs.append(v)
    q = dr.q()[seqs]
    return oracle.decode(q, ks, vs, wl.scale, threads=threads)


def oracle_decode_all(step, chunk: int = 32, threads=None) -> np.ndarray:
    """fp64 outputs of every decode sequence of a PagedStep, computed chunk
    sequences at a time (bounded host memory at full workload sizes):
    [B][n_q][d], or [B][q_per_seq][n_q][d] for several query rows per
    sequence (query i at position L - q_per_seq + i, causal among the rows)."""
    from concurrent.futures import ThreadPoolExecutor
    dr, wl = step.draws, step.wl
    prefix = dr.prefix_kv() if step.prefix else None
    q = dr.q()
    outs = []
    draw = lambda s: dr.seq_kv(s, int(step.lens[s]), bool(step.sharers[s]), prefix)
    ex = ThreadPoolExecutor(8)
    for s0 in range(0, wl.batch, chunk):
        seqs = range(s0, min(wl.batch, s0 + chunk))
        ks, vs = [], []
        for k, v in ex.map(draw, seqs):      # seeded per sequence: order-independent
            k, v = stored_kv(wl, k, v)
            ks.append(k); vs.append(v)
        if wl.q_per_seq == 1:
            outs.append(oracle.decode(q[s0:s0 + len(ks)], ks, vs, wl.scale, threads=threads))
        else:
            outs.append(np.stack(oracle.prefill([q[s] for s in seqs], ks, vs, wl.scale,
                                                threads=threads)))
    ex.shutdown()
    return np.concatenate(outs)


def oracle_prefill_all(step, threads=None) -> np.ndarray:
    """fp64 outputs of every chunked-prefill row of a PagedStep, [sum C][n_q][d]."""
    dr, wl = step.draws, step.wl
    qs, ks, vs = [], [], []
    for r in range(step.R):
        k, v = stored_kv(wl, *dr.prefill_kv(r, int(step.p_lens[r])))
        qs.append(dr.prefill_q(r)); ks.append(k); vs.append(v)
    return np.concatenate(oracle.prefill(qs, ks, vs, wl.scale, threads=threads))


def check_low_precision(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype,
                        tol: float = 2e-3) -> float:
    """Output stored in bf16/fp16: |got - ref| <= tol + half an ulp of ref in
    that dtype (the store's own rounding).  Returns the largest excess."""
    g = got.detach().float().cpu().numpy().astype(np.float64)
    excess = np.abs(g - ref) - (tol + half_ulp(ref, dtype))
    return float(excess.max())


def oracle_prefill_rows(step, r: int, rows, threads=None) -> np.ndarray:
    """fp64 outputs of chosen query rows of prefill request r: row i attends
    keys 0..L-C+i, i.e. a decode over the truncated logical K/V."""
    dr, wl = step.draws, step.wl
    L, C = int(step.p_lens[r]), int(step.p_chunk[r])
    k, v = stored_kv(wl, *dr.prefill_kv(r, L))
    q = dr.prefill_q(r)
    outs = []
    for i in rows:
        p = L - C + i
        outs.append(oracle.decode(q[i:i + 1], [k[:p + 1]], [v[:p + 1]], wl.scale, threads=threads)[0])
    return np.stack(outs)


def max_err(got: torch.Tensor, ref: np.ndarray) -> float:
    return float(np.max(np.abs(got.detach().float().cpu().numpy().astype(np.float64) - ref)))
