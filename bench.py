"""Benchmark of the paged-attention hot path on one GB300 (or N replicas).

A step is one pass of the whole hot path over one batch: append the new
tokens' K/V (pa_reshape_and_cache), decode one token per sequence (pa_decode:
split-K partitions plus the reduce), and the chunked-prefill requests when the
workload has any (pa_prefill_chunk).  The default workload is the Llama-3-8B
shaped decode batch: 256 sequences, 32 query / 8 KV heads, head_dim 128,
16-token blocks, lengths U[512, 4096], bf16 — about 2.4 GB of K/V per step,
far more than the 129 MB L2, so no flush is needed between steps.

Metric: unique K/V bytes the decode must read per step / step time, in GB/s,
plus decode tokens/s and steps/s.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU fp64 oracle, timed on host cores
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged-attn decode KV-read GB/s (% of GB300 HBM peak); decode tokens/s"
DEFAULT_WORKLOAD = "llama3-8b-bf16"
FALLBACK_HBM_GBS = 6800.0

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch,
# valid only while the kernel sources are byte-identical to what was profiled
# (sha256 prefix of DECODE_SOURCES / PREFILL_SOURCES).  Decode: (bytes, unique
# K/V bytes of the captured launch, what was captured); a record of another
# batch of the same workload is scaled by its unique K/V bytes.
NCU_TRAFFIC = {
    ("llama3-8b-bf16", "156a5e1d9ddf2e4e"): (2371995904 + 13372672, 2359717888,
                                             "full 256-sequence batch, one-pass capture"),
    ("llama3-8b-fp8", "156a5e1d9ddf2e4e"): (1188186112 + 12436224, 1179858944,
                                            "full 256-sequence batch, one-pass capture"),
}
# chunked prefill of the mixed step (the compact-pool capture runs the same four
# chunks as the 60 GB pool): bytes per launch
NCU_PREFILL_TRAFFIC = {
    ("mixed-llama3-8b-bf16", "32cbb231cfdc1f9a"): (98471424 + 4715776, "compact pool, --set full"),
    ("mixed-llama3-8b-fp8", "32cbb231cfdc1f9a"): (57562624 + 1404672, "compact pool, --set full"),
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _peaks_tensor():
    """Dense bf16 tensor peak: the sustained cuBLAS figure (kernels timed inside a
    long step loop)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["bf16_tflops_sustained"]), "bf16_tflops_sustained (measured)"
    except Exception:
        return 1700.0, "bf16 sustained (fallback)"


# the kernels' sources: traffic figures hold only while these are unchanged
DECODE_SOURCES = ("decode_mma.cuh", "decode.cu", "decode_verify.cu", "pa_device.cuh")
PREFILL_SOURCES = ("prefill_tc.cu", "pa_device.cuh")


def _src_hash(names) -> str:
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "paged_kv_cache_25_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _cores() -> int:
    return len(os.sched_getaffinity(0))


# ---------------------------------------------------------------- ranks
def max_over_ranks(vals, device="cpu"):
    """Element-wise max of per-rank values over all ranks (timings: the job is
    as slow as its slowest replica).  No-op on a single process."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Weak scaling: every rank processes its own batch of the same size, so the
    job moves world x bytes_per_rank per step of the slowest rank."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- reference arm
def oracle_sample(wl_name: str, n_seqs: int | None, target_s: float, seed_offset: int = 0):
    """Times the CPU oracle on a bounded sample of the workload's decode batch.
    Returns (GB/s, seconds per sample, sample description, threads)."""
    import oracle
    from paged_kv_cache_25_gb300 import inputs
    wl = inputs.get(wl_name)
    dr = inputs.Draws(wl, wl.seed + seed_offset)
    lens, sharers = dr.decode_lens(), dr.sharers()
    prefix = dr.prefix_kv() if sharers.any() else None
    q_all = dr.q()
    threads = oracle.default_threads()
    row = 2 * wl.n_kv_heads * wl.head_dim * wl.pool_elem_bytes
    fp8 = wl.cache_dtype is not None

    def run(seqs):
        ks, vs = [], []
        for s in seqs:
            k, v = dr.seq_kv(s, int(lens[s]), bool(sharers[s]), prefix)
            if fp8:   # the pool holds E4M3 codes: the oracle reads their values
                k = oracle.dequantize_fp8(oracle.quantize_fp8(k, wl.kv_scale), wl.kv_scale)
                v = oracle.dequantize_fp8(oracle.quantize_fp8(v, wl.kv_scale), wl.kv_scale)
            ks.append(k); vs.append(v)
        t0 = time.perf_counter()
        if wl.q_per_seq == 1:
            oracle.decode(q_all[seqs], ks, vs, wl.scale, threads=threads)
        else:   # several query rows per sequence: chunks of q_per_seq rows
            oracle.prefill([q_all[s] for s in seqs], ks, vs, wl.scale, threads=threads)
        return time.perf_counter() - t0

    if n_seqs is None:
        probe = list(range(min(2, wl.batch)))
        t = run(probe)
        per_tok = t / max(1, int(lens[probe].sum()))
        want = target_s / max(per_tok, 1e-9)
        n, acc = 0, 0
        while n < wl.batch and acc < want:
            acc += int(lens[n]); n += 1
        n_seqs = max(1, n)
    seqs = list(range(n_seqs))
    t = run(seqs)
    kv = int(lens[seqs].sum()) * row
    desc = (f"first {n_seqs} of {wl.batch} decode sequences ({int(lens[seqs].sum())} of "
            f"{int(lens.sum())} tokens), fp64 oracle incl. its fp64 packing, {threads} threads")
    return kv / t / 1e9, t, desc, threads, n_seqs


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from paged_kv_cache_25_gb300 import inputs
    wl = inputs.get(args.workload)
    # size each step's sample so W + K steps take a few minutes at most
    _, t_probe, _, threads, n = oracle_sample(args.workload, None, 2.0)
    for _ in range(args.warmup):
        oracle_sample(args.workload, n, 0)
    vals, times = [], []
    desc = ""
    for _ in range(args.steps):
        v, t, desc, threads, _ = oracle_sample(args.workload, n, 0)
        vals.append(v); times.append(t)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "n_q_heads": wl.n_q_heads,
                   "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "sample_seqs": n},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def _ev():
    import torch
    return torch.cuda.Event(enable_timing=True)


def _nvtx(name):
    import torch
    return torch.cuda.nvtx.range(name)


def _flush_buffer(st, dev):
    """A 2 x L2 buffer to write before each timed step when the pool would
    otherwise sit in L2 (None when the pool is larger than that)."""
    import torch
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    pool_bytes = (st.k_cache.numel() * st.k_cache.element_size() +
                  st.v_cache.numel() * st.v_cache.element_size())
    if pool_bytes >= 2 * l2_bytes:
        return None, l2_bytes, pool_bytes
    return torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev), l2_bytes, pool_bytes


def _l2_note(flush, l2_bytes, pool_bytes, kv_unique):
    if flush is None:
        return (f"inputs larger than L2 ({pool_bytes / 1e9:.2f} GB pool, "
                f"{kv_unique / 1e9:.2f} GB of K/V read per step); no flush")
    return (f"L2 flushed before every timed step (a {2 * l2_bytes >> 20} MiB write, outside "
            f"the step's events); the pool ({pool_bytes / 1e6:.0f} MB) would fit in L2")


def timed_steps(st, stream, n, flush=None):
    """n steps, each bracketed by a pair of CUDA events on the step's stream
    and nothing else between its kernels (the L2 flush, if any, goes before
    the first event).  Returns the per-step times in ms."""
    import torch
    ev = [(_ev(), _ev()) for _ in range(n)]
    for i in range(n):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        st.step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def profiled_steps(st, stream, n, flush=None):
    """n steps, each bracketed by CUDA events on the step's stream, the decode
    kernel by the library's profiling events and the chunked prefill (if any)
    by events on its side stream.  Returns per-step lists in ms: step, decode
    kernel, prefill kernel (inside the step).  The events recorded between the
    step's kernels serialise them, so step times come from timed_steps."""
    import torch
    from paged_kv_cache_25_gb300 import binding as pa
    ev = [(_ev(), _ev()) for _ in range(n)]
    dk = [(_ev(), _ev()) for _ in range(n)]
    pf = [(_ev(), _ev()) for _ in range(n)] if st.R else [None] * n
    for a, b in dk:     # torch creates a CUDA event at its first record; the library
        a.record(stream)    # records these handles itself, so they must exist first
        b.record(stream)
    torch.cuda.synchronize()
    for i in range(n):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        pa.pa_set_profile_events(*dk[i])
        st.step(prefill_events=pf[i])
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    pa.pa_set_profile_events(None, None)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dec_ms = [a.elapsed_time(b) for a, b in dk]
    pf_ms = [a.elapsed_time(b) for a, b in pf] if st.R else None
    return step_ms, dec_ms, pf_ms


def prefill_alone_ms(st, stream, n):
    """The step's chunked-prefill call timed on its own (inside the step it
    shares the SMs with the decode launched beside it)."""
    import torch
    from paged_kv_cache_25_gb300 import binding as pa
    wl = st.wl
    pairs = []
    for i in range(n + 3):
        a_, b_ = _ev(), _ev()
        a_.record(stream)
        pa.pa_prefill_chunk(st.p_out, st.p_q_dev, st.k_cache, st.v_cache, st.p_block_tables,
                            st.query_start_loc, st.p_context_lens, int(st.p_chunk.max()),
                            wl.scale, wl.block_size, stream=stream, **st.kv_scales)
        b_.record(stream)
        if i >= 3:
            pairs.append((a_, b_))
    torch.cuda.synchronize()
    return [a_.elapsed_time(b_) for a_, b_ in pairs]


def _dtype_name(wl):
    if wl.cache_dtype is not None:
        return "e4m3 K/V, f16 products"
    return {"torch.bfloat16": "bf16", "torch.float16": "f16", "torch.float32": "f32"}[str(wl.dtype)]


def _traffic(name, kv_unique):
    """(bytes per launch, how it was obtained) or (None, reason)."""
    rec = NCU_TRAFFIC.get((name, _src_hash(DECODE_SOURCES)))
    if rec is None:
        return None, "no ncu capture of the current decode sources on this workload"
    b, u, how = rec
    return int(round(b * kv_unique / u)), how


def _prefill_traffic(name):
    rec = NCU_PREFILL_TRAFFIC.get((name, _src_hash(PREFILL_SOURCES)))
    return (rec[0], rec[1]) if rec else (None, "no ncu capture of the current prefill sources")


def _prefill_roofline(st, pf_ms):
    flops = st.prefill_flops()
    tf, tf_src = _peaks_tensor()
    achieved = flops / (statistics.mean(pf_ms) * 1e-3) / 1e12
    traffic, how = _prefill_traffic(st.wl.name)
    return flops, {
        "bound": "tensor", "achieved": achieved, "peak": tf, "unit": "TFLOP/s",
        "frac": achieved / tf, "traffic": traffic, "traffic_source": how,
        "kernel": "prefill_tc_kernel",
        "peak_source": tf_src, "kernel_ms_mean": statistics.mean(pf_ms),
        "kernel_ms_median": statistics.median(pf_ms), "launches_timed": len(pf_ms),
        "timing": "kernel alone (in the step it overlaps the decode)"}


def measure_workload(name, dev, phys, target_s=0.6, min_steps=50, max_steps=3000):
    """One record per workload: a fresh PagedStep, 10 warm-up steps, then
    at least min_steps steps (as many as fit in ~target_s) with per-step
    events; medians, the decode kernel's roofline, clocks over the loop."""
    import torch
    from paged_kv_cache_25_gb300 import binding as pa
    from paged_kv_cache_25_gb300 import inputs
    from paged_kv_cache_25_gb300.step import PagedStep
    wl = inputs.get(name)
    t0 = time.perf_counter()
    st = PagedStep(wl, device=dev)
    setup_s = time.perf_counter() - t0
    stream = torch.cuda.current_stream(dev)
    flush, l2_bytes, pool_bytes = _flush_buffer(st, dev)
    for _ in range(10):
        st.step()
    torch.cuda.synchronize(dev)
    probe = timed_steps(st, stream, 5, flush)
    n = int(min(max_steps, max(min_steps, target_s / max(statistics.median(probe), 1e-3) * 1e3)))
    clocks = ClockSampler(phys)
    clocks.start()
    time.sleep(0.3)
    with _nvtx(f"workload {name}"):
        step_ms = timed_steps(st, stream, n, flush)
    clk = clocks.stop()
    with _nvtx(f"workload {name} kernels"):
        _, dec_ms, pf_ms = profiled_steps(st, stream, min(n, 500), flush)
    assert pa.pa_get_device_error() == 0
    kv_unique = st.kv_bytes_unique()
    peak, peak_kind = _peaks()
    med = statistics.median(step_ms)
    dmean, dmed = statistics.mean(dec_ms), statistics.median(dec_ms)
    achieved = kv_unique / (dmean * 1e-3) / 1e9
    rec = {
        "workload": wl.name, "dtype": _dtype_name(wl), "batch": wl.batch,
        "n_q_heads": wl.n_q_heads, "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
        "block_size": wl.block_size, "q_per_seq": wl.q_per_seq, "prefill_requests": st.R,
        "num_blocks": st.num_blocks, "steps": n, "warmup": 10,
        "ms_per_step_median": med, "ms_per_step_mean": statistics.mean(step_ms),
        "value": kv_unique / (med * 1e-3) / 1e9, "unit": "GB/s",
        "decode_tokens_per_s": wl.batch * wl.q_per_seq / (med * 1e-3),
        "steps_per_s": 1e3 / med,
        "kv_bytes_unique_per_step": kv_unique,
        "kv_bytes_block_granular_per_step": st.kv_bytes_block_granular(),
        "kv_bytes_logical_per_step": st.kv_bytes_logical(),
        "decode_kernel_ms_mean": dmean, "decode_kernel_ms_median": dmed,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _traffic(wl.name, kv_unique)[0],
                     "traffic_source": _traffic(wl.name, kv_unique)[1],
                     "kernel": "decode_mma_kernel", "peak_source": f"hbm_gbs ({peak_kind})"},
        "l2": _l2_note(flush, l2_bytes, pool_bytes, kv_unique),
        "clocks": clk, "setup_s": setup_s,
    }
    if st.R:
        rec["prefill_kernel_ms_in_step_median"] = statistics.median(pf_ms)
        rec["prefill_tokens_per_s"] = int(st.p_chunk.sum()) / (med * 1e-3)
        alone = prefill_alone_ms(st, stream, max(50, min(n, 200)))
        rec["prefill_flops_per_step"], rec["roofline_prefill"] = _prefill_roofline(st, alone)
    if wl.batch <= 64 and wl.cache_dtype is None and wl.q_per_seq == 1:
        # BASELINE's CPU plan: the oracle single-threaded on the small configs
        rec["cpu_baseline_1thread"] = oracle_one_thread(st)
    del st
    torch.cuda.empty_cache()
    return rec


def oracle_one_thread(st):
    """The oracle over the whole decode batch of a small workload on one host
    thread (inputs regenerated from the seeded draws, packing excluded)."""
    import oracle
    dr, wl = st.draws, st.wl
    kv = [dr.seq_kv(s, int(st.lens[s])) for s in range(wl.batch)]
    q = dr.q()
    t0 = time.perf_counter()
    oracle.decode(q, [k for k, _ in kv], [v for _, v in kv], wl.scale, threads=1)
    t = time.perf_counter() - t0
    kvb = st.kv_bytes_logical()
    return {"value": kvb / t / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": t, "sample": f"all {wl.batch} decode sequences, one thread"}


OTHER_WORKLOADS = ("tiny-fp32", "tinyllama-bf16", "opt13b-fp16", "mixed-llama3-8b-bf16",
                   "llama3-8b-fp8", "llama3-8b-bf16-verify4", "mixed-llama3-8b-fp8")


def run_ours(args, rank, world, local_rank):
    import torch
    from paged_kv_cache_25_gb300 import binding as pa
    from paged_kv_cache_25_gb300 import build as pa_build
    from paged_kv_cache_25_gb300 import inputs
    from paged_kv_cache_25_gb300.step import PagedStep

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:                    # one builder; the other ranks load its library
        pa_build.build()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    pa.lib()
    wl = inputs.get(args.workload)
    if args.batch:
        wl = dataclasses.replace(wl, batch=args.batch)
    if args.compact_pool:
        wl = dataclasses.replace(wl, pool="scale", pool_arg=1.5)
    st = PagedStep(wl, seed=wl.seed + rank, device=dev)
    stream = torch.cuda.current_stream(dev)
    torch.cuda.synchronize(dev)
    assert pa.pa_get_device_error() == 0

    # launches of this library per step: cache write, decode, the split-K
    # reduce when some sequence spans several partitions, the chunked prefill
    launches_per_step = 2 + (1 if st.workspace is not None else 0) + (1 if st.R else 0)
    warmup = max(args.warmup, 3)
    for _ in range(warmup):
        st.step()
    torch.cuda.synchronize(dev)

    # ---- device-timed region: inputs resident in HBM ---------------------
    # K steps back to back between two events on the step's stream; with a
    # pool small enough to sit in L2, each step is preceded by a 2 x L2 write
    # outside its own events and the time is the sum of the steps' events.
    flush, l2_bytes, pool_bytes = _flush_buffer(st, dev)
    t_start, t_stop = _ev(), _ev()
    sev = [(_ev(), _ev()) for _ in range(args.steps)] if flush is not None else None
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    phys = int(vis[local_rank]) if len(vis) > local_rank and vis[local_rank].strip().isdigit() else local_rank
    clocks = ClockSampler(phys)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)   # let the sampler start before the timed region
    with _nvtx("timed steps"):
        t_start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush.fill_(i & 0xFF)
                sev[i][0].record(stream)
            st.step()
            if flush is not None:
                sev[i][1].record(stream)
        t_stop.record(stream)
        torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    assert pa.pa_get_device_error() == 0
    ms_total = (t_start.elapsed_time(t_stop) if flush is None else
                sum(a.elapsed_time(b) for a, b in sev))

    # ---- per-step times (median) and the decode kernel per launch, in loops of
    # their own after the timed region
    n_prof = max(args.steps, args.kernel_steps)
    with _nvtx("step times"):
        step_ms = timed_steps(st, stream, n_prof, flush)
    with _nvtx("kernel timing"):
        _, decode_ms, prefill_ms = profiled_steps(st, stream, n_prof, flush)
    assert pa.pa_get_device_error() == 0

    # ---- end to end through the public API with host buffers --------------
    # Every step uploads its inputs from pinned host memory and reads its
    # outputs back.  The inputs travel as one packed pinned buffer (one copy
    # per step, the tensors are views into it; likewise the outputs), so the
    # host issues few calls.  With inputs larger than L2 the copies are
    # pipelined: two device buffer sets, uploads on one copy stream and
    # read-backs on another, so step i+1's upload and step i-1's read-back
    # overlap step i's kernels; a set is reused only after its previous
    # step's read-back.
    B = wl.batch
    pin_of = ("q", "new_k", "new_v", "new_slots", "block_tables", "context_lens", "p_q_dev",
              "query_start_loc", "p_block_tables", "p_context_lens")
    own = st.io_set()
    ins = [n for n in pin_of if n in own]
    outs = [n for n in ("out", "p_out") if n in own]

    def layout(names):
        off, pos = {}, 0
        for n in names:
            off[n] = pos
            pos += -(-own[n].numel() * own[n].element_size() // 256) * 256
        return off, pos

    in_off, in_bytes = layout(ins)
    out_off, out_bytes = layout(outs)

    def views(buf, names, off):
        return {n: buf[off[n]:off[n] + own[n].numel() * own[n].element_size()]
                .view(own[n].dtype).view(own[n].shape) for n in names}

    host_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    for n, v in views(host_in, ins, in_off).items():
        v.copy_(own[n].cpu())
    host_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    dev_in = [torch.empty(in_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    dev_out = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    sets = [{**views(dev_in[b_], ins, in_off), **views(dev_out[b_], outs, out_off)}
            for b_ in range(2)]
    h2d, d2h = in_bytes, out_bytes
    e2e_steps = max(1, min(args.steps, 200))
    copy = torch.cuda.Stream(device=dev)      # uploads
    back = torch.cuda.Stream(device=dev)      # read-backs
    up = [torch.cuda.Event(), torch.cuda.Event()]
    comp = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    for ev_ in done:
        ev_.record(stream)

    def e2e_step(i):
        b = i & 1
        copy.wait_event(done[b])        # step i-2 is done with this buffer set
        with torch.cuda.stream(copy):
            dev_in[b].copy_(host_in, non_blocking=True)
        up[b].record(copy)
        stream.wait_event(up[b])
        st.step(io=sets[b])
        comp[b].record(stream)
        back.wait_event(comp[b])
        with torch.cuda.stream(back):
            host_out[b].copy_(dev_out[b], non_blocking=True)
        done[b].record(back)

    def e2e_serial():
        dev_in[0].copy_(host_in, non_blocking=True)
        st.step(io=sets[0])
        host_out[0].copy_(dev_out[0], non_blocking=True)

    for i in range(3):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    with _nvtx("end to end"):
        if flush is None:
            e0, e1 = _ev(), _ev()
            e0.record(stream)
            copy.wait_stream(stream)
            back.wait_stream(stream)
            for i in range(e2e_steps):
                e2e_step(i)
            stream.wait_stream(back)        # the last read-back is inside the timed region
            e1.record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = e0.elapsed_time(e1) / e2e_steps
            e2e_mode = "pipelined: uploads and read-backs on two copy streams, double-buffered"
        else:   # a flush between steps: one step at a time
            eev = [(_ev(), _ev()) for _ in range(e2e_steps)]
            for i in range(e2e_steps):
                flush.fill_(i & 0xFF)
                eev[i][0].record(stream)
                e2e_serial()
                eev[i][1].record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = sum(a.elapsed_time(b) for a, b in eev) / e2e_steps
            e2e_mode = "serial: upload, step, read-back per flushed step"

    # ---- reductions over ranks (max time) --------------------------------
    ms_step = ms_total / args.steps
    dec_ms = statistics.mean(decode_ms)
    ms_step, e2e_ms, dec_ms = max_over_ranks([ms_step, e2e_ms, dec_ms], dev)

    kv_unique = st.kv_bytes_unique()
    value = whole_job_gbs(kv_unique, world, ms_step)
    peak, peak_kind = _peaks()
    # algorithmic bytes of the main decode kernel per launch: the unique K/V
    # bytes (q, the output and the partials are < 0.5 % and not counted)
    achieved = kv_unique / (dec_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": _dtype_name(wl),
        "data": "synthetic (seeded N(0,1) K/V/Q, random block scatter)",
        "config": {"workload": wl.name, "batch": B, "n_q_heads": wl.n_q_heads,
                   "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "num_blocks": st.num_blocks,
                   "prefill_requests": st.R, "q_per_seq": wl.q_per_seq,
                   "parallelism": f"replicas x{world}",
                   "l2": _l2_note(flush, l2_bytes, pool_bytes, kv_unique)},
        "decode_tokens_per_s": world * B * wl.q_per_seq / (ms_step * 1e-3),
        "steps_per_s": 1e3 / ms_step,
        "pct_of_hbm_peak": 100.0 * value / world / peak,
        "kv_bytes_unique_per_step": kv_unique,
        "kv_bytes_block_granular_per_step": st.kv_bytes_block_granular(),
        "kv_bytes_logical_per_step": st.kv_bytes_logical(),
        "ms_per_step_median": statistics.median(step_ms),
        "decode_kernel_ms": dec_ms,
        "decode_kernel_ms_median": statistics.median(decode_ms),
        "kernel_timing": (f"after the timed region: {n_prof} steps each bracketed by CUDA events "
                          f"(ms_per_step_median), then {n_prof} more with the decode kernel "
                          "bracketed by events on the step's stream (decode_kernel_ms)"),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": _traffic(wl.name, kv_unique)[0],
                     "traffic_source": _traffic(wl.name, kv_unique)[1],
                     "kernel": "decode_mma_kernel", "peak_source": f"hbm_gbs ({peak_kind})"},
        "e2e": {"value": whole_job_gbs(kv_unique, world, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": e2e_mode},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if st.R:
        alone = prefill_alone_ms(st, stream, max(20, min(args.steps, 100)))
        line["prefill_flops_per_step"], line["roofline_prefill"] = _prefill_roofline(st, alone)
        line["prefill_kernel_ms_in_step"] = statistics.mean(prefill_ms)
        line["prefill_tokens_per_s"] = world * int(st.p_chunk.sum()) / (ms_step * 1e-3)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, t, desc, threads, _ = oracle_sample(wl.name, None, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": t}
    if world == 1 and args.workloads != "none":
        del st, sets, dev_in, dev_out
        torch.cuda.empty_cache()
        names = (OTHER_WORKLOADS if args.workloads == "all" else
                 tuple(n for n in args.workloads.split(",") if n))
        recs = []
        for name in names:
            if name == wl.name:
                continue
            recs.append(measure_workload(name, dev, phys))
        line["workloads"] = recs
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--compact-pool", action="store_true",
                    help="size the pool at 1.5x the blocks needed (profiling a smaller case)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's decode batch (profiling a smaller case)")
    ap.add_argument("--kernel-steps", type=int, default=200,
                    help="steps of the per-launch timing loop after the timed region")
    ap.add_argument("--workloads", default="all",
                    help="'all' (every other configuration, one record each, one GPU only), "
                         "'none', or a comma-separated list of workload names")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
