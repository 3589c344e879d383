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

# ncu DRAM traffic of the main decode kernel on this workload, per launch
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only while the kernel
# sources are byte-identical to what was profiled (sha256 of DECODE_SOURCES).
NCU_TRAFFIC = {
    # one-pass ncu captures (--metrics dram__bytes_read.sum,dram__bytes_write.sum,
    # full-size workload, 4th launch); profiles/decode_dram_full_size.md
    ("llama3-8b-bf16", 256, "ad80b383e235384f"): 2371977216 + 13616640,
    ("llama3-8b-fp8", 256, "ad80b383e235384f"): 1188184576 + 12948224,
    ("llama3-8b-bf16-verify4", 256, "ad80b383e235384f"): 2384849152 + 44538624,
    ("opt13b-fp16", 128, "ad80b383e235384f"): 5371655936 + 8389376,
    ("mixed-llama3-8b-bf16", 192, "ad80b383e235384f"): 1446247936 + 9858304,
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


# the decode kernel's sources: traffic figures hold only while these are unchanged
DECODE_SOURCES = ("decode_mma.cuh", "decode.cu", "decode_verify.cu", "pa_device.cuh")


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

    launches_per_step = 2 + (1 if st.workspace is not None else 0) + (1 if st.R else 0)
    for _ in range(max(args.warmup, 3)):
        st.step()
    torch.cuda.synchronize(dev)

    # ---- device-timed region: inputs resident in HBM ---------------------
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)] if st.R else [None] * args.steps
    for a, b in ev:            # torch creates the CUDA event at its first record
        a.record(stream)
        b.record(stream)
    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # A pool that fits in L2 twice over would be read from L2 in steady state:
    # then every timed step is preceded by a write of a 2 x L2 buffer, outside
    # the step's own events, and the step time is the mean of those events.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    pool_bytes = st.k_cache.numel() * st.k_cache.element_size() * 2
    flush = None
    if pool_bytes < 2 * l2_bytes:
        flush = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)] if flush is not None else None
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    phys = int(vis[local_rank]) if len(vis) > local_rank and vis[local_rank].strip().isdigit() else local_rank
    clocks = ClockSampler(phys)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.start()
    time.sleep(0.3)   # let the sampler start before the timed region
    t_start.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
            sev[i][0].record(stream)
        pa.pa_set_profile_events(*ev[i])
        st.step(prefill_events=pev[i])
        if flush is not None:
            sev[i][1].record(stream)
    t_stop.record(stream)
    torch.cuda.synchronize(dev)
    pa.pa_set_profile_events(None, None)
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    assert pa.pa_get_device_error() == 0
    ms_total = (t_start.elapsed_time(t_stop) if flush is None else
                sum(a.elapsed_time(b) for a, b in sev))
    decode_ms = [a.elapsed_time(b) for a, b in ev]
    prefill_ms = [a.elapsed_time(b) for a, b in pev] if st.R else None

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
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
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
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(e2e_steps)]
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
    kv_logical = st.kv_bytes_logical()
    value = whole_job_gbs(kv_unique, world, ms_step)
    peak, peak_kind = _peaks()
    # algorithmic bytes of the main decode kernel per launch: the unique K/V
    # bytes plus q, the output/partials are < 0.5% and not counted
    achieved = kv_unique / (dec_ms * 1e-3) / 1e9
    src = _src_hash(DECODE_SOURCES)
    tr = NCU_TRAFFIC.get((wl.name, B, src))
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 K/V, f16 products" if wl.cache_dtype is not None else
                  {"torch.bfloat16": "bf16", "torch.float16": "f16", "torch.float32": "f32"}[str(wl.dtype)]),
        "data": "synthetic (seeded N(0,1) K/V/Q, random block scatter)",
        "config": {"workload": wl.name, "batch": B, "n_q_heads": wl.n_q_heads,
                   "n_kv_heads": wl.n_kv_heads, "head_dim": wl.head_dim,
                   "block_size": wl.block_size, "num_blocks": st.num_blocks,
                   "prefill_requests": st.R, "q_per_seq": wl.q_per_seq,
                   "parallelism": f"replicas x{world}",
                   "l2": (f"inputs larger than L2 ({pool_bytes / 1e9:.2f} GB pool, "
                          f"{kv_unique / 1e9:.2f} GB of K/V read per step); no flush"
                          if flush is None else
                          f"L2 flushed before every timed step (a {2 * l2_bytes >> 20} MiB write, "
                          "outside the step's events); the pool "
                          f"({pool_bytes / 1e6:.0f} MB) would fit in L2")},
        "decode_tokens_per_s": world * B * wl.q_per_seq / (ms_step * 1e-3),
        "steps_per_s": 1e3 / ms_step,
        "pct_of_hbm_peak": 100.0 * value / world / peak,
        "kv_bytes_unique_per_step": kv_unique, "kv_bytes_logical_per_step": kv_logical,
        "decode_kernel_ms": dec_ms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": tr,
                     "kernel": "decode_mma_kernel", "peak_source": f"hbm_gbs ({peak_kind})"},
        "e2e": {"value": whole_job_gbs(kv_unique, world, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": e2e_mode},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if st.R:
        # inside the step the prefill shares SMs with the decode launched beside
        # it, so its roofline is taken from the kernel alone: the same call,
        # timed with events on its own, after the step's timed region
        alone = []
        for i in range(max(20, min(args.steps, 100)) + 3):
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            pa.pa_prefill_chunk(st.p_out, st.p_q_dev, st.k_cache, st.v_cache, st.p_block_tables,
                                st.query_start_loc, st.p_context_lens, int(st.p_chunk.max()),
                                wl.scale, wl.block_size, stream=stream, **st.kv_scales)
            b_.record(stream)
            if i >= 3:
                alone.append((a_, b_))
        torch.cuda.synchronize(dev)
        pf_ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in alone)
        flops = st.prefill_flops()
        tf = _peaks_tensor()
        line["prefill_flops_per_step"] = flops
        line["prefill_kernel_ms"] = pf_ms
        line["prefill_kernel_ms_in_step"] = statistics.mean(prefill_ms)
        line["roofline_prefill"] = {
            "bound": "tensor", "achieved": flops / (pf_ms * 1e-3) / 1e12, "peak": tf[0],
            "unit": "TFLOP/s", "frac": flops / (pf_ms * 1e-3) / 1e12 / tf[0], "traffic": None,
            "kernel": "prefill_tc_kernel", "peak_source": tf[1],
            "timing": "kernel alone (in the step it overlaps the decode)"}
        line["prefill_tokens_per_s"] = world * int(st.p_chunk.sum()) / (ms_step * 1e-3)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, t, desc, threads, _ = oracle_sample(wl.name, None, args.cpu_seconds)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": desc, "seconds": t}
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
