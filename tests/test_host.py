"""CPU-only checks of the C-ABI library: it builds, loads and exports every
symbol include/pa.h declares; its host allocator, page tables, slot mapping and
sizing agree bit for bit with the oracle; its host-side argument checks reject
bad calls before touching the GPU."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import build, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    return pa.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "pa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert len(names) >= 20
    h = C.CDLL(build.LIB)
    for n in names:
        assert hasattr(h, n), n
    assert set(names) == set(pa.EXPORTED)


def test_built_for_sm_103a_only():
    # the build asks nvcc for exactly one target
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_tables_and_slots_match_oracle_allocator(name):
    wl = inputs.get(name)
    dr = inputs.Draws(wl)
    lens, sharers = dr.decode_lens(), dr.sharers()
    bs = wl.block_size
    prefix = wl.shared_prefix_tokens if sharers.any() else 0
    nb = 200_000 if wl.pool != "fixed" else int(wl.pool_arg)
    mb = -(-int(lens.max()) // bs)
    order = dr.free_order(nb)
    ours = pa.Allocator(nb, order)
    ref = oracle.Allocator(nb, order)
    t1 = ours.build_tables(lens, mb, bs, sharers, prefix)
    t2 = ref.build_tables(lens, mb, bs, sharers, prefix)
    assert np.array_equal(t1, t2)
    assert ours.num_free() == ref.num_free()
    if prefix:
        pid = int(t1[np.nonzero(sharers)[0][0], 0])
        assert ours.refcount(pid) == ref.refcount(pid) == int(sharers.sum())
    seq = np.repeat(np.arange(len(lens), dtype=np.int32), 3)
    pos = np.stack([np.zeros_like(lens), lens // 2, lens - 1], 1).reshape(-1).astype(np.int32)
    assert np.array_equal(pa.pa_slot_mapping(t1, bs, seq, pos), oracle.slot_mapping(t2, bs, seq, pos))


def test_allocator_free_and_share_match_oracle():
    order = np.random.default_rng(3).permutation(50).astype(np.int32)
    a, b = pa.Allocator(50, order), oracle.Allocator(50, order)
    x, y = a.blocks(20), b.take(20)
    assert np.array_equal(x, y)
    a.share(x[:5]); b.share(y[:5])
    a.free(x); b.release(y)
    assert a.num_free() == b.num_free() == 45
    assert np.array_equal(a.blocks(45), b.take(45))
    assert a.blocks(1) is None and b.take(1) is None


def test_allocator_rejects_bad_order_and_overflow():
    with pytest.raises(pa.PAError):
        pa.Allocator(4, [0, 1, 1, 2])
    a = pa.Allocator(4)
    with pytest.raises(pa.PAError):
        a.build_tables([40, 40], 3, 16)       # 6 blocks from a pool of 4
    assert a.num_free() == 4                   # nothing taken on failure
    with pytest.raises(pa.PAError):
        pa.pa_slot_mapping(np.array([[0, -1]], np.int32), 16, [0], [20])


def test_sizing_matches_oracle_and_pages():
    for args in [(40, 40, 128, 2), (32, 8, 128, 2), (48, 8, 128, 2), (22, 4, 64, 2), (1, 8, 128, 1)]:
        assert pa.pa_kv_bytes_per_token(*args) == oracle.kv_bytes_per_token(*args)
    assert pa.pa_pool_blocks(54 << 30, 16, 131072) == 27648
    assert pa.pa_pool_blocks(60_000_000_000, 32, 4096) == oracle.pool_blocks(60_000_000_000, 32, 4096)


class _Fake:
    """Stands in for a device tensor in calls that must fail host checks."""

    def __init__(self, ptr, shape, dtype):
        self.ptr, self.shape, self.dtype = ptr, shape, dtype


def _raw_decode(out=0x1000, q=0x2000, kc=0x3000, vc=0x4000, bt=0x5000, cl=0x6000, nb=64, bs=16,
                n_kv=8, d=128, dt=2, mb=16, B=4, n_q=32, scale=0.1, blk=16, ws=None, ws_bytes=0):
    desc = pa._Desc(nb, bs, n_kv, d, dt)
    return pa.lib().pa_decode(out, dt, q, kc, vc, C.byref(desc), bt, mb, cl, B, n_q, scale, blk,
                              ws, ws_bytes, None)


def test_decode_host_validation_before_any_launch():
    assert _raw_decode(out=None) == pa.PA_ERR_INVALID_ARG
    assert _raw_decode(q=0x2004) == pa.PA_ERR_INVALID_ARG              # misaligned
    assert _raw_decode(n_q=30) == pa.PA_ERR_INVALID_ARG                # not a multiple of n_kv
    assert _raw_decode(blk=32) == pa.PA_ERR_INVALID_ARG                # != cache block size
    assert _raw_decode(bs=8, blk=8) == pa.PA_ERR_UNSUPPORTED
    assert _raw_decode(d=80) == pa.PA_ERR_UNSUPPORTED
    assert _raw_decode(scale=float("inf")) == pa.PA_ERR_INVALID_ARG
    assert _raw_decode(dt=7) == pa.PA_ERR_INVALID_ARG
    # a long table needs a workspace: none given
    assert _raw_decode(mb=4096 // 16 * 4) == pa.PA_ERR_WORKSPACE
    need = pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 4096 * 4)
    assert need > 0
    assert _raw_decode(mb=1024, ws=0x10000, ws_bytes=need - 1) == pa.PA_ERR_WORKSPACE
    assert _raw_decode(mb=1024, ws=0x10010, ws_bytes=need) == pa.PA_ERR_INVALID_ARG  # alignment
    assert _raw_decode(B=0) == pa.PA_OK                                  # nothing to do
    assert _raw_decode(n_q=30) == pa.PA_ERR_INVALID_ARG
    assert "n_q_heads" in pa.lib().pa_last_error_message().decode()


def test_workspace_size_rules():
    # a single partition needs only the 256-byte control area
    assert pa.pa_decode_workspace_size(256, 32, 8, 128, 16, 16) == 256
    w = pa.pa_decode_workspace_size(256, 32, 8, 128, 16, 4096)
    assert w >= 256 * 32 * 4 * 128 * 4      # at least 4 partitions of fp32 partial outputs
    assert pa.pa_decode_workspace_size(0, 32, 8, 128, 16, 4096) == 0
    # partitions shrink (1024 -> 256 tokens) when a batch offers little work:
    # 4 sequences x 8 KV heads x 16 partitions = 512 units >= 300
    small = pa.pa_decode_workspace_size(4, 32, 8, 128, 16, 4096)
    assert small >= 256 + 4 * 32 * 16 * 128 * 4
    assert small < 256 + 4 * 32 * 32 * 128 * 4


def test_cache_write_host_validation():
    desc = pa._Desc(64, 16, 8, 128, 2)
    f = pa.lib().pa_reshape_and_cache
    assert f(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0, C.byref(desc), None) == pa.PA_OK
    assert f(0x1000, 0x2000, 0x3000, 0x4000, 0x5004, 3, C.byref(desc), None) == pa.PA_ERR_INVALID_ARG
    assert f(0x1008, 0x2000, 0x3000, 0x4000, 0x5000, 3, C.byref(desc), None) == pa.PA_ERR_INVALID_ARG
    assert f(None, 0x2000, 0x3000, 0x4000, 0x5000, 3, C.byref(desc), None) == pa.PA_ERR_INVALID_ARG
    assert f(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, -1, C.byref(desc), None) == pa.PA_ERR_INVALID_ARG


def test_prefill_host_validation():
    desc = pa._Desc(64, 16, 8, 128, 0)  # fp32 pool: prefill is bf16/fp16/FP8 only
    f = pa.lib().pa_prefill_chunk
    args = [0x1000, 0, 0x2000, 0x3000, 0x4000, C.byref(desc), 0x5000, 8, 0x6000, 0x7000, 2, 16, 32,
            0.1, 16, None, 0, None]
    assert f(*args) == pa.PA_ERR_UNSUPPORTED
    desc2 = pa._Desc(64, 16, 8, 128, 2)
    args[5] = C.byref(desc2)
    args[12] = 30
    assert f(*args) == pa.PA_ERR_INVALID_ARG
    args[12] = 32
    args[10] = 0
    assert f(*args) == pa.PA_OK                                        # no requests


def test_prefill_fp8_host_validation():
    """FP8 pools need finite positive scales and a bf16/fp16 activation type;
    head sizes outside {64, 128} are refused before any launch."""
    f = pa.lib().pa_prefill_chunk

    def call(desc):
        return f(0x1000, 0, 0x2000, 0x3000, 0x4000, C.byref(desc), 0x5000, 8, 0x6000, 0x7000, 2,
                 16, 32, 0.1, 16, None, 0, None)

    fp8 = pa.PA_FP8_E4M3
    assert call(pa._Desc(64, 16, 8, 128, fp8, 0.0, 0.0, pa.PA_BF16)) == pa.PA_ERR_INVALID_ARG
    assert call(pa._Desc(64, 16, 8, 128, fp8, 0.5, float("nan"), pa.PA_BF16)) == pa.PA_ERR_INVALID_ARG
    assert call(pa._Desc(64, 16, 8, 128, fp8, 0.5, 0.5, -1)) == pa.PA_ERR_INVALID_ARG
    assert call(pa._Desc(64, 16, 8, 128, fp8, 0.5, 0.5, pa.PA_F32)) == pa.PA_ERR_INVALID_ARG
    assert call(pa._Desc(64, 16, 8, 96, fp8, 0.5, 0.5, pa.PA_BF16)) == pa.PA_ERR_UNSUPPORTED
    assert "FP8" in pa.lib().pa_last_error_message().decode() or \
        "head_dim" in pa.lib().pa_last_error_message().decode()


def test_stored_dram_traffic_matches_the_kernel_sources():
    """The bench reports ncu DRAM bytes only for the kernel sources they were
    captured on (keyed by a hash of those sources): the headline and FP8
    decode batches and both mixed steps' prefills have a capture of the
    sources as they stand, and each capture is at least the unique bytes."""
    import importlib.util
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dh = bench._src_hash(bench.DECODE_SOURCES)
    ph = bench._src_hash(bench.PREFILL_SOURCES)
    for name in ("llama3-8b-bf16", "llama3-8b-fp8"):
        traffic, unique = bench.NCU_TRAFFIC[(name, dh)][:2]
        assert unique <= traffic <= 1.05 * unique
    for name in ("mixed-llama3-8b-bf16", "mixed-llama3-8b-fp8"):
        assert (name, ph) in bench.NCU_PREFILL_TRAFFIC
