"""GPU parity: cache write (bit-exact) and paged decode (within tolerance)
against the CPU oracle, on seeded inputs of every workload shape, through the
C ABI."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import inputs
from paged_kv_cache_25_gb300.step import PagedStep
from tests.helpers import TOL, check_low_precision, half_ulp, max_err, oracle_decode, oracle_decode_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_25_gb300 import build
    build.build()
    pa.lib()
    assert pa.pa_get_device_error() == 0


def _check_clean():
    assert pa.pa_get_device_error() == 0


def _small(seed, B, n_q, n_kv, d, bs, dtype, lens, std=1.0):
    return inputs.random_case(seed, B, n_q, n_kv, d, bs, dtype, lens, std=std)


# ------------------------------------------------------------------ cache write

@pytest.mark.parametrize("name", ["tiny-fp32", "tinyllama-bf16"])
def test_cache_write_whole_pool_bit_exact(name):
    wl = inputs.get(name)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    _check_clean()
    # oracle: its own allocator from the same seeded free order, its own slots
    dr = inputs.Draws(wl)
    a = oracle.Allocator(st.num_blocks, dr.free_order(st.num_blocks))
    tables = a.build_tables(st.lens, st.max_blocks, wl.block_size)
    assert np.array_equal(tables, st.tables)
    kvs = dr.all_seq_kv(st.lens)
    seq = np.concatenate([np.full(L, s) for s, L in enumerate(st.lens)])
    pos = np.concatenate([np.arange(L) for L in st.lens])
    slots = oracle.slot_mapping(tables, wl.block_size, seq, pos)
    K = torch.cat([k for k, _ in kvs]); V = torch.cat([v for _, v in kvs])
    nan_pool = torch.full(tuple(st.k_cache.shape), float("nan"), dtype=wl.dtype)
    kc, vc = oracle.cache_write(nan_pool, nan_pool, K, V, slots, wl.block_size)
    got_k = st.k_cache.cpu().contiguous().view(torch.uint8).numpy().reshape(-1)
    got_v = st.v_cache.cpu().contiguous().view(torch.uint8).numpy().reshape(-1)
    assert np.array_equal(got_k, kc) and np.array_equal(got_v, vc)


def test_cache_write_skips_negative_and_flags_out_of_range():
    nb, n_kv, bs, d = 4, 2, 16, 64
    kc = torch.full((nb, n_kv, bs, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    k = torch.randn(3, n_kv, d, device="cuda").to(torch.bfloat16)
    v = torch.randn(3, n_kv, d, device="cuda").to(torch.bfloat16)
    slots = torch.tensor([5, -1, 2 * bs + 3], dtype=torch.int64, device="cuda")
    pa.pa_reshape_and_cache(k, v, kc, vc, slots)
    _check_clean()
    assert torch.equal(kc[0, :, 5], k[0]) and torch.equal(vc[2, :, 3], v[2])
    assert int((~torch.isnan(kc.float())).sum()) == 2 * n_kv * d
    bad = torch.tensor([nb * bs], dtype=torch.int64, device="cuda")
    before = kc.clone()
    pa.pa_reshape_and_cache(k[:1], v[:1], kc, vc, bad)
    assert pa.pa_get_device_error() == pa.PA_ERR_OUT_OF_RANGE
    assert torch.equal(kc.view(torch.int16), before.view(torch.int16))
    _check_clean()


# ------------------------------------------------------------------ decode, full

@pytest.mark.parametrize("name", ["tiny-fp32", "tinyllama-bf16"])
def test_decode_all_outputs(name):
    wl = inputs.get(name)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    _check_clean()
    ref = oracle_decode(st)
    err = max_err(st.out, ref)
    assert err <= TOL[wl.dtype], err


CASES = [
    # seed, B, n_q, n_kv, d, bs, dtype, lens
    (1, 5, 8, 8, 128, 16, torch.bfloat16, [1, 15, 16, 17, 1000]),          # MHA, edge lengths
    (2, 4, 32, 8, 128, 16, torch.bfloat16, [513, 512, 511, 2049]),          # partition edges
    (3, 3, 16, 1, 64, 32, torch.float16, [31, 32, 33]),                     # MQA g=16: 2 sub-groups
    (4, 6, 12, 4, 64, 16, torch.bfloat16, [1, 2, 100, 300, 700, 1200]),     # g=3
    (5, 2, 40, 40, 128, 16, torch.float16, [2048, 7]),                      # OPT shape
    (6, 3, 8, 2, 128, 32, torch.bfloat16, [9000, 64, 65]),                  # long, bs 32
    (7, 4, 4, 2, 64, 16, torch.float32, [7, 16, 33, 1500]),                 # fp32 split
    (8, 3, 8, 4, 96, 16, torch.bfloat16, [40, 600, 1]),                     # CUDA-core shape
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{c[0]}" for c in CASES])
def test_decode_edge_shapes(case):
    seed, B, n_q, n_kv, d, bs, dtype, lens = case
    wl = _small(seed, B, n_q, n_kv, d, bs, dtype, lens)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    _check_clean()
    ref = oracle_decode(st)
    err = max_err(st.out, ref)
    assert err <= TOL[dtype], err


def test_decode_1024_token_partitions_all_outputs():
    """A batch large enough for the widest partitions (64 sequences x 8 KV heads
    x 5 partitions of the longest context = 2560 units >= 8 per resident CTA):
    lengths on every 1024-token edge, plus a ragged spread, all outputs checked."""
    edges = [1, 15, 16, 17, 1023, 1024, 1025, 2047, 2048, 2049, 3071, 4096, 4097, 5000]
    rng = np.random.default_rng(77)
    lens = edges + [int(x) for x in rng.integers(1, 5001, size=64 - len(edges))]
    wl = _small(41, 64, 32, 8, 128, 16, torch.bfloat16, lens)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    _check_clean()
    ref = oracle_decode(st)
    err = max_err(st.out, ref)
    assert err <= TOL[torch.bfloat16], err


def test_decode_more_sequences_than_the_prefix_table():
    """2,100 sequences (past the 1,024 whose partition prefix sums fit in shared
    memory): units are numbered per (sequence, partition index) instead; every
    output checked, lengths spanning one to several partitions."""
    rng = np.random.default_rng(55)
    lens = [int(x) for x in rng.integers(1, 3001, size=2100)]
    lens[:7] = [1, 1023, 1024, 1025, 2048, 2049, 3000]
    wl = _small(56, 2100, 8, 2, 64, 16, torch.bfloat16, lens)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    _check_clean()
    ref = oracle_decode(st)
    err = max_err(st.out, ref)
    assert err <= TOL[torch.bfloat16], err


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_decode_low_precision_output(dtype):
    wl = _small(21, 4, 32, 8, 128, 16, dtype, [20, 300, 1024, 3000])
    st = PagedStep(wl, out_dtype=dtype)
    st.step()
    torch.cuda.synchronize()
    _check_clean()
    ref = oracle_decode(st)
    got = st.out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= TOL[dtype] + half_ulp(ref, dtype))


def test_decode_permutation_invariance_bit_identical():
    """Any scatter of the same logical rows gives the same bits: the kernel's
    reduction order depends only on logical positions."""
    outs = []
    for seed in (31, 32, 33):
        wl = _small(30, 4, 8, 2, 128, 16, torch.bfloat16, [50, 700, 1300, 17])
        st = PagedStep(wl, out_dtype=torch.float32)
        # same draws except the free-queue order
        alt = inputs.Draws(wl, seed=seed)
        st2_order = alt.free_order(st.num_blocks)
        st.alloc = pa.Allocator(st.num_blocks, st2_order)
        st.tables = st.alloc.build_tables(st.lens, st.max_blocks, wl.block_size)
        st.k_cache.fill_(float("nan")); st.v_cache.fill_(float("nan"))
        st._prefill_context(1 << 16)
        st.block_tables = torch.from_numpy(st.tables).cuda()
        seq = np.arange(wl.batch, dtype=np.int32)
        st.new_slots = torch.from_numpy(pa.pa_slot_mapping(st.tables, wl.block_size, seq,
                                                           (st.lens - 1).astype(np.int32))).cuda()
        st.step()
        torch.cuda.synchronize()
        outs.append(st.out.cpu())
    _check_clean()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_decode_split_invariance_batch_of_one_vs_many():
    """The partition size follows the batch size; results agree within tolerance."""
    wl = _small(40, 6, 32, 8, 128, 16, torch.bfloat16, [4000, 100, 2500, 900, 3333, 64])
    big = PagedStep(wl, out_dtype=torch.float32)
    big.step()
    one = _small(40, 1, 32, 8, 128, 16, torch.bfloat16, [4000])
    small = PagedStep(one, out_dtype=torch.float32)
    small.step()
    torch.cuda.synchronize()
    _check_clean()
    assert float((big.out[0] - small.out[0]).abs().max()) <= 2e-3
    ref = oracle_decode(small)
    assert max_err(small.out, ref) <= 2e-3


def test_decode_gqa_equals_mha_with_repeated_kv_heads():
    g = 4
    wl = _small(50, 3, 8, 2, 64, 16, torch.bfloat16, [100, 33, 700])
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    kc = st.k_cache.repeat_interleave(g, dim=1).contiguous()
    vc = st.v_cache.repeat_interleave(g, dim=1).contiguous()
    out = torch.empty_like(st.out)
    ws = pa.pa_decode_workspace_size(wl.batch, 8, 8, 64, 16, st.max_blocks * 16)
    w = torch.empty(max(ws, 1), dtype=torch.uint8, device="cuda")
    pa.pa_decode(out, st.q, kc, vc, st.block_tables, st.context_lens, wl.scale, 16, w)
    torch.cuda.synchronize()
    _check_clean()
    assert float((out - st.out).abs().max()) <= 2e-3


def test_decode_out_of_range_block_id_is_flagged_not_read():
    wl = _small(60, 2, 8, 2, 128, 16, torch.bfloat16, [40, 70])
    st = PagedStep(wl, out_dtype=torch.float32)
    bt = st.block_tables.clone()
    bt[1, 2] = st.num_blocks + 7
    pa.pa_decode(st.out, st.q, st.k_cache, st.v_cache, bt, st.context_lens, wl.scale, 16,
                 st.workspace)
    assert pa.pa_get_device_error() == pa.PA_ERR_OUT_OF_RANGE
    bt[1, 2] = -3
    pa.pa_decode(st.out, st.q, st.k_cache, st.v_cache, bt, st.context_lens, wl.scale, 16,
                 st.workspace)
    assert pa.pa_get_device_error() == pa.PA_ERR_OUT_OF_RANGE
    _check_clean()


def test_decode_host_checks_launch_nothing():
    wl = _small(61, 2, 8, 2, 128, 16, torch.bfloat16, [4000, 70])
    st = PagedStep(wl, out_dtype=torch.float32)
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(st.out, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens,
                     wl.scale, 16, None)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode(st.out, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens,
                     wl.scale, 32, st.workspace)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    # zero sequences: a no-op
    pa.pa_decode(st.out[:0], st.q[:0], st.k_cache, st.v_cache, st.block_tables[:0],
                 st.context_lens[:0], wl.scale, 16, st.workspace)
    _check_clean()


# ------------------------------------------------------------------ full-size workloads

@pytest.mark.parametrize("name", ["llama3-8b-bf16", "opt13b-fp16", "mixed-llama3-8b-bf16"])
def test_decode_full_size_all_outputs(name):
    """Every output of the full-size decode batch (all sequences x all query
    heads x all head-dim elements), once stored in fp32 (<= 2e-3) and once in
    the workload's own dtype, as the bench times it (<= 2e-3 + half an ulp)."""
    wl = inputs.get(name)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    out_lp = torch.full(tuple(st.out.shape), float("nan"), dtype=wl.dtype, device="cuda")
    pa.pa_decode(out_lp, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens,
                 wl.scale, wl.block_size, st.workspace)
    torch.cuda.synchronize()
    _check_clean()
    ref = oracle_decode_all(st)
    assert ref.shape == tuple(st.out.shape)
    err = max_err(st.out, ref)
    assert err <= TOL[wl.dtype], err
    assert check_low_precision(out_lp, ref, wl.dtype) <= 0.0
