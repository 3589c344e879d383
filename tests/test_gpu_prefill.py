"""GPU parity of chunked prefill over paged context against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import inputs
from paged_kv_cache_25_gb300.step import PagedStep
from tests.helpers import TOL, check_low_precision, half_ulp, max_err, oracle_prefill_all

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_25_gb300 import build
    build.build()
    assert pa.pa_get_device_error() == 0


def _run_case(seed, specs, n_q, n_kv, d, bs, dtype, out_dtype=torch.float32):
    """specs: list of (cached tokens, chunk).  Writes the context and the chunk
    through pa_reshape_and_cache, runs pa_prefill_chunk, returns (out, ref)."""
    rng = np.random.default_rng(seed)
    R = len(specs)
    lens = [c + n for c, n in specs]
    nb = sum(-(-L // bs) for L in lens) + 5
    order = rng.permutation(nb).astype(np.int32)
    alloc = pa.Allocator(nb, order)
    mb = max(-(-L // bs) for L in lens)
    tables = alloc.build_tables(lens, mb, bs)
    g = torch.Generator().manual_seed(seed)
    ks = [torch.randn(L, n_kv, d, generator=g).to(dtype) for L in lens]
    vs = [torch.randn(L, n_kv, d, generator=g).to(dtype) for L in lens]
    qs = [torch.randn(n, n_q, d, generator=g).to(dtype) for _, n in specs]
    kc = torch.full((nb, n_kv, bs, d), float("nan"), dtype=dtype, device="cuda")
    vc = kc.clone()
    seq = np.concatenate([np.full(L, r, np.int32) for r, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    slots = torch.from_numpy(pa.pa_slot_mapping(tables, bs, seq, pos)).cuda()
    pa.pa_reshape_and_cache(torch.cat(ks).cuda(), torch.cat(vs).cuda(), kc, vc, slots)
    qsl = np.zeros(R + 1, np.int32)
    qsl[1:] = np.cumsum([n for _, n in specs])
    out = torch.full((int(qsl[-1]), n_q, d), float("nan"), dtype=out_dtype, device="cuda")
    pa.pa_prefill_chunk(out, torch.cat(qs).cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                        torch.from_numpy(qsl).cuda(),
                        torch.tensor(lens, dtype=torch.int32, device="cuda"),
                        max(n for _, n in specs), 1.0 / np.sqrt(d), bs)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    scale = float(np.float32(1.0 / np.sqrt(d)))
    ref = np.concatenate(oracle.prefill(qs, ks, vs, scale))
    return out, ref


CASES = [
    # seed, specs (ctx, chunk), n_q, n_kv, d, bs, dtype
    (1, [(0, 37)], 4, 4, 64, 16, torch.bfloat16),                         # plain causal prefill
    (2, [(0, 200), (100, 1), (33, 47)], 32, 8, 128, 16, torch.bfloat16),  # ragged, several tiles
    (3, [(500, 64), (0, 16), (16, 16)], 8, 1, 64, 32, torch.float16),     # MQA g=8
    (4, [(1000, 130)], 40, 40, 128, 16, torch.float16),                   # MHA
    (5, [(47, 200), (1, 3)], 12, 4, 128, 32, torch.bfloat16),             # g=3, rows straddle
    # CTAs go longest request first: equal context lengths (ties by index)
    (6, [(100, 20), (290, 50), (100, 20), (0, 120), (339, 1)], 8, 2, 128, 16, torch.bfloat16),
    # more requests than the kernel ranks (64): call order
    (7, [(int(c), int(n)) for c, n in zip(np.random.default_rng(7).integers(0, 60, 70),
                                          np.random.default_rng(8).integers(1, 10, 70))],
     4, 2, 64, 16, torch.float16),
]


@pytest.mark.parametrize("case", CASES, ids=[f"p{c[0]}" for c in CASES])
def test_prefill_small_all_rows(case):
    seed, specs, n_q, n_kv, d, bs, dtype = case
    out, ref = _run_case(seed, specs, n_q, n_kv, d, bs, dtype)
    err = max_err(out, ref)
    assert err <= TOL[dtype], err


def test_prefill_bf16_output():
    out, ref = _run_case(9, [(300, 100), (0, 50)], 32, 8, 128, 16, torch.bfloat16,
                         out_dtype=torch.bfloat16)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2e-3 + half_ulp(ref, torch.bfloat16))


def test_prefill_chunk_of_one_matches_decode():
    d, bs, n_q, n_kv = 128, 16, 32, 8
    out, ref = _run_case(11, [(77, 1)], n_q, n_kv, d, bs, torch.bfloat16)
    assert max_err(out, ref) <= 2e-3


def test_prefill_mixed_workload_all_rows():
    """The mixed step's four 512-row chunks over 1024-8192 cached tokens: every
    output row of every head, stored in fp32 (<= 2e-3) and in bf16 (<= 2e-3 +
    half an ulp), against the oracle's chunked prefill."""
    wl = inputs.get("mixed-llama3-8b-bf16")
    st = PagedStep(wl, out_dtype=torch.float32, prefill_out_dtype=torch.float32)
    st.step()
    out_lp = torch.full(tuple(st.p_out.shape), float("nan"), dtype=wl.dtype, device="cuda")
    pa.pa_prefill_chunk(out_lp, st.p_q_dev, st.k_cache, st.v_cache, st.p_block_tables,
                        st.query_start_loc, st.p_context_lens, int(st.p_chunk.max()), wl.scale,
                        wl.block_size)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ref = oracle_prefill_all(st)
    assert ref.shape == tuple(st.p_out.shape)
    assert max_err(st.p_out, ref) <= 2e-3
    assert check_low_precision(out_lp, ref, wl.dtype) <= 0.0


def test_prefill_chunk_longer_than_max_query_len_is_flagged():
    """max_query_len sizes the grid; a request whose chunk is longer is reported
    in the device error word instead of silently leaving rows unwritten."""
    d, bs, n_q, n_kv, C = 64, 16, 8, 2, 300
    nb = 5                                          # table entries reuse blocks 0..4
    tables = np.arange(-(-C // bs), dtype=np.int32)[None, :] % nb
    kc = torch.zeros((nb, n_kv, bs, d), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    q = torch.zeros((C, n_q, d), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((C, n_q, d), dtype=torch.float32, device="cuda")
    pa.pa_prefill_chunk(o, q, kc, vc, torch.from_numpy(np.ascontiguousarray(tables)).cuda(),
                        torch.tensor([0, C], dtype=torch.int32, device="cuda"),
                        torch.tensor([C], dtype=torch.int32, device="cuda"), 64, 0.125, bs)
    assert pa.pa_get_device_error() == pa.PA_ERR_OUT_OF_RANGE
    assert pa.pa_get_device_error() == 0


def test_prefill_negative_and_zero_scale():
    """The kernel takes the max on raw scores; a negative scale must flip it."""
    import torch
    for scale in (-0.09, 0.0):
        d, bs, n_q, n_kv = 64, 16, 8, 2
        rng = np.random.default_rng(5)
        L, C = 90, 40
        nb = 10
        alloc = pa.Allocator(nb, rng.permutation(nb).astype(np.int32))
        tables = alloc.build_tables([L], 6, bs)
        g = torch.Generator().manual_seed(3)
        k = torch.randn(L, n_kv, d, generator=g).to(torch.bfloat16)
        v = torch.randn(L, n_kv, d, generator=g).to(torch.bfloat16)
        qq = torch.randn(C, n_q, d, generator=g).to(torch.bfloat16)
        kc = torch.full((nb, n_kv, bs, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        vc = kc.clone()
        slots = torch.from_numpy(pa.pa_slot_mapping(tables, bs, np.zeros(L, np.int32),
                                                    np.arange(L, dtype=np.int32))).cuda()
        pa.pa_reshape_and_cache(k.cuda(), v.cuda(), kc, vc, slots)
        out = torch.empty((C, n_q, d), dtype=torch.float32, device="cuda")
        pa.pa_prefill_chunk(out, qq.cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                            torch.tensor([0, C], dtype=torch.int32, device="cuda"),
                            torch.tensor([L], dtype=torch.int32, device="cuda"), C, scale, bs)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        ref = oracle.prefill([qq], [k], [v], float(np.float32(scale)))[0]
        assert max_err(out, ref) <= 2e-3
