"""Multi-query decode (verification of drafted tokens) against the oracle's
chunked prefill with chunks of q_per_seq rows: query i of sequence s sits at
context_lens[s] - q_per_seq + i and sees the keys up to it."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import inputs
from tests.helpers import TOL, check_low_precision, max_err, oracle_decode_all, stored_kv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_25_gb300 import build
    build.build()
    assert pa.pa_get_device_error() == 0


class Case:
    """Pools holding every sequence's K/V (NaN elsewhere), tables, lengths, q."""

    def __init__(self, seed, B, n_q, n_kv, d, bs, dtype, lens, nq, cache_dtype=None, kv_scale=1.0):
        wl = inputs.random_case(seed, B, n_q, n_kv, d, bs, dtype, lens, cache_dtype=cache_dtype,
                                kv_scale=kv_scale)
        self.wl, self.nq = wl, nq
        dr = inputs.Draws(wl)
        self.lens = np.array(lens, np.int32)
        mb = -(-int(self.lens.max()) // bs)
        nb = int(1.5 * sum(-(-int(x) // bs) for x in lens)) + 4
        alloc = pa.Allocator(nb, dr.free_order(nb))
        self.tables = alloc.build_tables(self.lens, mb, bs)
        self.kv = [dr.seq_kv(s, int(self.lens[s])) for s in range(B)]
        pool_dt = wl.pool_dtype
        shape = (nb, n_kv, bs, d)
        if pool_dt == torch.float8_e4m3fn:
            self.kc = torch.full(shape, 0x7F, dtype=torch.uint8, device="cuda").view(pool_dt)
            self.vc = torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8,
                                 device="cuda").view(pool_dt)
            self.scales = {"k_scale": kv_scale, "v_scale": kv_scale}
        else:
            self.kc = torch.full(shape, float("nan"), dtype=dtype, device="cuda")
            self.vc = torch.full_like(self.kc, float("nan"))
            self.scales = {}
        seq = np.concatenate([np.full(int(L), s, np.int32) for s, L in enumerate(self.lens)])
        pos = np.concatenate([np.arange(int(L), dtype=np.int32) for L in self.lens])
        slots = torch.from_numpy(pa.pa_slot_mapping(self.tables, bs, seq, pos)).cuda()
        k = torch.cat([x[0] for x in self.kv]).cuda()
        v = torch.cat([x[1] for x in self.kv]).cuda()
        if self.scales:
            pa.pa_reshape_and_cache_quant(k, v, self.kc, self.vc, slots, **self.scales)
        else:
            pa.pa_reshape_and_cache(k, v, self.kc, self.vc, slots)
        g = torch.Generator().manual_seed(seed + 7)
        self.q = torch.randn(B, nq, n_q, d, generator=g).to(dtype)
        self.max_ctx = mb * bs

    def run(self, out_dtype=torch.float32, workspace=None):
        wl = self.wl
        out = torch.full((wl.batch, self.nq, wl.n_q_heads, wl.head_dim), float("nan"),
                         dtype=out_dtype, device="cuda")
        need = pa.pa_decode_verify_workspace_size(wl.batch, self.nq, wl.n_q_heads, wl.n_kv_heads,
                                                  wl.head_dim, wl.block_size, self.max_ctx)
        ws = workspace if workspace is not None else torch.empty(need, dtype=torch.uint8,
                                                                 device="cuda")
        pa.pa_decode_verify(out, self.q.cuda(), self.kc, self.vc,
                            torch.from_numpy(self.tables).cuda(),
                            torch.from_numpy(self.lens).cuda(), wl.scale, wl.block_size, ws,
                            **self.scales)
        return out

    def oracle(self):
        kv = [stored_kv(self.wl, k, v) for k, v in self.kv]
        outs = oracle.prefill([self.q[s] for s in range(self.wl.batch)], [x[0] for x in kv],
                              [x[1] for x in kv], self.wl.scale)
        return np.stack(outs)


CASES = [
    # seed, B, n_q, n_kv, d, bs, dtype, lens, q_per_seq
    (1, 4, 32, 8, 128, 16, torch.bfloat16, [4, 17, 300, 2100], 4),        # g 4 x 4 rows: 2 sub-groups
    (2, 3, 16, 2, 128, 16, torch.bfloat16, [2, 129, 130], 2),             # g 8 x 2: 2 sub-groups
    (3, 5, 8, 8, 64, 32, torch.float16, [8, 9, 64, 700, 1500], 8),        # MHA, 8 rows per head
    (4, 3, 12, 4, 128, 16, torch.bfloat16, [5, 131, 1000], 5),            # g 3 x 5 = 15 rows
    (5, 2, 32, 8, 128, 32, torch.bfloat16, [16, 4096], 16),               # 16 drafts: 8 sub-groups
    (6, 4, 4, 1, 64, 16, torch.float16, [1, 3, 258, 1029], 1),            # one row: plain decode
    (7, 3, 16, 2, 64, 32, torch.float16, [12, 300, 1500], 3),             # 24 rows: 16 + 8, d 64
]


@pytest.mark.parametrize("case", CASES, ids=[f"v{c[0]}" for c in CASES])
def test_verify_matches_oracle(case):
    seed, B, n_q, n_kv, d, bs, dtype, lens, nq = case
    c = Case(seed, B, n_q, n_kv, d, bs, dtype, lens, nq)
    out = c.run()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert max_err(out, c.oracle()) <= TOL[dtype]


def test_verify_last_partition_shorter_than_the_queries():
    """128-token partitions (small batch) with lengths 129/130 and 4 queries:
    the last partition holds 1-2 keys, invisible to the first queries, whose
    partial results there must be empty (not NaN)."""
    c = Case(11, 2, 8, 2, 128, 16, torch.bfloat16, [129, 130], 4)
    out = c.run()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.isfinite(out).all()
    assert max_err(out, c.oracle()) <= TOL[torch.bfloat16]


def test_verify_large_batch_1024_token_partitions():
    rng = np.random.default_rng(12)
    edges = [4, 1024, 1025, 1026, 1027, 1028, 2049, 3000]
    lens = edges + [int(x) for x in rng.integers(4, 4097, size=64 - len(edges))]
    c = Case(12, 64, 32, 8, 128, 16, torch.bfloat16, lens, 4)
    out = c.run()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert max_err(out, c.oracle()) <= TOL[torch.bfloat16]


def test_verify_fp8_pool():
    c = Case(13, 6, 32, 8, 128, 16, torch.bfloat16, [4, 40, 600, 1300, 2500, 4100], 4,
             cache_dtype=torch.float8_e4m3fn, kv_scale=1.0 / 64)
    out = c.run()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert max_err(out, c.oracle()) <= TOL[torch.bfloat16]


def test_verify_one_query_is_bit_identical_to_decode():
    c = Case(14, 5, 32, 8, 128, 16, torch.bfloat16, [1, 33, 700, 1500, 4000], 1)
    out = c.run()
    wl = c.wl
    out2 = torch.empty(wl.batch, wl.n_q_heads, wl.head_dim, dtype=torch.float32, device="cuda")
    ws = torch.empty(pa.pa_decode_workspace_size(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                                                 wl.block_size, c.max_ctx),
                     dtype=torch.uint8, device="cuda")
    pa.pa_decode(out2, c.q[:, 0].contiguous().cuda(), c.kc, c.vc, torch.from_numpy(c.tables).cuda(),
                 torch.from_numpy(c.lens).cuda(), wl.scale, wl.block_size, ws)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.equal(out[:, 0], out2)


def test_verify_sequence_shorter_than_its_queries_is_flagged():
    c = Case(15, 2, 8, 2, 64, 16, torch.bfloat16, [3, 50], 4)   # sequence 0: 3 keys, 4 queries
    out = c.run()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == pa.PA_ERR_OUT_OF_RANGE
    assert torch.isnan(out[0]).all()                  # not written
    k1, v1 = c.kv[1]                                   # sequence 1 is still right
    ref = oracle.prefill([c.q[1]], [k1], [v1], c.wl.scale)[0]
    assert max_err(out[1], ref) <= TOL[torch.bfloat16]
    assert pa.pa_get_device_error() == 0


def test_verify_host_checks():
    c = Case(16, 2, 8, 2, 64, 16, torch.bfloat16, [20, 50], 2)
    wl = c.wl
    out = torch.empty(2, 2, 8, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(pa.PAError):                    # workspace too small
        pa.pa_decode_verify(out, c.q.cuda(), c.kc, c.vc, torch.from_numpy(c.tables).cuda(),
                            torch.from_numpy(c.lens).cuda(), wl.scale, wl.block_size,
                            torch.empty(16, dtype=torch.uint8, device="cuda"))
    q17 = torch.zeros(2, 17, 8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PAError):                    # more than 16 rows per sequence
        pa.pa_decode_verify(torch.empty(2, 17, 8, 64, device="cuda"), q17, c.kc, c.vc,
                            torch.from_numpy(c.tables).cuda(), torch.from_numpy(c.lens).cuda(),
                            wl.scale, wl.block_size,
                            torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert pa.pa_get_device_error() == 0


def test_verify_full_size_workload_all_outputs():
    """The Llama-3-8B batch with 4 query rows per sequence, as the bench runs
    it (cache write of the 4 new rows, then the multi-query decode): every
    output, in fp32 and in bf16."""
    from paged_kv_cache_25_gb300.step import PagedStep
    wl = inputs.get("llama3-8b-bf16-verify4")
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    out_lp = torch.full(tuple(st.out.shape), float("nan"), dtype=wl.dtype, device="cuda")
    pa.pa_decode_verify(out_lp, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens,
                        wl.scale, wl.block_size, st.workspace)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ref = oracle_decode_all(st)
    assert ref.shape == tuple(st.out.shape)
    assert max_err(st.out, ref) <= TOL[wl.dtype]
    assert check_low_precision(out_lp, ref, wl.dtype) <= 0.0
