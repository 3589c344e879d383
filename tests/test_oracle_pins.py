"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: figures the
pages print (tests/golden, cited), closed forms, library routines on special
cases (torch's scaled_dot_product_attention in fp64), invariants, and brute
force on tiny inputs.  The set is chosen so that a plausible slip (a dropped
scale, a wrong sign, a wrong GQA index, an off-by-one causal bound, a swapped
K/V operand, a wrong block offset) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_25_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _golden(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- sizes

def test_kv_bytes_per_token_worked_figures(golden_dir):
    g = _golden(golden_dir, "kv_sizes.json")
    for row in g["per_token"]:
        got = oracle.kv_bytes_per_token(row["n_layers"], row["n_kv_heads"], row["head_dim"],
                                        row["elem_bytes"])
        if row["kind"] == "exact":
            assert got == row["bytes"], row["cite"]
        else:
            assert abs(got - row["bytes"]) <= row["rel_tol"] * row["bytes"], row["cite"]


def test_kv_bytes_per_sequence_worked_figures(golden_dir):
    g = _golden(golden_dir, "kv_sizes.json")
    for row in g["per_sequence"]:
        got = oracle.kv_bytes_per_token(row["n_layers"], row["n_kv_heads"], row["head_dim"],
                                        row["elem_bytes"]) * row["tokens"]
        if row["kind"] == "exact":
            assert got == row["bytes"], row["cite"]
        else:
            assert abs(got - row["bytes"]) <= row["rel_tol"] * row["bytes"], row["cite"]


def test_kv_formula_scales_linearly_in_every_factor():
    base = oracle.kv_bytes_per_token(3, 5, 64, 2)
    assert oracle.kv_bytes_per_token(6, 5, 64, 2) == 2 * base
    assert oracle.kv_bytes_per_token(3, 10, 64, 2) == 2 * base
    assert oracle.kv_bytes_per_token(3, 5, 128, 2) == 2 * base
    assert oracle.kv_bytes_per_token(3, 5, 64, 1) * 2 == base       # fp8 halves it
    assert base == 2 * 3 * 5 * 64 * 2                                 # K and V: the leading 2


def test_pool_worked_example(golden_dir):
    p = _golden(golden_dir, "kv_sizes.json")["pool"]
    assert p["block_size"] * p["bytes_per_token"] == p["block_bytes"]
    blocks = oracle.pool_blocks(p["pool_bytes"], p["block_size"], p["bytes_per_token"])
    assert blocks == p["blocks"], p["cite"]
    assert blocks * p["block_size"] == p["tokens"]
    assert round(p["tokens"] / p["concurrency_at"], 1) == p["concurrency"]


def test_mixed_workload_pool_size():
    wl = inputs.get("mixed-llama3-8b-bf16")
    per_tok = oracle.kv_bytes_per_token(1, wl.n_kv_heads, wl.head_dim, wl.elem_bytes)
    assert per_tok == 4096
    assert oracle.pool_blocks(int(wl.pool_arg), wl.block_size, per_tok) == 457763


def test_blocks_for_tokens(golden_dir):
    d = _golden(golden_dir, "block_table_diagram.json")["thirty_tokens"]
    assert oracle.blocks_for_tokens(d["tokens"], 16) == d["blocks"]
    waste = d["blocks"] * 16 - d["tokens"]
    assert 0 <= waste <= d["max_waste"]
    # a new block exactly every block_size tokens; waste always < block size
    for bs in (16, 32):
        prev = 0
        for L in range(1, 5 * bs + 1):
            n = oracle.blocks_for_tokens(L, bs)
            assert n == prev + (1 if (L - 1) % bs == 0 else 0)
            assert 0 <= n * bs - L < bs
            prev = n


# ------------------------------------------------------------ allocator

def test_allocator_fifo_refcount_and_return():
    order = [5, 2, 7, 0, 1, 3, 4, 6]
    a = oracle.Allocator(8, order)
    assert a.num_free() == 8
    x = a.take(3)
    assert list(x) == [5, 2, 7]
    assert a.num_free() == 5 and a.refcount(5) == 1
    assert a.take(6) is None and a.num_free() == 5       # not enough: nothing taken
    a.share([2])
    assert a.refcount(2) == 2
    a.release([2])
    assert a.refcount(2) == 1 and a.num_free() == 5      # still held by one sharer
    a.release(x)
    assert a.num_free() == 8                             # all blocks back immediately
    y = a.take(8)
    assert list(y) == [0, 1, 3, 4, 6, 5, 2, 7]           # freed blocks went to the tail


def test_tables_follow_page_diagram(golden_dir):
    d = _golden(golden_dir, "block_table_diagram.json")
    bs = d["block_size"]
    order = d["table"] + [i for i in range(16) if i not in d["table"]]
    a = oracle.Allocator(16, order)
    t = a.build_tables([d["tokens_shown"]], max_blocks=4, block_size=bs)
    assert list(t[0]) == d["table"] + [-1]
    ex = d["examples"]
    slots = oracle.slot_mapping(t, bs, [0] * len(ex), [e["pos"] for e in ex])
    assert list(slots) == [e["phys"] * bs + e["offset"] for e in ex]


def test_tables_new_block_every_bs_tokens_and_sharing():
    bs = 16
    a = oracle.Allocator(64, np.arange(64)[::-1].copy())
    lens = [16, 17, 33, 1]
    t = a.build_tables(lens, max_blocks=4, block_size=bs)
    assert [int((row >= 0).sum()) for row in t] == [1, 2, 3, 1]
    assert a.num_free() == 64 - 7
    # sharers: the prefix blocks are taken once and shared, refcount = #sharers
    a2 = oracle.Allocator(64, np.arange(64))
    lens = [40, 50, 10, 70]
    sharer = [1, 0, 0, 1]
    t2 = a2.build_tables(lens, max_blocks=6, block_size=bs, sharer=sharer, prefix_tokens=32)
    assert list(t2[0][:2]) == [0, 1] and list(t2[3][:2]) == [0, 1]
    assert a2.refcount(0) == 2 and a2.refcount(1) == 2
    assert list(t2[0][:3]) == [0, 1, 2]            # own block after the prefix
    assert list(t2[1][:5]) == [3, 4, 5, 6, -1]     # 50 tokens: 4 blocks
    assert list(t2[2][:2]) == [7, -1]
    assert list(t2[3][:6]) == [0, 1, 8, 9, 10, -1]  # 70 tokens: 2 shared + 3 own
    assert a2.num_free() == 64 - 11


# ------------------------------------------------------ cache write, gather

def _nan_pool(nb, n_kv, bs, d, dtype):
    return torch.full((nb, n_kv, bs, d), float("nan"), dtype=dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_cache_write_then_gather_roundtrip(dtype):
    wl = inputs.random_case(7, 3, 4, 2, 64, 16, dtype, [5, 16, 40])
    dr = inputs.Draws(wl)
    lens = dr.decode_lens()
    nb = 12
    a = oracle.Allocator(nb, dr.free_order(nb))
    t = a.build_tables(lens, max_blocks=3, block_size=16)
    kvs = dr.all_seq_kv(lens, threads=1)
    seq = np.concatenate([np.full(L, s) for s, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L) for L in lens])
    slots = oracle.slot_mapping(t, 16, seq, pos)
    assert len(set(slots.tolist())) == len(slots)           # no two tokens share a slot
    K = torch.cat([k for k, _ in kvs]); V = torch.cat([v for _, v in kvs])
    kc0, vc0 = _nan_pool(nb, 2, 16, 64, dtype), _nan_pool(nb, 2, 16, 64, dtype)
    kc, vc = oracle.cache_write(kc0, vc0, K, V, slots, 16)
    kc_t = torch.from_numpy(kc).view(dtype).reshape(kc0.shape)
    vc_t = torch.from_numpy(vc).view(dtype).reshape(vc0.shape)
    for s, L in enumerate(lens):
        gk = oracle.gather(kc_t, t[s], int(L))
        gv = oracle.gather(vc_t, t[s], int(L))
        assert np.array_equal(gk, kvs[s][0].contiguous().view(torch.uint8).numpy().reshape(-1))
        assert np.array_equal(gv, kvs[s][1].contiguous().view(torch.uint8).numpy().reshape(-1))
    # every slot not written keeps its sentinel bytes
    written = np.zeros(nb * 16, bool)
    written[slots] = True
    kc_rows = kc_t.permute(0, 2, 1, 3).reshape(nb * 16, -1)
    assert torch.isnan(kc_rows[torch.from_numpy(~written)].float()).all()
    assert not torch.isnan(kc_rows[torch.from_numpy(written)].float()).any()


def test_cache_write_skips_negative_slots_and_diagram_slot():
    dtype = torch.float32
    kc0, vc0 = _nan_pool(16, 1, 16, 4, dtype), _nan_pool(16, 1, 16, 4, dtype)
    k = torch.arange(8, dtype=dtype).reshape(2, 1, 4)
    v = -k
    kc, vc = oracle.cache_write(kc0, vc0, k, v, [3 * 16 + 1, -1], 16)   # token t17 of seq A
    kc_t = torch.from_numpy(kc).view(dtype).reshape(16, 1, 16, 4)
    vc_t = torch.from_numpy(vc).view(dtype).reshape(16, 1, 16, 4)
    assert torch.equal(kc_t[3, 0, 1], k[0, 0]) and torch.equal(vc_t[3, 0, 1], v[0, 0])
    assert int((~torch.isnan(kc_t)).sum()) == 4


def test_gather_is_permutation_invariant():
    """Any scatter of the same logical rows over physical blocks gathers back to
    the same logical K/V, so attention over it is identical."""
    dtype = torch.bfloat16
    wl = inputs.random_case(11, 2, 4, 2, 64, 16, dtype, [37, 20])
    dr = inputs.Draws(wl)
    lens = dr.decode_lens()
    kvs = dr.all_seq_kv(lens, threads=1)
    outs = []
    for perm_seed in (1, 2, 3):
        nb = 10
        order = np.random.default_rng(perm_seed).permutation(nb).astype(np.int32)
        a = oracle.Allocator(nb, order)
        t = a.build_tables(lens, max_blocks=3, block_size=16)
        seq = np.concatenate([np.full(L, s) for s, L in enumerate(lens)])
        pos = np.concatenate([np.arange(L) for L in lens])
        slots = oracle.slot_mapping(t, 16, seq, pos)
        K = torch.cat([k for k, _ in kvs]); V = torch.cat([v for _, v in kvs])
        kc, vc = oracle.cache_write(_nan_pool(nb, 2, 16, 64, dtype), _nan_pool(nb, 2, 16, 64, dtype),
                                    K, V, slots, 16)
        kc_t = torch.from_numpy(kc).view(dtype).reshape(nb, 2, 16, 64)
        vc_t = torch.from_numpy(vc).view(dtype).reshape(nb, 2, 16, 64)
        ks = [torch.from_numpy(oracle.gather(kc_t, t[s], int(L))).view(dtype).reshape(int(L), 2, 64)
              for s, L in enumerate(lens)]
        vs = [torch.from_numpy(oracle.gather(vc_t, t[s], int(L))).view(dtype).reshape(int(L), 2, 64)
              for s, L in enumerate(lens)]
        outs.append(oracle.decode(dr.q(), ks, vs, wl.scale, threads=1))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


# ------------------------------------------------------------- attention

def _sdpa(q, k, v, scale, causal=False, mask=None):
    """torch's scaled_dot_product_attention in fp64 on the CPU.
    q [Lq][n_q][d], k/v [Lk][n_kv][d] -> [Lq][n_q][d]."""
    qq = q.to(torch.float64).permute(1, 0, 2).unsqueeze(0)
    kk = k.to(torch.float64).permute(1, 0, 2).unsqueeze(0)
    vv = v.to(torch.float64).permute(1, 0, 2).unsqueeze(0)
    o = torch.nn.functional.scaled_dot_product_attention(
        qq, kk, vv, attn_mask=mask, is_causal=causal, scale=scale,
        enable_gqa=qq.shape[1] != kk.shape[1])
    return o.squeeze(0).permute(1, 0, 2).numpy()


def test_decode_hand_example():
    # q=(1,0), K rows (1,0),(0,0), scale 1: weights e/(e+1), 1/(e+1)
    q = torch.tensor([[[1.0, 0.0]]], dtype=torch.float64)
    k = torch.tensor([[[1.0, 0.0]], [[0.0, 0.0]]], dtype=torch.float64)
    v = torch.tensor([[[1.0, 2.0]], [[3.0, 4.0]]], dtype=torch.float64)
    out = oracle.decode(q, [k], [v], 1.0, threads=1)
    e = math.e
    assert np.allclose(out[0, 0], [(e + 3) / (e + 1), (2 * e + 4) / (e + 1)], rtol=0, atol=1e-15)


@pytest.mark.parametrize("n_q,n_kv", [(4, 4), (4, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("scale", [0.125, 0.7])
def test_decode_matches_library_sdpa(n_q, n_kv, scale):
    g = torch.Generator().manual_seed(n_q * 10 + n_kv)
    lens = [1, 5, 37]
    q = torch.randn(3, n_q, 32, generator=g, dtype=torch.float64)
    ks = [torch.randn(L, n_kv, 32, generator=g, dtype=torch.float64) for L in lens]
    vs = [torch.randn(L, n_kv, 32, generator=g, dtype=torch.float64) for L in lens]
    out = oracle.decode(q, ks, vs, scale, threads=2)
    for s in range(3):
        ref = _sdpa(q[s:s + 1], ks[s], vs[s], scale)
        assert np.allclose(out[s], ref[0], rtol=0, atol=1e-12)


def test_decode_gqa_equals_mha_with_repeated_kv():
    g = torch.Generator().manual_seed(3)
    q = torch.randn(2, 8, 16, generator=g, dtype=torch.float64)
    ks = [torch.randn(L, 2, 16, generator=g, dtype=torch.float64) for L in (9, 4)]
    vs = [torch.randn(L, 2, 16, generator=g, dtype=torch.float64) for L in (9, 4)]
    out = oracle.decode(q, ks, vs, 0.25, threads=1)
    ks4 = [k.repeat_interleave(4, dim=1) for k in ks]
    vs4 = [v.repeat_interleave(4, dim=1) for v in vs]
    assert np.array_equal(out, oracle.decode(q, ks4, vs4, 0.25, threads=1))
    # a different grouping (head h -> kv h % n_kv) gives a different answer here
    ks_bad = [k.repeat(1, 4, 1) for k in ks]
    vs_bad = [v.repeat(1, 4, 1) for v in vs]
    assert not np.allclose(out, oracle.decode(q, ks_bad, vs_bad, 0.25, threads=1))


def test_decode_closed_forms():
    g = torch.Generator().manual_seed(5)
    d = 16
    q = torch.randn(1, 2, d, generator=g, dtype=torch.float64)
    # L = 1: the output is v0, exactly
    k1 = torch.randn(1, 1, d, generator=g, dtype=torch.float64)
    v1 = torch.randn(1, 1, d, generator=g, dtype=torch.float64)
    out = oracle.decode(q, [k1], [v1], 0.3, threads=1)
    assert np.array_equal(out[0, 0], v1[0, 0].numpy()) and np.array_equal(out[0, 1], v1[0, 0].numpy())
    # constant keys: uniform weights, the output is the mean of V
    kc = torch.randn(1, 1, d, generator=g, dtype=torch.float64).repeat(20, 1, 1)
    vc = torch.randn(20, 1, d, generator=g, dtype=torch.float64)
    out = oracle.decode(q, [kc], [vc], 0.3, threads=1)
    assert np.allclose(out[0, 0], vc[:, 0].mean(0).numpy(), atol=1e-14)
    # scale 0: uniform weights as well
    kr = torch.randn(20, 1, d, generator=g, dtype=torch.float64)
    out = oracle.decode(q, [kr], [vc], 0.0, threads=1)
    assert np.allclose(out[0, 0], vc[:, 0].mean(0).numpy(), atol=1e-14)
    # one dominant logit: the output is that row of V
    kd = torch.zeros(20, 1, d, dtype=torch.float64)
    kd[13, 0] = 100.0 * q[0, 0]
    out = oracle.decode(q[:, :1], [kd], [vc], 1.0, threads=1)
    assert np.allclose(out[0, 0], vc[13, 0].numpy(), atol=1e-12)


def test_decode_reads_only_first_L_rows():
    """Rows at or beyond L must not matter; the oracle only ever sees L rows,
    so truncating a longer sequence equals passing the shorter one."""
    g = torch.Generator().manual_seed(9)
    q = torch.randn(1, 2, 8, generator=g, dtype=torch.float64)
    k = torch.randn(10, 1, 8, generator=g, dtype=torch.float64)
    v = torch.randn(10, 1, 8, generator=g, dtype=torch.float64)
    a = oracle.decode(q, [k[:6]], [v[:6]], 0.5, threads=1)
    ref = _sdpa(q, k[:6], v[:6], 0.5)
    assert np.allclose(a[0], ref[0], atol=1e-13)


@pytest.mark.parametrize("n_q,n_kv", [(4, 4), (4, 1), (6, 2)])
def test_prefill_matches_library_sdpa_with_offset_causal_mask(n_q, n_kv):
    g = torch.Generator().manual_seed(17 + n_q)
    d = 16
    specs = [(0, 7), (5, 3), (30, 9)]              # (cached tokens, chunk)
    qs, ks, vs = [], [], []
    for ctx, c in specs:
        qs.append(torch.randn(c, n_q, d, generator=g, dtype=torch.float64))
        ks.append(torch.randn(ctx + c, n_kv, d, generator=g, dtype=torch.float64))
        vs.append(torch.randn(ctx + c, n_kv, d, generator=g, dtype=torch.float64))
    outs = oracle.prefill(qs, ks, vs, 0.4, threads=3)
    for (ctx, c), q, k, v, o in zip(specs, qs, ks, vs, outs):
        L = ctx + c
        # query i sits at position ctx + i and sees keys 0..ctx+i
        mask = torch.arange(L)[None, :] <= (ctx + torch.arange(c))[:, None]
        ref = _sdpa(q, k, v, 0.4, mask=mask)
        assert np.allclose(o, ref, atol=1e-12)
        if ctx == 0:
            assert np.allclose(o, _sdpa(q, k, v, 0.4, causal=True), atol=1e-12)


def test_prefill_chunk_of_one_equals_decode_and_chunks_compose():
    g = torch.Generator().manual_seed(23)
    n_q, n_kv, d, L = 4, 2, 16, 25
    k = torch.randn(L, n_kv, d, generator=g, dtype=torch.float64)
    v = torch.randn(L, n_kv, d, generator=g, dtype=torch.float64)
    q = torch.randn(10, n_q, d, generator=g, dtype=torch.float64)
    # a chunk of 1 at the last position is a decode step
    one = oracle.prefill([q[-1:]], [k], [v], 0.3, threads=1)[0]
    dec = oracle.decode(q[-1:], [k], [v], 0.3, threads=1)
    assert np.array_equal(one, dec)
    # chunks c1 + c2 over the same context equal one chunk of c1 + c2
    whole = oracle.prefill([q], [k], [v], 0.3, threads=1)[0]
    first = oracle.prefill([q[:6]], [k[:L - 4]], [v[:L - 4]], 0.3, threads=1)[0]
    second = oracle.prefill([q[6:]], [k], [v], 0.3, threads=1)[0]
    assert np.array_equal(whole, np.concatenate([first, second]))


def test_decode_threads_do_not_change_bits():
    wl = inputs.get("tiny-fp32")
    dr = inputs.Draws(wl)
    lens = dr.decode_lens()
    kvs = dr.all_seq_kv(lens, threads=1)
    a = oracle.decode(dr.q(), [k for k, _ in kvs], [v for _, v in kvs], wl.scale, threads=1)
    b = oracle.decode(dr.q(), [k for k, _ in kvs], [v for _, v in kvs], wl.scale, threads=5)
    assert np.array_equal(a, b)


def test_copy_blocks_copy_on_write_example():
    """[Sharing] two tables share a block; the diverging sharer gets a copy of
    that one block and its own table entry is updated; the original stays."""
    dtype = torch.float32
    nb, n_kv, bs, d = 6, 2, 4, 8
    g = torch.Generator().manual_seed(0)
    k = torch.randn(nb, n_kv, bs, d, generator=g)
    v = torch.randn(nb, n_kv, bs, d, generator=g)
    a = oracle.Allocator(nb, np.arange(nb))
    shared = a.take(1)
    a.share(shared)                       # two sequences point at block 0
    new = a.take(1)                       # sequence B diverges: copy 0 -> 1
    dk, dv = oracle.copy_blocks(k, v, k, v, [[int(shared[0]), int(new[0])]])
    a.release(shared)                     # B drops its reference to the shared block
    kk = torch.from_numpy(dk).view(dtype).reshape(k.shape)
    vv = torch.from_numpy(dv).view(dtype).reshape(v.shape)
    assert torch.equal(kk[1], k[0]) and torch.equal(vv[1], v[0])      # the copy
    assert torch.equal(kk[0], k[0]) and torch.equal(kk[2:], k[2:])    # nothing else moves
    assert a.refcount(int(shared[0])) == 1 and a.refcount(int(new[0])) == 1
    # a copy then gathers to the same logical rows through the updated table
    tb_a, tb_b = [int(shared[0])], [int(new[0])]
    assert np.array_equal(oracle.gather(kk, tb_a, 3), oracle.gather(kk, tb_b, 3))


def test_copy_blocks_swap_round_trip_and_chains():
    nb, n_kv, bs, d = 5, 1, 2, 4
    k = torch.arange(nb * n_kv * bs * d, dtype=torch.float32).reshape(nb, n_kv, bs, d)
    v = -k
    host_k = torch.zeros_like(k); host_v = torch.zeros_like(v)
    hk, hv = oracle.copy_blocks(k, v, host_k, host_v, [[3, 0], [1, 4]])     # out to "CPU"
    hk_t = torch.from_numpy(hk).view(torch.float32).reshape(k.shape)
    hv_t = torch.from_numpy(hv).view(torch.float32).reshape(v.shape)
    assert torch.equal(hk_t[0], k[3]) and torch.equal(hk_t[4], k[1]) and torch.equal(hv_t[0], v[3])
    back_k, _ = oracle.copy_blocks(hk_t, hv_t, torch.zeros_like(k), torch.zeros_like(v), [[0, 2], [4, 0]])
    bk = torch.from_numpy(back_k).view(torch.float32).reshape(k.shape)
    assert torch.equal(bk[2], k[3]) and torch.equal(bk[0], k[1])
    # every source block is read as it was before the call (copies run in
    # parallel on the GPU), so the order of the pairs does not matter
    m = [[0, 1], [3, 2], [4, 0]]
    ck1, _ = oracle.copy_blocks(k, v, k, v, m)
    ck2, _ = oracle.copy_blocks(k, v, k, v, m[::-1])
    assert np.array_equal(ck1, ck2)
    ckt = torch.from_numpy(ck1).view(torch.float32).reshape(k.shape)
    assert torch.equal(ckt[1], k[0]) and torch.equal(ckt[2], k[3]) and torch.equal(ckt[0], k[4])


# ------------------------------------------------------------- fp8 e4m3

def test_fp8_e4m3_decode_known_codes():
    """Values fixed by the E4M3 format definition (bias 7, 3 mantissa bits)."""
    known = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
             0x39: 1.125, 0x40: 2.0, 0x7E: 448.0, 0x7D: 416.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in known.items():
        assert oracle.fp8_decode(c) == v, hex(c)
    assert math.isnan(oracle.fp8_decode(0x7F)) and math.isnan(oracle.fp8_decode(0xFF))


def test_fp8_e4m3_round_trip_monotone_ties_saturation():
    vals = [oracle.fp8_decode(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))                 # strictly increasing
    # all 254 non-NaN codes, both zeros included: decode then encode is the
    # identity (decode(0x80) is -0.0, whose sign bit the encoder keeps)
    codes = list(range(0x7F)) + list(range(0x80, 0xFF))
    assert len(codes) == 254
    for c in codes:
        assert oracle.fp8_encode(oracle.fp8_decode(c)) == c, hex(c)   # exact round trip
    assert math.copysign(1.0, oracle.fp8_decode(0x80)) == -1.0 and oracle.fp8_decode(0x80) == 0.0
    assert oracle.fp8_encode(1.0625) == 0x38                           # tie -> even mantissa
    assert oracle.fp8_encode(1.1875) == 0x3A
    assert oracle.fp8_encode(1.07) == 0x39                             # nearest
    assert oracle.fp8_encode(1000.0) == 0x7E and oracle.fp8_encode(-1e30) == 0xFE
    assert oracle.fp8_encode(2.0 ** -11) == 0x00                       # below half the smallest
    assert oracle.fp8_encode(3 * 2.0 ** -11) == 0x01                   # rounds up to 2^-9
    # signed zero: the sign bit is kept, also when a negative magnitude rounds to 0
    assert oracle.fp8_encode(0.0) == 0x00 and oracle.fp8_encode(-0.0) == 0x80
    assert oracle.fp8_encode(-2.0 ** -11) == 0x80 and oracle.fp8_encode(-1e-30) == 0x80
    assert oracle.fp8_encode(-3 * 2.0 ** -11) == 0x81
    # ties at the top: 464 lies halfway between 448 (even mantissa) and 480 (not
    # finite in E4M3), so it saturates like anything larger
    assert oracle.fp8_encode(464.0) == 0x7E and oracle.fp8_encode(-470.0) == 0xFE


def test_fp8_e4m3_matches_library_cast_in_range():
    """torch's float8_e4m3fn cast is round-to-nearest-even and keeps the sign
    of zero; it turns magnitudes of 480 and more into NaN instead of
    saturating, so saturation is compared as a clamp to +-448 before the cast."""
    g = torch.Generator().manual_seed(1)
    x = torch.cat([torch.randn(4000, generator=g) * 60, torch.randn(2000, generator=g) * 0.01,
                   torch.randn(2000, generator=g) * 1e-3,          # many round to +-0
                   torch.tensor([0.0, -0.0, -1e-9, 1e-9, 447.9, 448.0, 449.0, 463.9, 464.0,
                                 464.1, 479.0, 480.0, 1000.0, 3.0e38, -448.5, -500.0, -3.0e38])])
    ours = oracle.quantize_fp8(x, 1.0)
    lib = x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)
    assert (ours == 0x80).sum() > 0 and (ours == 0x00).sum() > 0 and (ours == 0xFE).sum() > 0
    # every code's value, positive and negative zero included, casts to itself
    all_vals = torch.tensor([oracle.fp8_decode(c) for c in range(0x7F)] +
                            [oracle.fp8_decode(c) for c in range(0x80, 0xFF)], dtype=torch.float32)
    assert np.array_equal(oracle.quantize_fp8(all_vals, 1.0),
                          all_vals.to(torch.float8_e4m3fn).view(torch.uint8).numpy())


def test_fp8_quantize_divides_in_fp32_then_rounds():
    scale = 0.0125
    x = torch.tensor([1.0, -3.3, 0.05, 5.0], dtype=torch.float32)     # within 448 * scale
    codes = oracle.quantize_fp8(x, scale)
    for xi, c in zip(x.tolist(), codes.tolist()):
        q = np.float32(xi) / np.float32(scale)
        assert c == oracle.fp8_encode(float(q))
    deq = oracle.dequantize_fp8(codes, scale)
    # relative rounding error of 3 mantissa bits is at most 2^-4
    assert np.all(np.abs(deq - x.numpy()) <= 0.0625 * np.abs(x.numpy()) + 2.0 ** -9 * scale)
    assert oracle.quantize_fp8(torch.tensor([9.0]), scale)[0] == 0x7E   # 720 saturates to 448


@pytest.mark.parametrize("piece", [2, 4])
def test_cache_write_transposed_v_layout(piece):
    """Row t of V that goes to slot (block b, offset o) lands column-wise in
    its piece of P tokens: element i at [b][h][o / P][i][o % P]; it holds the
    same values as the row-major pool.  P = the block size is the whole block
    transposed."""
    nb, n_kv, bs, d = 3, 2, 4, 5
    v = torch.arange(3 * n_kv * d, dtype=torch.float32).reshape(3, n_kv, d) + 1
    slots = [1 * bs + 2, 2 * bs + 0, 0 * bs + 3]
    vt = oracle.cache_write_vt(torch.zeros(nb, n_kv, bs // piece, d, piece), v, slots, bs)
    vt = torch.from_numpy(vt).view(torch.float32).reshape(nb, n_kv, bs // piece, d, piece)
    for t, s in enumerate(slots):
        b, o = divmod(s, bs)
        assert torch.equal(vt[b, :, o // piece, :, o % piece], v[t])
    assert int((vt != 0).sum()) == v.numel()
    _, vr = oracle.cache_write(torch.zeros(nb, n_kv, bs, d), torch.zeros(nb, n_kv, bs, d), v, v,
                               slots, bs)
    vr = torch.from_numpy(vr).view(torch.float32).reshape(nb, n_kv, bs // piece, piece, d)
    assert torch.equal(vr.transpose(3, 4), vt)
