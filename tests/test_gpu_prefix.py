"""Decode over block tables handed out by the host prefix cache: requests that
share a token prefix share its full blocks, only the tokens past their hits are
written, and the decode still equals the oracle on each request's own logical
K/V, also after cached blocks have been evicted and reused."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import inputs
from tests.helpers import TOL, max_err

pytestmark = pytest.mark.gpu

SEED, BS, NQ, NKV, D, DT = 2024, 16, 8, 2, 128, torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_25_gb300 import build
    build.build()
    assert pa.pa_get_device_error() == 0


def _admit(pc, toks, kc, vc, mb):
    """Acquire a table, write the K/V rows past the hits, commit.  None when
    the pool cannot supply the request's new blocks."""
    r = pc.acquire(toks, mb)
    if r is None:
        return None
    k, table = r
    if kc is not None:
        kk, vv = inputs.token_keyed_kv(SEED, toks, NKV, D, DT)
        pos = np.arange(k * BS, len(toks), dtype=np.int32)
        if len(pos):
            slots = pa.pa_slot_mapping(table[None, :], BS, np.zeros(len(pos), np.int32), pos)
            pa.pa_reshape_and_cache(kk[pos].contiguous().cuda(), vv[pos].contiguous().cuda(), kc,
                                    vc, torch.from_numpy(slots).cuda())
    pc.commit(toks, table)
    return k, table


def _decode_and_check(live, kc, vc, mb, qseed):
    B = len(live)
    tables = np.stack([t for _, t in live]).astype(np.int32)
    lens = np.array([len(x) for x, _ in live], np.int32)
    q = torch.randn(B, NQ, D, generator=torch.Generator().manual_seed(qseed)).to(DT)
    out = torch.empty(B, NQ, D, dtype=torch.float32, device="cuda")
    ws = torch.empty(pa.pa_decode_workspace_size(B, NQ, NKV, D, BS, int(lens.max())),
                     dtype=torch.uint8, device="cuda")
    pa.pa_decode(out, q.cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                 torch.from_numpy(lens).cuda(), float(1 / np.sqrt(D)), BS, ws)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ks, vs = zip(*(inputs.token_keyed_kv(SEED, x, NKV, D, DT) for x, _ in live))
    ref = oracle.decode(q, list(ks), list(vs), float(np.float32(1 / np.sqrt(D))))
    assert max_err(out, ref) <= TOL[DT]


def _scenario(on_gpu):
    nb, mb = 40, 8
    rng = np.random.default_rng(7)
    pc = pa.PrefixCache(nb, BS, rng.permutation(nb))
    kc = torch.full((nb, NKV, BS, D), float("nan"), dtype=DT, device="cuda") if on_gpu else None
    vc = torch.full_like(kc, float("nan")) if on_gpu else None
    stem = list(inputs.token_stream(SEED, 0, 80, 1000))

    def request(i):
        cut = int(rng.integers(0, 81))
        return stem[:cut] + list(inputs.token_stream(SEED, i, int(rng.integers(1, 40)), 1000))

    # wave 1: six requests off one system prompt
    live, hits = [], 0
    for i in range(1, 7):
        toks = request(i)
        k, table = _admit(pc, toks, kc, vc, mb)
        hits += k
        live.append((toks, table))
    assert hits > 0                                  # some prefix blocks were shared
    if kc is not None:
        _decode_and_check(live, kc, vc, mb, 1)

    # wave 2: keep at most five requests live; admitting more drains the free
    # queue, after which new blocks come from evicted cached ones
    evictions = 0
    for i in range(7, 60):
        toks = request(i)
        new_blocks = -(-len(toks) // BS) - pc.lookup(toks)
        while True:
            short = new_blocks > pc.num_free()
            r = _admit(pc, toks, kc, vc, mb)
            if r is not None:
                evictions += short
                live.append((toks, r[1]))
                break
            pc.release(live.pop(0)[1])               # pool exhausted: retire the oldest
        if len(live) > 5:
            pc.release(live.pop(0)[1])
    assert evictions > 0 and pc.num_cached() >= 1
    if kc is not None:
        _decode_and_check(live, kc, vc, mb, 2)
    return evictions


def test_decode_over_prefix_cache_tables_with_sharing_and_eviction():
    assert _scenario(on_gpu=True) > 0
