"""GPU parity of whole-block copies (copy-on-write) and swaps (device <->
pinned host) against the oracle, bit for bit, plus a copy-on-write fork whose
two branches then decode correctly."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_25_gb300 import binding as pa
from tests.helpers import max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_25_gb300 import build
    build.build()
    assert pa.pa_get_device_error() == 0


def _pool(nb, n_kv, bs, d, dtype, seed, nan_frac=0.1):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(nb, n_kv, bs, d, generator=g)
    x[torch.rand(x.shape, generator=g) < nan_frac] = float("nan")
    return x.to(dtype)


def _as(b, like):
    return torch.from_numpy(b).view(like.dtype).reshape(like.shape)


@pytest.mark.parametrize("dtype,bs,d", [(torch.bfloat16, 16, 128), (torch.float32, 32, 64),
                                        (torch.float16, 16, 64)])
def test_copy_blocks_bit_exact(dtype, bs, d):
    nb, n_kv = 40, 4
    k, v = _pool(nb, n_kv, bs, d, dtype, 1), _pool(nb, n_kv, bs, d, dtype, 2)
    perm = np.random.default_rng(3).permutation(nb)
    mapping = np.stack([perm[:12], perm[12:24]], 1).astype(np.int32)   # disjoint sources / targets
    kd, vd = k.cuda(), v.cuda()
    pa.pa_copy_blocks(kd, vd, torch.from_numpy(mapping).cuda())
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ek, ev = oracle.copy_blocks(k, v, k, v, mapping)
    assert np.array_equal(kd.cpu().view(torch.uint8).numpy().reshape(-1), ek)
    assert np.array_equal(vd.cpu().view(torch.uint8).numpy().reshape(-1), ev)


def test_swap_device_to_pinned_host_and_back():
    nb, n_kv, bs, d, dtype = 64, 8, 16, 128, torch.bfloat16
    k, v = _pool(nb, n_kv, bs, d, dtype, 4), _pool(nb, n_kv, bs, d, dtype, 5)
    kd, vd = k.cuda(), v.cuda()
    host_k = torch.zeros((16, n_kv, bs, d), dtype=dtype).pin_memory()
    host_v = torch.zeros((16, n_kv, bs, d), dtype=dtype).pin_memory()
    out_map = np.array([[5, 0], [63, 3], [17, 15], [0, 7]], np.int32)
    pa.pa_swap_blocks(kd, vd, host_k, host_v, torch.from_numpy(out_map).cuda())
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ek, ev = oracle.copy_blocks(k, v, torch.zeros_like(host_k), torch.zeros_like(host_v), out_map)
    assert np.array_equal(host_k.view(torch.uint8).numpy().reshape(-1), ek)
    assert np.array_equal(host_v.view(torch.uint8).numpy().reshape(-1), ev)
    # back into other device blocks, with the mapping itself in pinned host memory
    in_map = torch.from_numpy(np.array([[0, 40], [3, 41], [15, 2]], np.int32)).pin_memory()
    pa.pa_swap_blocks(host_k, host_v, kd, vd, in_map)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    bk, bv = oracle.copy_blocks(_as(ek, host_k), _as(ev, host_v), k, v, in_map.numpy())
    assert np.array_equal(kd.cpu().view(torch.uint8).numpy().reshape(-1), bk)
    assert np.array_equal(vd.cpu().view(torch.uint8).numpy().reshape(-1), bv)


def test_copy_blocks_out_of_range_flagged_and_skipped():
    nb = 8
    k = _pool(nb, 2, 16, 64, torch.bfloat16, 6).cuda()
    v = _pool(nb, 2, 16, 64, torch.bfloat16, 7).cuda()
    before = k.clone()
    pa.pa_copy_blocks(k, v, torch.tensor([[1, nb]], dtype=torch.int32, device="cuda"))
    assert pa.pa_get_device_error() == pa.PA_ERR_OUT_OF_RANGE
    assert torch.equal(k.view(torch.int16), before.view(torch.int16))
    assert pa.pa_get_device_error() == 0


def test_copy_on_write_fork_then_decode():
    """Two sequences share a 40-token prompt (3 blocks of 16, the last one
    half full).  B forks: it gets a copy of the shared last block before
    appending its own tokens; A appends into the original.  Both then decode
    correctly against their own logical K/V."""
    dtype, n_q, n_kv, d, bs = torch.bfloat16, 8, 2, 64, 16
    g = torch.Generator().manual_seed(9)
    prompt_k = torch.randn(40, n_kv, d, generator=g).to(dtype)
    prompt_v = torch.randn(40, n_kv, d, generator=g).to(dtype)
    tail = {s: (torch.randn(10, n_kv, d, generator=g).to(dtype),
                torch.randn(10, n_kv, d, generator=g).to(dtype)) for s in "AB"}
    nb = 12
    alloc = pa.Allocator(nb)
    shared = alloc.blocks(3)
    alloc.share(shared)                                  # A and B both point at them
    kc = torch.full((nb, n_kv, bs, d), float("nan"), dtype=dtype, device="cuda")
    vc = kc.clone()
    slots = pa.pa_slot_mapping(np.array([shared]), bs, np.zeros(40, np.int32),
                               np.arange(40, dtype=np.int32))
    pa.pa_reshape_and_cache(prompt_k.cuda(), prompt_v.cuda(), kc, vc, torch.from_numpy(slots).cuda())
    # B writes into the shared, partly filled block 2: copy on write
    assert alloc.refcount(int(shared[2])) == 2
    cow = alloc.blocks(1)
    pa.pa_copy_blocks(kc, vc, torch.tensor([[int(shared[2]), int(cow[0])]], dtype=torch.int32,
                                           device="cuda"))
    alloc.free(shared[2:3])
    tab = {"A": list(shared) + [-1] * 1, "B": list(shared[:2]) + [int(cow[0])] + [-1]}
    for s in "AB":
        extra = alloc.blocks(1)
        tab[s][3] = int(extra[0])
    tables = np.array([tab["A"], tab["B"]], np.int32)
    seq = np.repeat(np.arange(2, dtype=np.int32), 10)
    pos = np.tile(np.arange(40, 50, dtype=np.int32), 2)
    slots = pa.pa_slot_mapping(tables, bs, seq, pos)
    nk = torch.cat([tail["A"][0], tail["B"][0]]).cuda()
    nv = torch.cat([tail["A"][1], tail["B"][1]]).cuda()
    pa.pa_reshape_and_cache(nk, nv, kc, vc, torch.from_numpy(slots).cuda())
    q = torch.randn(2, n_q, d, generator=g).to(dtype)
    out = torch.empty((2, n_q, d), dtype=torch.float32, device="cuda")
    ws = torch.empty(pa.pa_decode_workspace_size(2, n_q, n_kv, d, bs, 4 * bs), dtype=torch.uint8,
                     device="cuda")
    pa.pa_decode(out, q.cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                 torch.tensor([50, 50], dtype=torch.int32, device="cuda"), 0.125, bs, ws)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ks = [torch.cat([prompt_k, tail[s][0]]) for s in "AB"]
    vs = [torch.cat([prompt_v, tail[s][1]]) for s in "AB"]
    ref = oracle.decode(q, ks, vs, 0.125)
    assert max_err(out, ref) <= 2e-3
