"""FP8 (E4M3) KV pools: the quantizing cache write is bit-exact against the
oracle's codec, and decode over the codes matches the oracle's attention over
the dequantized values (codes times the per-tensor scale)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import inputs
from paged_kv_cache_25_gb300.step import PagedStep
from tests.helpers import max_err, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_25_gb300 import build
    build.build()
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("act,scale", [(torch.bfloat16, 1.0 / 64), (torch.float16, 0.0125),
                                       (torch.float32, 0.0125)])
def test_fp8_cache_write_whole_pool_bit_exact(act, scale):
    nb, n_kv, bs, d, T = 20, 4, 16, 128, 150
    g = torch.Generator().manual_seed(2)
    k = (torch.randn(T, n_kv, d, generator=g) * 2).to(act)
    v = (torch.randn(T, n_kv, d, generator=g) * 2).to(act)
    k[0, 0, :4] = torch.tensor([500.0, -1e4, 3.3e-4, 0.0])     # saturation, tiny, zero
    slots = np.random.default_rng(3).permutation(nb * bs)[:T].astype(np.int64)
    slots[5] = -1                                               # padding token
    kc = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    vc = torch.full((nb, n_kv, d, bs), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    pa.pa_reshape_and_cache_quant(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda(),
                                  k_scale=scale, v_scale=scale)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kq = torch.from_numpy(oracle.quantize_fp8(k, scale))
    vq = torch.from_numpy(oracle.quantize_fp8(v, scale))
    pool0 = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8)
    ek, _ = oracle.cache_write(pool0, pool0, kq, vq, slots, bs)
    # V codes land in the transposed layout [block][head][d][offset]
    ev = oracle.cache_write_vt(torch.full((nb, n_kv, d, bs), 0x7F, dtype=torch.uint8), vq, slots, bs)
    assert np.array_equal(kc.view(torch.uint8).cpu().numpy().reshape(-1), ek)
    assert np.array_equal(vc.view(torch.uint8).cpu().numpy().reshape(-1), ev)


CASES = [
    # seed, B, n_q, n_kv, d, bs, act dtype, lens, scale
    (1, 4, 32, 8, 128, 16, torch.bfloat16, [1, 17, 600, 3000], 1.0 / 64),
    (2, 3, 8, 1, 64, 32, torch.float16, [33, 500, 1200], 0.0125),
    (3, 3, 40, 40, 128, 16, torch.float16, [2048, 5, 100], 0.0125),
    (4, 2, 16, 4, 64, 16, torch.bfloat16, [4100, 64], 1.0 / 64),
]


@pytest.mark.parametrize("case", CASES, ids=[f"f{c[0]}" for c in CASES])
def test_fp8_decode_matches_oracle_on_dequantized_kv(case):
    seed, B, n_q, n_kv, d, bs, act, lens, scale = case
    wl = inputs.random_case(seed, B, n_q, n_kv, d, bs, act, lens,
                            cache_dtype=torch.float8_e4m3fn, kv_scale=scale)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ref = oracle_decode(st)
    assert max_err(st.out, ref) <= 2e-3


def test_fp8_decode_full_size_sampled():
    wl = inputs.get("llama3-8b-fp8")
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    order = np.argsort(st.lens)
    seqs = sorted({int(order[0]), int(order[-1]), 3, 77, 200})
    ref = oracle_decode(st, seqs)
    assert max_err(st.out[seqs], ref) <= 2e-3
    assert torch.isfinite(st.out).all()


def test_fp8_prefill_is_refused():
    nb = 4
    kc = torch.zeros((nb, 2, 16, 64), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    out = torch.empty((8, 4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_prefill_chunk(out, torch.zeros((8, 4, 64), dtype=torch.bfloat16, device="cuda"), kc, kc,
                            torch.zeros((1, 4), dtype=torch.int32, device="cuda"),
                            torch.tensor([0, 8], dtype=torch.int32, device="cuda"),
                            torch.tensor([8], dtype=torch.int32, device="cuda"), 8, 0.125, 16)
    assert e.value.status in (pa.PA_ERR_UNSUPPORTED, pa.PA_ERR_INVALID_ARG)
