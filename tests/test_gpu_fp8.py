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
from tests.helpers import (check_low_precision, half_ulp, max_err, oracle_decode, oracle_decode_all,
                           oracle_prefill_all)

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
    # signed zeros: -0.0 and negatives whose quotient rounds to zero keep the
    # sign bit (code 0x80), positive ones give 0x00
    k[1, 1, :6] = torch.tensor([-0.0, -1e-9, -1e-6, 0.0, 1e-9, -0.0])
    v[2, 0, :6] = torch.tensor([-0.0, -1e-9, -1e-6, 0.0, 1e-9, -0.0])
    slots = np.random.default_rng(3).permutation(nb * bs)[:T].astype(np.int64)
    slots[5] = -1                                               # padding token
    kc = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    vc = torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8,
                    device="cuda").view(torch.float8_e4m3fn)
    pa.pa_reshape_and_cache_quant(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda(),
                                  k_scale=scale, v_scale=scale)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kq = torch.from_numpy(oracle.quantize_fp8(k, scale))
    vq = torch.from_numpy(oracle.quantize_fp8(v, scale))
    pool0 = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8)
    ek, _ = oracle.cache_write(pool0, pool0, kq, vq, slots, bs)
    # V codes land in the transposed layout [block][head][offset / 16][d][offset % 16]
    ev = oracle.cache_write_vt(torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8),
                               vq, slots, bs)
    assert np.array_equal(kc.view(torch.uint8).cpu().numpy().reshape(-1), ek)
    assert np.array_equal(vc.view(torch.uint8).cpu().numpy().reshape(-1), ev)
    # the negative-zero code is among the expected bytes of both pools (unless
    # the slot of token 1 / 2 is the skipped one)
    assert (kq[1, 1, :3] == 0x80).all() and (vq[2, 0, :3] == 0x80).all()
    assert (ek == 0x80).any() and (ev == 0x80).any()


@pytest.mark.parametrize("bs,d", [(16, 128), (32, 64), (32, 128), (16, 64)])
def test_fp8_cache_write_slot_patterns_bit_exact(bs, d):
    """Slot patterns the writer stores differently: 16 aligned consecutive slots
    (whole 16-byte rows of the transposed V slab), aligned runs of 4, an
    unaligned run, scattered slots, padding (-1) and a ragged tail of tokens.
    Every byte of both pools equals the oracle's writes of the oracle's codes."""
    nb, n_kv = 12, 3
    rng = np.random.default_rng(bs + d)
    runs = [np.arange(2 * bs, 2 * bs + 16),                 # aligned 16
            np.arange(5 * bs + 4, 5 * bs + 8),              # aligned 4 ...
            np.arange(7 * bs + 0, 7 * bs + 4),
            np.array([3 * bs + 1, 3 * bs + 2, 3 * bs + 3, 3 * bs + 4]),   # unaligned 4
            np.arange(9 * bs + 3, 9 * bs + 19) % (nb * bs),  # unaligned 16 (may cross a block)
            np.array([-1, 11 * bs + 7, -1, 0]),              # padding and scattered
            rng.permutation(np.arange(4 * bs, 5 * bs))[:7]]  # ragged tail of 7
    slots = np.concatenate(runs).astype(np.int64)
    assert len(np.unique(slots[slots >= 0])) == int((slots >= 0).sum())   # no slot twice
    T = len(slots)
    g = torch.Generator().manual_seed(bs * d)
    k = (torch.randn(T, n_kv, d, generator=g) * 3).to(torch.bfloat16)
    v = (torch.randn(T, n_kv, d, generator=g) * 3).to(torch.bfloat16)
    kc = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    vc = torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8,
                    device="cuda").view(torch.float8_e4m3fn)
    pa.pa_reshape_and_cache_quant(k.cuda(), v.cuda(), kc, vc, torch.from_numpy(slots).cuda(),
                                  k_scale=0.05, v_scale=0.03)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kq = torch.from_numpy(oracle.quantize_fp8(k, 0.05))
    vq = torch.from_numpy(oracle.quantize_fp8(v, 0.03))
    pool0 = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8)
    ek, _ = oracle.cache_write(pool0, pool0, kq, kq, slots, bs)
    ev = oracle.cache_write_vt(torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8),
                               vq, slots, bs)
    assert np.array_equal(kc.view(torch.uint8).cpu().numpy().reshape(-1), ek)
    assert np.array_equal(vc.view(torch.uint8).cpu().numpy().reshape(-1), ev)


@pytest.mark.parametrize("bs,d", [(16, 128), (32, 64)])
def test_fp8_cache_write_of_codes_bit_exact(bs, d):
    """Rows that already hold E4M3 codes, written through pa_reshape_and_cache
    and through pa_reshape_and_cache_quant with the codes' own dtype: K codes
    land row-major, V codes in the pool's transposed layout, every byte as
    the oracle's writes of the same codes."""
    nb, n_kv, T = 12, 2, 100
    rng = np.random.default_rng(9)
    codes_k = rng.integers(0, 256, size=(T, n_kv, d), dtype=np.uint8)
    codes_v = rng.integers(0, 256, size=(T, n_kv, d), dtype=np.uint8)
    slots = rng.permutation(nb * bs)[:T].astype(np.int64)
    slots[7] = -1
    k = torch.from_numpy(codes_k).cuda().view(torch.float8_e4m3fn)
    v = torch.from_numpy(codes_v).cuda().view(torch.float8_e4m3fn)
    pool0 = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8)
    ek, _ = oracle.cache_write(pool0, pool0, torch.from_numpy(codes_k), torch.from_numpy(codes_k),
                               slots, bs)
    ev = oracle.cache_write_vt(torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8),
                               torch.from_numpy(codes_v), slots, bs)
    for entry in ("plain", "quant"):
        kc = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
        vc = torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8,
                        device="cuda").view(torch.float8_e4m3fn)
        sl = torch.from_numpy(slots).cuda()
        if entry == "plain":
            pa.pa_reshape_and_cache(k, v, kc, vc, sl, k_scale=0.5, v_scale=0.25)
        else:
            pa.pa_reshape_and_cache_quant(k, v, kc, vc, sl, k_scale=0.5, v_scale=0.25)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        assert np.array_equal(kc.view(torch.uint8).cpu().numpy().reshape(-1), ek), entry
        assert np.array_equal(vc.view(torch.uint8).cpu().numpy().reshape(-1), ev), entry


CASES = [
    # seed, B, n_q, n_kv, d, bs, act dtype, lens, scale
    (1, 4, 32, 8, 128, 16, torch.bfloat16, [1, 17, 600, 3000], 1.0 / 64),
    (2, 3, 8, 1, 64, 32, torch.float16, [33, 500, 1200], 0.0125),
    (3, 3, 40, 40, 128, 16, torch.float16, [2048, 5, 100], 0.0125),
    (4, 2, 16, 4, 64, 16, torch.bfloat16, [4100, 64], 1.0 / 64),
]


TRANSPOSED_CASES = [
    # up to 4 query heads a KV head run the transposed kernel: every group
    # size 1-4 with both head dims and both block sizes among them
    (5, 3, 8, 4, 128, 32, torch.bfloat16, [2, 1023, 1500], 1.0 / 64),   # g=2
    (6, 4, 12, 4, 64, 32, torch.float16, [17, 32, 800, 2100], 0.0125),  # g=3
    (7, 3, 12, 3, 128, 16, torch.bfloat16, [48, 1, 3000], 1.0 / 64),    # g=4, 3 KV heads
    (8, 2, 6, 6, 64, 32, torch.bfloat16, [5000, 31], 1.0 / 64),         # g=1, d 64, bs 32
]
CASES = CASES + TRANSPOSED_CASES


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


def test_fp8_decode_full_size_all_outputs():
    """Every output of the Llama-3-8B batch over the FP8 pool, in fp32 and in
    bf16, against the oracle's attention over the dequantized codes."""
    wl = inputs.get("llama3-8b-fp8")
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    out_lp = torch.full(tuple(st.out.shape), float("nan"), dtype=wl.dtype, device="cuda")
    pa.pa_decode(out_lp, st.q, st.k_cache, st.v_cache, st.block_tables, st.context_lens,
                 wl.scale, wl.block_size, st.workspace, **st.kv_scales)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    ref = oracle_decode_all(st)
    assert max_err(st.out, ref) <= 2e-3
    assert check_low_precision(out_lp, ref, wl.dtype) <= 0.0


@pytest.mark.parametrize("q_pow2", [24, -30])
@pytest.mark.parametrize("d", [128, 64])
def test_fp8_decode_bf16_queries_outside_fp16_range(q_pow2, d):
    """bf16 queries far above fp16's largest value or below its smallest normal
    over an FP8 pool (the decode MMAs run on fp16 operands: each q row is
    scaled by a power of two first, undone in the row's softmax scale).  q
    times 2^k with the attention scale times 2^-k gives the same scores, so the
    oracle's outputs for the unscaled q are the reference."""
    wl = inputs.random_case(41, 4, 32, 8, d, 16, torch.bfloat16, [1, 40, 700, 2100],
                            cache_dtype=torch.float8_e4m3fn, kv_scale=1.0 / 64)
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    out = torch.full(tuple(st.out.shape), float("nan"), dtype=torch.float32, device="cuda")
    q = st.q * 2.0 ** q_pow2                                  # exact: a power of two
    pa.pa_decode(out, q, st.k_cache, st.v_cache, st.block_tables, st.context_lens,
                 wl.scale * 2.0 ** -q_pow2, wl.block_size, st.workspace, **st.kv_scales)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert torch.isfinite(q.float()).all() and torch.equal(q.double() * 2.0 ** -q_pow2, st.q.double())
    assert max_err(out, oracle_decode(st)) <= 2e-3


def _fp8_prefill_case(seed, specs, n_q, n_kv, d, bs, act, scale, out_dtype=torch.float32,
                      v_scale=None, q_pow2=0):
    """specs: list of (cached tokens, chunk).  The context and the chunk go
    through the quantizing cache write; the oracle attends over the codes
    times the scale (v_scale for V when given).  q_pow2 = k multiplies q by
    2^k and the attention scale by 2^-k (the same scores)."""
    vsc = scale if v_scale is None else v_scale
    rng = np.random.default_rng(seed)
    R = len(specs)
    lens = [c + n for c, n in specs]
    nb = sum(-(-L // bs) for L in lens) + 5
    alloc = pa.Allocator(nb, rng.permutation(nb).astype(np.int32))
    mb = max(-(-L // bs) for L in lens)
    tables = alloc.build_tables(lens, mb, bs)
    g = torch.Generator().manual_seed(seed)
    ks = [torch.randn(L, n_kv, d, generator=g).to(act) for L in lens]
    vs = [torch.randn(L, n_kv, d, generator=g).to(act) for L in lens]
    qs = [(torch.randn(n, n_q, d, generator=g) * 2.0 ** q_pow2).to(act) for _, n in specs]
    att = float(np.float32(2.0 ** -q_pow2 / np.sqrt(d)))
    kc = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    vc = torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8,
                    device="cuda").view(torch.float8_e4m3fn)
    seq = np.concatenate([np.full(L, r, np.int32) for r, L in enumerate(lens)])
    pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    slots = torch.from_numpy(pa.pa_slot_mapping(tables, bs, seq, pos)).cuda()
    pa.pa_reshape_and_cache_quant(torch.cat(ks).cuda(), torch.cat(vs).cuda(), kc, vc, slots,
                                  k_scale=scale, v_scale=vsc)
    qsl = np.zeros(R + 1, np.int32)
    qsl[1:] = np.cumsum([n for _, n in specs])
    out = torch.full((int(qsl[-1]), n_q, d), float("nan"), dtype=out_dtype, device="cuda")
    pa.pa_prefill_chunk(out, torch.cat(qs).cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                        torch.from_numpy(qsl).cuda(),
                        torch.tensor(lens, dtype=torch.int32, device="cuda"),
                        max(n for _, n in specs), att, bs, k_scale=scale, v_scale=vsc)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    kd = [oracle.dequantize_fp8(oracle.quantize_fp8(x, scale), scale) for x in ks]
    vd = [oracle.dequantize_fp8(oracle.quantize_fp8(x, vsc), vsc) for x in vs]
    ref = np.concatenate(oracle.prefill(qs, kd, vd, att))
    return out, ref


PREFILL_CASES = [
    # seed, specs (ctx, chunk), n_q, n_kv, d, bs, act dtype, scale
    (21, [(0, 37)], 4, 4, 64, 16, torch.bfloat16, 1.0 / 64),                        # plain causal
    (22, [(0, 200), (100, 1), (33, 47)], 32, 8, 128, 16, torch.bfloat16, 1.0 / 64),  # ragged
    (23, [(500, 64), (0, 16), (16, 16)], 8, 1, 64, 32, torch.float16, 0.0125),       # MQA, bs 32
    (24, [(1000, 130)], 8, 8, 128, 32, torch.float16, 0.0125),                       # MHA, tail 106
    (25, [(47, 200), (1, 3), (300, 129)], 12, 4, 128, 32, torch.bfloat16, 1.0 / 64),  # g=3
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=[f"fp{c[0]}" for c in PREFILL_CASES])
def test_fp8_prefill_matches_oracle_on_dequantized_kv(case):
    out, ref = _fp8_prefill_case(*case)
    assert max_err(out, ref) <= 2e-3


def test_fp8_prefill_bf16_output_and_unequal_scales():
    out, ref = _fp8_prefill_case(26, [(300, 100), (0, 50)], 32, 8, 128, 16, torch.bfloat16,
                                 1.0 / 64, out_dtype=torch.bfloat16, v_scale=0.0125)
    got = out.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2e-3 + half_ulp(ref, torch.bfloat16))


@pytest.mark.parametrize("q_pow2", [24, -30])
def test_fp8_prefill_bf16_queries_outside_fp16_range(q_pow2):
    """bf16 queries far above fp16's largest value or below its smallest normal
    (the FP8 path multiplies on fp16 operands: each q row is scaled by a power
    of two first, undone in the row's softmax scale)."""
    out, ref = _fp8_prefill_case(27, [(200, 70), (0, 33)], 8, 2, 128, 16, torch.bfloat16,
                                 1.0 / 64, q_pow2=q_pow2)
    assert max_err(out, ref) <= 2e-3


def test_fp8_prefill_needs_scales():
    nb = 4
    kc = torch.zeros((nb, 2, 16, 64), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    vc = torch.zeros((nb, 2, 64, 16), dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    out = torch.empty((8, 4, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(pa.PAError) as e:   # no scales: refused on the host
        pa.pa_prefill_chunk(out, torch.zeros((8, 4, 64), dtype=torch.bfloat16, device="cuda"), kc, vc,
                            torch.zeros((1, 4), dtype=torch.int32, device="cuda"),
                            torch.tensor([0, 8], dtype=torch.int32, device="cuda"),
                            torch.tensor([8], dtype=torch.int32, device="cuda"), 8, 0.125, 16)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    assert pa.pa_get_device_error() == 0


@pytest.mark.parametrize("act", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("subnormal", [True, False], ids=["subnormal", "full-range"])
def test_fp8_prefill_widens_every_code_exactly(act, subnormal):
    """K = 0 makes attention uniform, so each output row is the plain mean of
    the visible V values; V holds E4M3 values (scale 1) that the quantizer
    keeps exactly: only subnormal codes (m * 2^-9), or codes of every
    exponent.  A widening that flushed or misplaced a code shows up here far
    above the fp32 rounding of the mean."""
    n_q, n_kv, d, bs, L = 8, 2, 128, 16, 300
    rng = np.random.default_rng(31 if subnormal else 32)
    if subnormal:
        v = rng.integers(-7, 8, size=(L, n_kv, d)) * 2.0 ** -9
    else:
        e = rng.integers(-6, 9, size=(L, n_kv, d)).astype(np.float64)
        m = rng.integers(0, 8, size=(L, n_kv, d))
        v = rng.choice([-1.0, 1.0], size=(L, n_kv, d)) * (1 + m / 8) * 2.0 ** e
        v = np.clip(v, -448.0, 448.0)                           # the largest finite code
    vt = torch.from_numpy(v).to(act)
    assert torch.equal(vt.double(), torch.from_numpy(v))       # exact in the activation dtype
    k = torch.zeros(L, n_kv, d, dtype=act)
    nb = -(-L // bs) + 2
    tables = np.arange(-(-L // bs), dtype=np.int32)[None, :]
    kc = torch.full((nb, n_kv, bs, d), 0x7F, dtype=torch.uint8, device="cuda").view(torch.float8_e4m3fn)
    vc = torch.full((nb, n_kv, bs // 16, d, 16), 0x7F, dtype=torch.uint8,
                    device="cuda").view(torch.float8_e4m3fn)
    slots = torch.from_numpy(pa.pa_slot_mapping(tables, bs, np.zeros(L, np.int32),
                                                np.arange(L, dtype=np.int32))).cuda()
    pa.pa_reshape_and_cache_quant(k.cuda(), vt.cuda(), kc, vc, slots, k_scale=1.0, v_scale=1.0)
    C = 70
    q = torch.randn(C, n_q, d, generator=torch.Generator().manual_seed(3)).to(act)
    out = torch.empty(C, n_q, d, dtype=torch.float32, device="cuda")
    pa.pa_prefill_chunk(out, q.cuda(), kc, vc, torch.from_numpy(tables).cuda(),
                        torch.tensor([0, C], dtype=torch.int32, device="cuda"),
                        torch.tensor([L], dtype=torch.int32, device="cuda"), C, 0.1, bs,
                        k_scale=1.0, v_scale=1.0)
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    got = out.cpu().numpy().astype(np.float64)
    g = n_q // n_kv
    for i in range(C):
        mean = v[:L - C + i + 1].mean(axis=0)                     # [n_kv][d]
        ref = np.repeat(mean, g, axis=0)
        bound = 1e-5 * (np.abs(v).max() if not subnormal else 2.0 ** -6)
        assert np.abs(got[i] - ref).max() <= bound, i


def test_fp8_mixed_workload_all_outputs():
    """The continuous-batching step over an FP8 pool: every decode output and
    every prefill row against the oracle on the dequantized K/V."""
    wl = inputs.get("mixed-llama3-8b-fp8")
    st = PagedStep(wl, out_dtype=torch.float32, prefill_out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert max_err(st.out, oracle_decode_all(st)) <= 2e-3
    assert max_err(st.p_out, oracle_prefill_all(st)) <= 2e-3
