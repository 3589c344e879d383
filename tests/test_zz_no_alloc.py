"""pa_decode_no_alloc: decode for callers that cannot allocate device memory.

Such callers (a host runtime that gives all free HBM to its KV block pool and
offers plugins no allocator, or a latency-critical loop that cannot pay for
cudaMalloc's synchronisation) pass only inputs and outputs; the split-K scratch
is a fixed array inside the library.  This file is collected last on purpose.
Its checks: through the C ABI, two calls in a row each match pa_decode with a
caller workspace, and the CPU oracle's fp64 attention, within the decode
tolerance; a batch too large for the fixed scratch is refused before anything
runs.
"""
import pytest
import torch

from paged_kv_cache_25_gb300 import binding as pa
from paged_kv_cache_25_gb300 import inputs
from paged_kv_cache_25_gb300.step import PagedStep
from tests.helpers import TOL, max_err, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_25_gb300 import build
    build.build()
    assert pa.pa_get_device_error() == 0


def test_no_alloc_matches_workspace_decode_twice():
    wl = inputs.random_case(71, 8, 32, 8, 128, 16, torch.bfloat16,
                            [4000, 17, 512, 513, 2049, 1, 3000, 900])
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    need = pa.pa_decode_workspace_size(wl.batch, wl.n_q_heads, wl.n_kv_heads, wl.head_dim,
                                       wl.block_size, st.max_blocks * wl.block_size)
    assert 0 < need <= pa.PA_DECODE_NO_ALLOC_SCRATCH_BYTES
    ref = st.out.clone()
    exact = oracle_decode(st)                # fp64 attention of the same inputs
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        pa.pa_decode_no_alloc(out, st.q, st.k_cache, st.v_cache, st.block_tables,
                              st.context_lens, wl.scale, wl.block_size)
        torch.cuda.synchronize()
        assert pa.pa_get_device_error() == 0
        assert float((out - ref).abs().max()) <= TOL[wl.dtype]
        assert max_err(out, exact) <= TOL[wl.dtype]


def test_no_alloc_rejects_batches_beyond_its_scratch():
    wl = inputs.random_case(72, 2, 32, 8, 128, 16, torch.bfloat16, [100, 200])
    st = PagedStep(wl, out_dtype=torch.float32)
    n_seq, max_blocks = 256, 256             # would need ~33 MB of scratch
    need = pa.pa_decode_workspace_size(n_seq, 32, 8, 128, 16, max_blocks * 16)
    assert need > pa.PA_DECODE_NO_ALLOC_SCRATCH_BYTES
    q = torch.zeros((n_seq, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((n_seq, 32, 128), dtype=torch.float32, device="cuda")
    bt = torch.zeros((n_seq, max_blocks), dtype=torch.int32, device="cuda")
    cl = torch.ones(n_seq, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_decode_no_alloc(out, q, st.k_cache, st.v_cache, bt, cl, wl.scale, 16)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    assert "scratch" in str(e.value)
    assert pa.pa_get_device_error() == 0
