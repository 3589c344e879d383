"""Failure detection without a GPU fault: a bounded wait that runs out records
PA_ERR_TIMEOUT, the kernel returns, and the context keeps working."""
import time

import pytest
import torch

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


def test_wait_that_never_completes_times_out_and_context_survives():
    scratch = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    pa.pa_selftest_bounded_wait(20_000, scratch)          # 20 ms limit
    assert pa.pa_get_device_error() == pa.PA_ERR_TIMEOUT   # synchronizes the stream
    elapsed = time.perf_counter() - t0
    assert int(scratch.item()) == 2                        # the kernel went on after giving up
    assert 0.015 < elapsed < 5.0
    assert pa.pa_get_device_error() == 0                   # the word was cleared
    # the context is still usable: a decode right after is correct
    wl = inputs.random_case(81, 2, 8, 2, 64, 16, torch.bfloat16, [100, 700])
    st = PagedStep(wl, out_dtype=torch.float32)
    st.step()
    torch.cuda.synchronize()
    assert pa.pa_get_device_error() == 0
    assert max_err(st.out, oracle_decode(st)) <= 2e-3


def test_selftest_argument_checks():
    scratch = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PAError):
        pa.pa_selftest_bounded_wait(0, scratch)
    with pytest.raises(pa.PAError):
        pa.pa_selftest_bounded_wait(10, None)
