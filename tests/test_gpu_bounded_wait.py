"""The error path of the kernels' bounded waits, run on the GPU without
faulting or hanging it: the test hook pkv_test_bounded_wait makes a CTA wait
on an mbarrier phase that nothing completes, with the same wait and drain the
decode kernels use.  The wait and the drain must give up within their limit
(time or poll count), report PKV_DEV_TIMEOUT | PKV_DEV_DRAIN_TIMEOUT, and
leave the context usable: a decode step afterwards matches the oracle."""
import time

import pytest
import torch

import paged_kv_cache_311_gb300 as pkv
from tests.gpu_support import TOL, gpu_decode, max_err, oracle_decode
from tests.util import small_case

pytestmark = pytest.mark.gpu

BOTH = pkv.DEV_TIMEOUT | pkv.DEV_DRAIN_TIMEOUT


def _timed_hook(limit_ns, max_polls):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    a.record()
    pkv.bounded_wait_hook(st, limit_ns, max_polls)
    b.record()
    torch.cuda.synchronize()
    return int(st.item()), a.elapsed_time(b), time.perf_counter() - t0


def test_wait_gives_up_at_its_time_limit():
    status, ms, wall = _timed_hook(1_000_000, 0)          # 1 ms limit, default poll cap
    assert status == BOTH
    assert 1.0 <= ms < 1000.0 and wall < 5.0               # the wait and the drain, then return


def test_wait_gives_up_at_its_poll_cap():
    """A cap of 4096 polls ends the wait long before a 2 s time limit."""
    status, ms, wall = _timed_hook(2_000_000_000, 4096)
    assert status == BOTH
    assert ms < 500.0 and wall < 5.0


def test_context_still_usable_after_a_timeout():
    status, _, _ = _timed_hook(1_000_000, 0)
    assert status == BOTH
    case = small_case(77, dtype="bf16", B=3, H=8, Hk=2, D=128, bs=16, lens=(5, 700, 1500))
    ref, st = oracle_decode(case)
    assert st == 0
    for P in (0, 512):
        got, gst, _ = gpu_decode(case, partition_size=P)
        assert gst == 0
        assert max_err(got, ref) <= TOL["bf16"]


def test_hook_rejects_bad_arguments():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for limit in (0, 2_000_000_001):
        with pytest.raises(pkv.PkvError):
            pkv.bounded_wait_hook(st, limit)
    torch.cuda.synchronize()
    assert st.item() == 0
