"""Failure detection without a GPU fault.

Every wait in the library's kernels (cross-CTA completion counters, mbarrier phases of the
operand, accumulator and C rings) is bounded: when it runs out the kernel ORs
GNS_DEVST_TIMEOUT into the device status word and returns, so the context stays usable.
gns_selftest_bounded_wait runs those same wait helpers with a short limit on a counter that
nothing increments and an mbarrier phase that nothing completes. The Python API reports
what the GPU flags when the caller passes no status word of its own.
"""
import ctypes
import time

import pytest

torch = pytest.importorskip("torch")
gns = pytest.importorskip("matrix_orthogonalizing_optimizer_gb300")
from matrix_orthogonalizing_optimizer_gb300 import _lib  # noqa: E402

pytestmark = pytest.mark.gpu

LIMIT_US = 20000  # 20 ms per wait


def _run(counter, target):
    lib = _lib.load()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    rc = lib.gns_selftest_bounded_wait(counter.data_ptr(), target, LIMIT_US, st.data_ptr(), out.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0, _lib.last_error()
    torch.cuda.synchronize()
    return int(st.item()), [int(v) for v in out.cpu()], time.perf_counter() - t0


def test_unreachable_counter_and_mbarrier_time_out():
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")   # nothing increments it
    st, (ns, ok), wall = _run(counter, 1)
    assert st == _lib.GNS_DEVST_TIMEOUT
    assert ok == 0                                               # neither wait succeeded
    assert 2 * LIMIT_US * 1000 <= ns < 10 * LIMIT_US * 1000      # each ran its limit, no longer
    assert wall < 5.0
    # the context is still usable: a real call right after gives a finite, flag-free result
    x = (torch.randn((2, 128, 512), device="cuda") / 512 ** 0.5).to(torch.bfloat16)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gns.gram_ns_batched(x, status=st2)[0]
    torch.cuda.synchronize()
    assert int(st2.item()) == 0 and bool(torch.isfinite(out.float()).all())


def test_reached_counter_passes_and_only_the_mbarrier_times_out():
    counter = torch.full((1,), 5, dtype=torch.int32, device="cuda")
    st, (ns, ok), _ = _run(counter, 5)
    assert st == _lib.GNS_DEVST_TIMEOUT and ok == 1
    assert LIMIT_US * 1000 <= ns < 2 * LIMIT_US * 1000


def test_argument_errors_enqueue_nothing():
    lib = _lib.load()
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.gns_selftest_bounded_wait(None, 1, LIMIT_US, None, None, s) == _lib.GNS_ERR_INVALID
    assert lib.gns_selftest_bounded_wait(counter.data_ptr(), 1, 0, None, None, s) == _lib.GNS_ERR_INVALID
    assert lib.gns_selftest_bounded_wait(counter.data_ptr(), 1, 3000000, None, None, s) == _lib.GNS_ERR_INVALID


def test_api_reports_device_flags_by_default():
    """A call without status= checks the API's own word after synchronising: the non-finite
    flag of an Inf input surfaces as GnsDeviceError; with check=False it stays in the word
    until check_status() reports it; a caller's own status tensor is left to the caller."""
    x = (torch.randn((1, 64, 256), device="cuda") / 16).to(torch.bfloat16)
    bad = x.clone()
    bad[0, 3, 7] = float("inf")
    with pytest.raises(gns.GnsDeviceError, match="non-finite"):
        gns.gram_ns_batched(bad)
    gns.gram_ns_batched(x)                      # reported and cleared: the next call is clean
    gns.gram_ns_batched(bad, check=False)       # no sync, no raise ...
    with pytest.raises(gns.GnsDeviceError):     # ... until the word is checked
        gns.check_status()
    gns.check_status()
    mine = torch.zeros(1, dtype=torch.int32, device="cuda")
    gns.gram_ns_batched(bad, status=mine)       # the caller's word: no raise
    torch.cuda.synchronize()
    assert int(mine.item()) == _lib.GNS_DEVST_NONFINITE
    with pytest.raises(gns.GnsDeviceError):
        gns.check_status(mine)
    assert int(mine.item()) == 0
