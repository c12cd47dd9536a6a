"""The time limit on the kernels' barrier waits, exercised on the GPU (needs a GB300).

Every wait of the library's kernels on a shared-memory barrier gives up after
a time limit, sets bit 0 of the device error flags and lets the kernel end;
once the bit is set, later waits give up at their first check of it. The
self-test entry point runs exactly that wait (bounded_wait) on a barrier that
nothing arrives on, with a 2 ms limit: no fault, no trap, no hang. The test
then checks that the host reads the bit, that reading clears it, and that the
layer's kernels run correctly afterwards.
"""
import pytest

import gated_ssm_temporal_gb300 as g
from gated_ssm_temporal_gb300.workloads import Workload, make_inputs
from gpu_helpers import NAMES_ALL, ensure_built, oracle_all, run_all, shape_of
from tolerance import assert_outputs

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000


def test_wait_gives_up_sets_the_flag_and_the_library_recovers():
    import torch
    ensure_built()
    assert g.m2scan_read_device_flags() == 0  # nothing before this test gave up
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    st = g.m2scan_selftest_wait_timeout(LIMIT_NS, out.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    assert st == g.M2SCAN_OK
    torch.cuda.synchronize()
    first_ns, second_ns, gave_up = (int(v) for v in out[:3].cpu())
    assert gave_up == 3, "both waits must give up (mask %d)" % gave_up
    # the first wait runs out its own limit (checked every 16 suspended
    # retries, so it ends within a fraction of a millisecond after it)
    assert LIMIT_NS <= first_ns < LIMIT_NS + 5_000_000, first_ns
    # the second sees the bit at its first check, long before its own limit
    assert second_ns < LIMIT_NS // 2, second_ns
    assert g.m2scan_read_device_flags() == 1  # bit 0, read by the host ...
    assert g.m2scan_read_device_flags() == 0  # ... and cleared by that read
    # the layer's kernels wait normally again
    x = make_inputs(Workload("after_timeout", 300, 8, 256, 16, 0.1, 77))
    got = run_all(x)
    assert_outputs(got, oracle_all(x), shape_of(x), NAMES_ALL)
    assert g.m2scan_read_device_flags() == 0


def test_selftest_rejects_bad_arguments():
    import torch
    ensure_built()
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    assert g.m2scan_selftest_wait_timeout(LIMIT_NS, 0, 0) == 1            # NULL
    assert g.m2scan_selftest_wait_timeout(LIMIT_NS, out.data_ptr() + 8, 0) == 3  # unaligned
    assert g.m2scan_selftest_wait_timeout(10, out.data_ptr(), 0) == 2       # limit out of range
    assert g.m2scan_selftest_wait_timeout(10**9, out.data_ptr(), 0) == 2
