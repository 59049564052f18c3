"""The fused kernels' mbarrier waits are bounded: a wait that runs out
records RA_ERR_TIMEOUT for the host and returns, and the context stays
usable.  The wait is made to run out on purpose with the library's
self-test kernel (an mbarrier expecting bytes that no copy delivers) -- no
fault, no hang, no memory touched."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


def test_expired_wait_is_reported_and_the_context_survives():
    torch.cuda.synchronize()
    assert ra.ra_check_device_errors() == 0  # nothing recorded (and cleared)
    ra.ra_selftest_wait_timeout(20_000)  # 20 ms limit
    torch.cuda.synchronize()
    assert ra.ra_check_device_errors() == 5  # RA_ERR_TIMEOUT
    assert ra.ra_check_device_errors() == 0  # the check cleared it
    # the context still works: a normal call is bit-exact and reports nothing
    n, p = 4, 100_003
    host = [synth.normal_f32(3, k, 1.0, 0, p) for k in range(n)]
    want = [h.copy() for h in host]
    oracle.ring_allreduce_avg_f32(want)
    rows = [torch.from_numpy(h).cuda() for h in host]
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    for r in rows:
        np.testing.assert_array_equal(r.cpu().numpy().view(np.uint32), want[0].view(np.uint32))
    assert ra.ra_check_device_errors() == 0


def test_selftest_rejects_out_of_range_limits():
    for bad in (0, -5, 10_000_001):
        with pytest.raises(ra.RaError):
            ra.ra_selftest_wait_timeout(bad)
