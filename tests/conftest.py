import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session", autouse=True)
def _build_host_libs():
    import oracle
    import synth
    oracle.build()
    synth.build()


@pytest.fixture(autouse=True)
def _no_device_error_record(request):
    # After every GPU test, in the product build and in the bounds-checked
    # build (GRADIENT_RING_ALL_CHECKED=1): no kernel left a record in the
    # device's error word -- neither a bounded wait that gave up
    # (RA_ERR_TIMEOUT: that block skipped its stores) nor, in the checked
    # build, an access outside the caller's buffers (RA_ERR_BOUNDS).  Tests
    # that cause a record on purpose read and clear it themselves.
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    import gradient_ring_all_gb300 as ra
    if ra._lib is None:  # the test never loaded the library
        return
    torch.cuda.synchronize()
    st = ra.ra_check_device_errors()
    assert st == ra.RA_OK, "a kernel left a device error record: %s" % ra.ra_status_str(st)
