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
def _no_out_of_bounds_access(request):
    # Under the bounds-checked build (GRADIENT_RING_ALL_CHECKED=1) every GPU
    # test must leave no record of a kernel touching memory outside the
    # caller's buffers.
    yield
    if os.environ.get("GRADIENT_RING_ALL_CHECKED") != "1" or request.node.get_closest_marker("gpu") is None:
        return
    import torch
    import gradient_ring_all_gb300 as ra
    torch.cuda.synchronize()
    assert ra.ra_check_device_errors() != ra.RA_ERR_BOUNDS, "a kernel accessed memory outside the caller's buffers"
