"""The bounds-checked build (libgradient_ring_all_checked.so): every kernel
verifies, before each global access, that the range lies inside the
caller's buffer it belongs to, skips it otherwise and records RA_ERR_BOUNDS.

1. The check fires: ra_selftest_bounds_check runs the fused all-reduce with
   the kernel told that the rows are one element shorter than the ring's
   segments, and RA_ERR_BOUNDS must be reported (nothing outside the rows is
   touched either way).
2. No entry point reads or writes outside the caller's buffers: the parity,
   fuzz, guard-band, graph and variant suites run again against the checked
   build; a conftest fixture fails any test that leaves a bounds record.

Each part runs in a child process, since the checked library is chosen when
the binding is imported."""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ENV = dict(os.environ, GRADIENT_RING_ALL_CHECKED="1")

SELFTEST = r"""
import sys
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
from gradient_ring_all_gb300 import build
build.build(checked=True)
import gradient_ring_all_gb300 as ra
import oracle, synth
assert ra.CHECKED
for dtype, layout in (("f32", "separate"), ("bf16", "separate"), ("f32", "strided")):
    n, p = 4, 100_003
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    if layout == "strided":
        big = torch.zeros(n * (p + 1), dtype=tdt, device="cuda")
        rows = [big[k * (p + 1):k * (p + 1) + p] for k in range(n)]
    else:
        rows = [torch.zeros(p, dtype=tdt, device="cuda") for _ in range(n)]
    torch.cuda.synchronize()
    assert ra.ra_check_device_errors() == ra.RA_OK
    ra.ra_selftest_bounds_check(rows)
    torch.cuda.synchronize()
    assert ra.ra_check_device_errors() == ra.RA_ERR_BOUNDS, (dtype, layout)
    assert ra.ra_check_device_errors() == ra.RA_OK  # cleared
# a correct call afterwards: bit-exact, nothing recorded
host = [synth.normal_f32(9, k, 1.0, 0, 100_003) for k in range(4)]
want = [h.copy() for h in host]
oracle.ring_allreduce_avg_f32(want)
rows = [torch.from_numpy(h).cuda() for h in host]
ra.ra_allreduce_avg(rows)
torch.cuda.synchronize()
for r in rows:
    np.testing.assert_array_equal(r.cpu().numpy().view(np.uint32), want[0].view(np.uint32))
assert ra.ra_check_device_errors() == ra.RA_OK
print("checked selftest: ok")
"""


def test_the_bounds_check_fires():
    r = subprocess.run([sys.executable, "-c", SELFTEST, ROOT], env=ENV, cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "checked selftest: ok" in r.stdout


def test_every_entry_point_stays_inside_the_callers_buffers():
    suites = ["tests/test_gpu_parity.py", "tests/test_gpu_fuzz.py", "tests/test_gpu_guards.py",
              "tests/test_gpu_graph.py", "tests/test_gpu_variants.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", *suites, "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider"],
                       env=ENV, cwd=ROOT, capture_output=True, text=True, timeout=3000)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])


def test_the_product_build_has_no_bounds_check():
    # the product library answers the self-test with RA_ERR_UNSUPPORTED
    code = ("import sys; sys.path.insert(0, sys.argv[1]); import torch; "
            "from gradient_ring_all_gb300 import build; build.build(checked=False); "
            "import gradient_ring_all_gb300 as ra; assert not ra.CHECKED; "
            "rows = [torch.zeros(10, device='cuda') for _ in range(2)]\n"
            "try:\n    ra.ra_selftest_bounds_check(rows)\nexcept ra.RaError as e:\n    assert e.status == 2; print('ok')")
    env = {k: v for k, v in os.environ.items() if k != "GRADIENT_RING_ALL_CHECKED"}
    r = subprocess.run([sys.executable, "-c", code, ROOT], env=env, cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and "ok" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])
