"""The bf16-on-the-wire ring and the single-reducer average against the CPU
oracle, bit for bit, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth
from gpu_util import to_device_rows, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


SHAPES = [(1, 10), (2, 7), (3, 1000), (4, 1_048_579), (5, 4099), (8, 70_001), (16, 40_000), (17, 3001), (32, 4096),
          (64, 700)]


@pytest.mark.parametrize("layout", ["separate", "offset", "mixed"])
@pytest.mark.parametrize("n,p", SHAPES)
def test_bf16_wire_matches_oracle(n, p, layout):
    host = [synth.student_t3_bf16(700 + n, k, 1e-3, 0, p) for k in range(n)]
    want = [r.copy() for r in host]
    oracle.ring_allreduce_avg_bf16_wire(want)
    rows = to_device_rows(host, layout=layout, pad=3)
    ra.ra_allreduce_avg_bf16_wire(rows)
    torch.cuda.synchronize()
    for r in rows:
        np.testing.assert_array_equal(to_host(r), want[0])


def test_bf16_wire_differs_from_binary32_partials():
    vals = np.array([256.0, 1.0, 1.0], np.float32)
    host = [np.array([v], np.float32).view(np.uint32).astype(np.uint32) >> 16 for v in vals]
    host = [h.astype(np.uint16) for h in host]
    a = to_device_rows(host)
    b = to_device_rows(host)
    ra.ra_allreduce_avg_bf16_wire(a)
    ra.ra_allreduce_avg(b)
    torch.cuda.synchronize()
    assert float(a[0].float()[0]) == 85.5 and float(b[0].float()[0]) == 86.0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["separate", "offset", "mixed"])
@pytest.mark.parametrize("n,p", SHAPES)
def test_single_reducer_matches_oracle(n, p, dtype, layout):
    if dtype == "f32":
        host = [synth.normal_f32(800 + n, k, 1.0, 0, p) for k in range(n)]
    else:
        host = [synth.student_t3_bf16(800 + n, k, 1e-3, 0, p) for k in range(n)]
    want = [r.copy() for r in host]
    sent, recv = oracle.single_reducer_avg(want)
    rows = to_device_rows(host, layout=layout, pad=1)
    traffic = ra.ra_allreduce_avg_single_reducer(rows)
    torch.cuda.synchronize()
    for r in rows:
        got = to_host(r)
        np.testing.assert_array_equal(got.view(np.uint32) if dtype == "f32" else got,
                                      want[0].view(np.uint32) if dtype == "f32" else want[0])
    assert [t[0] for t in traffic] == sent.tolist() and [t[1] for t in traffic] == recv.tolist()
