"""ra_allreduce_avg_staged_static: the staged ring for callers that cannot
allocate device memory (for example a plug-in whose host framework owns all
device memory through its own pool, or a loop that must not pay for the
device synchronisation cudaMalloc implies).  Its bf16 partial sums live in a
scratch array compiled into the library instead of a caller workspace.

Called through the C ABI (ctypes), its output must equal, bit for bit, the
output of the workspace entry point ra_allreduce_avg_staged on the same
inputs -- checked on two calls in a row, so the second call starts with the
first call's leftovers in the shared scratch array.  This file is collected
last and also passes alone in a fresh process.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


def _rows(n, p, bf16, seed, pad=0):
    out = []
    for k in range(n):
        if bf16:
            h = torch.from_numpy(synth.student_t3_bf16(seed, k, 1e-3, 0, p).view(np.int16)).view(torch.bfloat16)
        else:
            h = torch.from_numpy(synth.normal_f32(seed, k, 1e-3, 0, p))
        base = torch.empty(p + 16, dtype=h.dtype, device="cuda")
        t = base[pad:pad + p]
        t.copy_(h)
        out.append(t)
    return out


@pytest.mark.parametrize("dtype,n,p,pad", [("bf16", 8, 1_000_003, 0), ("bf16", 16, ra.RA_STAGED_STATIC_MAX_P, 0),
                                           ("bf16", 5, 77_777, 3), ("f32", 8, 1_000_003, 1)])
def test_matches_workspace_entry_point_on_two_calls(dtype, n, p, pad):
    bf16 = dtype == "bf16"
    for call, seed in enumerate((101, 202)):
        a = _rows(n, p, bf16, seed, pad)
        b = _rows(n, p, bf16, seed, pad)
        traffic_a = ra.ra_allreduce_avg_staged_static(a)
        traffic_b = ra.ra_allreduce_avg_staged(b)
        torch.cuda.synchronize()
        assert traffic_a == traffic_b
        for x, y in zip(a, b):
            # bit-exact, as every parity test here
            assert torch.equal(x.view(torch.int16 if bf16 else torch.int32),
                               y.view(torch.int16 if bf16 else torch.int32)), "call %d differs" % call
        for x in a[1:]:
            assert torch.equal(a[0], x)


def test_rejects_sizes_beyond_the_scratch():
    lib = ra.load()
    p = ra.RA_STAGED_STATIC_MAX_P + 1
    rows = [torch.empty(p, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    arr = (ctypes.c_void_p * 2)(*[r.data_ptr() for r in rows])
    st = lib.ra_allreduce_avg_staged_static(arr, 2, p, ra.RA_BF16, None, None)
    assert ra.ra_status_str(st) == "RA_ERR_UNSUPPORTED"
