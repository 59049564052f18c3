"""ra_allreduce_avg_staged_static: the staged ring for callers that cannot
allocate device memory (for example a plug-in whose host framework owns all
device memory through its own pool, or a loop that must not pay for the
device synchronisation cudaMalloc implies).  Its bf16 partial sums live in a
scratch array compiled into the library instead of a caller workspace.

Called through the C ABI (ctypes), its output must equal, bit for bit, the
output of the workspace entry point ra_allreduce_avg_staged on the same
inputs -- checked on two calls in a row, so the second call starts with the
first call's leftovers in the shared scratch array -- and the CPU oracle's
ring.  A warmed-up call must leave the device's free memory and torch's
allocator untouched: the call exists for callers that cannot allocate.
This file is collected last and also passes alone in a fresh process.
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
    """n device rows of p elements; `pad` is one element offset for every
    row, or a list with one offset per row (rows that disagree modulo 16
    bytes)."""
    out = []
    for k in range(n):
        if bf16:
            h = torch.from_numpy(synth.student_t3_bf16(seed, k, 1e-3, 0, p).view(np.int16)).view(torch.bfloat16)
        else:
            h = torch.from_numpy(synth.normal_f32(seed, k, 1e-3, 0, p))
        base = torch.empty(p + 16, dtype=h.dtype, device="cuda")
        off = pad[k % len(pad)] if isinstance(pad, list) else pad
        t = base[off:off + p]
        t.copy_(h)
        out.append(t)
    return out


@pytest.mark.parametrize("dtype,n,p,pad", [("bf16", 8, 1_000_003, 0), ("bf16", 16, ra.RA_STAGED_STATIC_MAX_P, 0),
                                           ("bf16", 5, 77_777, 3), ("f32", 8, 1_000_003, 1),
                                           ("bf16", 4, 300_001, [0, 1, 2, 3]), ("bf16", 6, 65_537, [5, 0, 3])])
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


def _host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("n,p,pad", [(8, ra.RA_STAGED_STATIC_MAX_P, 0), (5, 1_000_003, 3), (4, 262_147, [0, 1, 2, 3])])
def test_matches_the_oracle(n, p, pad):
    import oracle
    for seed in (303, 404):  # two calls in a row on the shared scratch array
        rows = _rows(n, p, True, seed, pad)
        want = [_host_bits(r) for r in rows]
        oracle.ring_allreduce_avg_bf16(want)
        ra.ra_allreduce_avg_staged_static(rows)
        torch.cuda.synchronize()
        for k, r in enumerate(rows):
            np.testing.assert_array_equal(_host_bits(r), want[k], err_msg="worker %d, seed %d" % (k, seed))


def test_allocates_no_device_memory():
    # Inputs made and the call warmed up first (its first call on a device
    # looks up the scratch array's address); then further calls must change
    # neither the device's free memory nor what torch's allocator holds.
    rows = _rows(8, ra.RA_STAGED_STATIC_MAX_P, True, 505)
    ra.ra_allreduce_avg_staged_static(rows)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0, reserved0 = torch.cuda.memory_allocated(), torch.cuda.memory_reserved()
    for _ in range(5):
        ra.ra_allreduce_avg_staged_static(rows)
        torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "device free memory changed by %d bytes" % (free0 - free1)
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.memory_reserved() == reserved0
