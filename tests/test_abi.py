"""The C-ABI library: it loads, exports every symbol the public header
declares, and its host-only calls (no GPU needed) behave as documented."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from gradient_ring_all_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def _declared(header):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(ra_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            names += _declared(os.path.join(ROOT, "include", h))
    assert "ra_allreduce_avg" in names and "ra_bucket_plan" in names
    for nm in names:
        assert hasattr(lib, nm), nm


def test_host_only_calls():
    import gradient_ring_all_gb300 as ra
    import oracle
    for p, n in [(1_048_579, 4), (17, 5), (3, 8), (0, 1)]:
        for c in range(n):
            assert ra.ra_chunk_range(p, n, c) == oracle.chunk_range(p, n, c)
    assert ra.ra_status_str(0) == "RA_OK" and ra.ra_status_str(3) == "RA_ERR_OVERLAP"
    assert ra.ra_staged_workspace_bytes(4, 1000, ra.RA_F32) == 0
    assert ra.ra_staged_workspace_bytes(4, 1000, ra.RA_BF16) >= 4000
    import synth
    wl = synth.WORKLOADS["transformer24_buckets_n4_f32"]
    plan = ra.ra_bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes)
    assert plan == oracle.bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes)
    assert len(plan) == 98
    for numel, eb, cap in [([10, 20, 30, 40], 4, 200), ([10, 50], 4, 200), ([], 4, 8), ([5, 100, 5], 2, 100),
                           (list(range(50)), 4, 64)]:
        assert ra.ra_bucket_plan(numel, eb, cap) == oracle.bucket_plan(numel, eb, cap)


def test_bad_arguments_are_rejected_before_any_launch(lib):
    # these fail argument checks on the host; nothing reaches the GPU
    vp = ctypes.c_void_p
    lib.ra_allreduce_avg.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64, ctypes.c_int, vp]
    lib.ra_allreduce_sgd.argtypes = [ctypes.POINTER(vp), ctypes.c_int, ctypes.c_int64, ctypes.c_int, vp,
                                     ctypes.c_float, vp]
    bufs = (vp * 4)(0x10000, 0x20000, 0x30000, 0x40000)
    INVALID, OVERLAP = 1, 3
    assert lib.ra_allreduce_avg(bufs, 0, 10, 0, None) == INVALID          # n < 1
    assert lib.ra_allreduce_avg(bufs, 65, 10, 0, None) == INVALID         # n > RA_MAX_N
    assert lib.ra_allreduce_avg(bufs, 4, -1, 0, None) == INVALID          # p < 0
    assert lib.ra_allreduce_avg(bufs, 4, 10, 7, None) == INVALID          # dtype
    assert lib.ra_allreduce_avg(None, 4, 10, 0, None) == INVALID          # bufs
    nul = (vp * 2)(0x10000, 0)
    assert lib.ra_allreduce_avg(nul, 2, 10, 0, None) == INVALID           # null row
    odd = (vp * 2)(0x10001, 0x20000)
    assert lib.ra_allreduce_avg(odd, 2, 10, 0, None) == INVALID           # misaligned element
    ov = (vp * 2)(0x10000, 0x10020)
    assert lib.ra_allreduce_avg(ov, 2, 10, 0, None) == OVERLAP            # 40-byte rows 32 bytes apart
    assert lib.ra_allreduce_sgd(bufs, 4, 10, 0, None, ctypes.c_float(0.1), None) == INVALID  # w null
    assert lib.ra_allreduce_sgd(bufs, 4, 10, 0, vp(0x10010), ctypes.c_float(0.1), None) == OVERLAP
    # p == 0 and n == 1 are no-ops that succeed without touching the device
    assert lib.ra_allreduce_avg(bufs, 4, 0, 0, None) == 0
    assert lib.ra_allreduce_avg(bufs, 1, 10, 0, None) == 0
