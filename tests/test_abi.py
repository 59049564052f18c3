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


def test_every_call_rejects_bad_arguments_on_the_host(lib):
    # fake, never-dereferenced addresses: each case fails an argument check
    # before the library touches CUDA
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    P = ctypes.POINTER
    INVALID, UNSUPPORTED, OVERLAP = 1, 2, 3
    F32, BF16 = 0, 1
    rows = (vp * 4)(0x100000, 0x200000, 0x300000, 0x400000)   # 1 MiB apart
    # every case below must fail its argument check: none may reach a launch
    p = 1000

    lib.ra_reduce_scatter_avg.argtypes = [P(vp), ctypes.c_int, i64, ctypes.c_int, P(vp), vp]
    lib.ra_all_gather.argtypes = [P(vp), ctypes.c_int, i64, ctypes.c_int, P(vp), vp]
    # shards: shard m holds chunk (m+1) mod 4 of 250 elements
    ov = (vp * 4)(0x900000, 0x900000 + 400, 0xA00000, 0xB00000)      # first two overlap
    assert lib.ra_reduce_scatter_avg(rows, 4, p, F32, ov, None) == OVERLAP
    assert lib.ra_all_gather(rows, 4, p, F32, ov, None) == OVERLAP
    into_rows = (vp * 4)(0x100000 + 64, 0xA00000, 0xB00000, 0xC00000)  # inside worker 0's array
    assert lib.ra_reduce_scatter_avg(rows, 4, p, F32, into_rows, None) == OVERLAP
    odd = (vp * 4)(0x900001, 0xA00000, 0xB00000, 0xC00000)             # not element-aligned
    assert lib.ra_reduce_scatter_avg(rows, 4, p, F32, odd, None) == INVALID
    nul = (vp * 4)(0, 0xA00000, 0xB00000, 0xC00000)
    assert lib.ra_all_gather(rows, 4, p, F32, nul, None) == INVALID

    class Bucket(ctypes.Structure):
        _fields_ = [("offset", i64), ("count", i64)]
    lib.ra_allreduce_avg_buckets.argtypes = [P(vp), ctypes.c_int, ctypes.c_int, P(Bucket), ctypes.c_int, vp]
    b = (Bucket * 2)(Bucket(0, 600), Bucket(500, 100))                  # overlap
    assert lib.ra_allreduce_avg_buckets(rows, 4, F32, b, 2, None) == OVERLAP
    b = (Bucket * 1)(Bucket(-1, 10))
    assert lib.ra_allreduce_avg_buckets(rows, 4, F32, b, 1, None) == INVALID
    b = (Bucket * 1)(Bucket(0, 300000))                                 # 1.2 MB rows, 1 MiB apart: overlap
    assert lib.ra_allreduce_avg_buckets(rows, 4, F32, b, 1, None) == OVERLAP

    class Traffic(ctypes.Structure):
        _fields_ = [("sent", i64), ("received", i64)]
    lib.ra_allreduce_avg_staged.argtypes = [P(vp), ctypes.c_int, i64, ctypes.c_int, vp, ctypes.c_size_t,
                                            P(Traffic), vp]
    lib.ra_staged_workspace_bytes.restype = ctypes.c_size_t
    need = lib.ra_staged_workspace_bytes(4, i64(p), BF16)
    assert lib.ra_allreduce_avg_staged(rows, 4, p, BF16, vp(0x900000), need - 1, None, None) == INVALID
    assert lib.ra_allreduce_avg_staged(rows, 4, p, BF16, None, need, None, None) == INVALID
    assert lib.ra_allreduce_avg_staged(rows, 4, p, BF16, vp(0x200000 + 16), need, None, None) == OVERLAP

    lib.ra_allreduce_avg_staged_static.argtypes = [P(vp), ctypes.c_int, i64, ctypes.c_int, P(Traffic), vp]
    far = (vp * 2)(0x10000000, 0x20000000)
    assert lib.ra_allreduce_avg_staged_static(far, 2, 4194304 + 1, BF16, None, None) == UNSUPPORTED

    lib.ra_allreduce_avg_host.argtypes = [P(vp), P(vp), ctypes.c_int, i64, ctypes.c_int, ctypes.c_int, vp]
    assert lib.ra_allreduce_avg_host(rows, None, 4, p, F32, 7, None) == INVALID     # mode
    assert lib.ra_allreduce_avg_host(None, None, 4, p, F32, 0, None) == INVALID

    lib.ra_reducer_create.argtypes = [P(vp), ctypes.c_int, ctypes.c_int, P(i64), ctypes.c_int, i64, P(vp)]
    h = vp()
    numel = (i64 * 2)(400, 600)
    assert lib.ra_reducer_create(rows, 4, F32, numel, 2, 0, ctypes.byref(h)) == INVALID          # cap
    assert lib.ra_reducer_create(rows, 4, 9, numel, 2, 1024, ctypes.byref(h)) == INVALID          # dtype
    big = (i64 * 2)(400, 300000)
    assert lib.ra_reducer_create(rows, 4, F32, big, 2, 1024, ctypes.byref(h)) == OVERLAP          # rows overlap
    assert lib.ra_reducer_create(rows, 4, F32, numel, 2, 1024, None) == INVALID

    lib.ra_bucket_plan.argtypes = [P(i64), ctypes.c_int, ctypes.c_int, i64, P(Bucket), ctypes.c_int,
                                   P(ctypes.c_int)]
    out = (Bucket * 1)()
    nb = ctypes.c_int(0)
    three = (i64 * 3)(100, 100, 100)
    assert lib.ra_bucket_plan(three, 3, 4, 400, out, 1, ctypes.byref(nb)) == INVALID              # max_out too small
    lib.ra_selftest_wait_timeout.argtypes = [ctypes.c_int, vp]
    assert lib.ra_selftest_wait_timeout(0, None) == INVALID


def test_bounds_selftest_on_the_host(lib):
    # the product library checks the arguments, then answers the bounds
    # self-test with RA_ERR_UNSUPPORTED (only the checked build runs it);
    # none of these reaches CUDA
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.ra_selftest_bounds_check.argtypes = [ctypes.POINTER(vp), ctypes.c_int, i64, ctypes.c_int, vp]
    INVALID, UNSUPPORTED, OVERLAP = 1, 2, 3
    rows = (vp * 2)(0x100000, 0x200000)
    assert lib.ra_selftest_bounds_check(None, 2, 1000, 0, None) == INVALID
    assert lib.ra_selftest_bounds_check(rows, 1, 1000, 0, None) == INVALID      # n < 2
    assert lib.ra_selftest_bounds_check(rows, 2, 1, 0, None) == INVALID         # p < 2
    assert lib.ra_selftest_bounds_check(rows, 2, 300000, 0, None) == OVERLAP    # 1.2 MB rows 1 MiB apart
    assert lib.ra_selftest_bounds_check(rows, 2, 1000, 0, None) == UNSUPPORTED
    lib.ra_status_str.restype = ctypes.c_char_p
    assert lib.ra_status_str(6) == b"RA_ERR_BOUNDS"


C_PROGRAM = r"""
#include <stdio.h>
#include "ring_allreduce.h"

int main(void) {
    int64_t b, e;
    ra_bucket plan[8];
    int nb = 0, k;
    int64_t numel[5] = {100, 200, 300, 50, 7};
    void *bufs[2];
    ra_chunk_range(1048579, 4, 3, &b, &e);
    printf("chunk %lld %lld\n", (long long)b, (long long)e);
    if (ra_bucket_plan(numel, 5, 4, 1000, plan, 8, &nb) != RA_OK) return 2;
    printf("buckets %d", nb);
    for (k = 0; k < nb; ++k) printf(" %lld:%lld", (long long)plan[k].offset, (long long)plan[k].count);
    printf("\n");
    bufs[0] = (void *)0x100000;
    bufs[1] = (void *)0x100020;  /* 40-byte rows 32 bytes apart */
    printf("overlap %d\n", (int)ra_allreduce_avg(bufs, 2, 10, RA_F32, NULL));
    printf("%s\n", ra_status_str(RA_ERR_BOUNDS));
    return 0;
}
"""


def test_the_header_is_c_and_links(lib):
    # a C99 program against the header and the library, host-only calls
    import subprocess
    import oracle
    d = os.path.join(ROOT, "tests", ".scratch", "c_abi")
    os.makedirs(d, exist_ok=True)
    src, exe = os.path.join(d, "abi.c"), os.path.join(d, "abi")
    with open(src, "w") as f:
        f.write(C_PROGRAM)
    libdir = os.path.join(ROOT, "gradient_ring_all_gb300", "lib")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                        os.path.join(ROOT, "include"), src, "-o", exe, "-L", libdir, "-lgradient_ring_all",
                        "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    lines = out.stdout.split("\n")
    assert lines[0] == "chunk 786435 1048579"
    want = oracle.bucket_plan([100, 200, 300, 50, 7], 4, 1000)
    assert lines[1] == "buckets %d" % len(want) + "".join(" %d:%d" % (o, c) for o, c in want)
    assert lines[2] == "overlap 3"
    assert lines[3] == "RA_ERR_BOUNDS"
    import shutil
    shutil.rmtree(d, ignore_errors=True)
