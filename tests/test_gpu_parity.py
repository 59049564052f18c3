"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Integer-exact comparisons: the ring fixes the summation order, so every
output must equal the oracle's bit for bit (binary32 and bf16 alike).  The
binary64 mean is checked within the stated tolerance of 1e-5 relative (in
norm, and per element against the recursive-summation bound).
"""
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
    torch.cuda.init()


def _host_rows(n, p, dtype, seed, scale=1.0):
    if dtype == "f32":
        return [synth.normal_f32(seed, k, scale, 0, p) for k in range(n)]
    return [synth.student_t3_bf16(seed, k, scale, 0, p) for k in range(n)]


def _oracle(rows, dtype):
    rows = [r.copy() for r in rows]
    if dtype == "f32":
        oracle.ring_allreduce_avg_f32(rows)
    else:
        oracle.ring_allreduce_avg_bf16(rows)
    return rows[0]


def _assert_rows_equal_oracle(dev_rows, want):
    for k, r in enumerate(dev_rows):
        got = to_host(r)
        if not np.array_equal(got.view(np.uint32 if got.dtype == np.float32 else np.uint16),
                              want.view(np.uint32 if want.dtype == np.float32 else np.uint16)):
            bad = np.nonzero(got != want)[0]
            raise AssertionError("worker %d differs from the oracle at %d elements, first %s: got %r want %r"
                                 % (k, bad.size, bad[:5], got[bad[:5]], want[bad[:5]]))


SHAPES = [(1, 10), (2, 1), (2, 7), (3, 2), (3, 100), (4, 1031), (5, 4099), (7, 333), (8, 0), (8, 7), (8, 8),
          (8, 9), (8, 70_001), (9, 5000), (16, 17), (16, 40_000), (17, 3001), (31, 999), (32, 32_768), (33, 100),
          (64, 6_400), (64, 63)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,p", SHAPES)
def test_fused_matches_oracle(n, p, dtype):
    host = _host_rows(n, p, dtype, seed=n * 1000 + p, scale=1.0)
    want = _oracle(host, dtype)
    rows = to_device_rows(host)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout,pad", [("offset", 1), ("offset", 3), ("offset", 5), ("mixed", 1), ("mixed", 3),
                                        ("packed", 0)])
@pytest.mark.parametrize("n,p", [(4, 1031), (8, 12_345), (3, 77_777), (16, 4_099)])
def test_fused_any_alignment(n, p, dtype, layout, pad):
    host = _host_rows(n, p, dtype, seed=7 + n + p)
    want = _oracle(host, dtype)
    rows = to_device_rows(host, layout=layout, pad=pad)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, want)


def test_ring4_uneven_1m_f32_full():
    wl = synth.WORKLOADS["ring4_uneven_1m_f32"]
    host = [wl.row(k) for k in range(wl.n)]
    want = _oracle(host, "f32")
    for layout in ("separate", "packed"):
        rows = to_device_rows(host, layout=layout)
        ra.ra_allreduce_avg(rows)
        torch.cuda.synchronize()
        _assert_rows_equal_oracle(rows, want)
    # against the binary64 mean: 1e-5 relative in norm and the per-element bound
    mean64 = oracle.mean_f64(host)
    got = to_host(rows[0]).astype(np.float64)
    assert np.linalg.norm(got - mean64) <= 1e-5 * np.linalg.norm(mean64)
    abs_mean = sum(np.abs(r.astype(np.float64)) for r in host) / wl.n
    assert np.all(np.abs(got - mean64) <= 1e-5 * abs_mean + 1e-45)


def test_adversarial_order_is_bit_exact():
    # values where the fold start changes the binary32 sum
    rng = np.random.default_rng(11)
    n, p = 5, 10_007
    choices = np.array([2.0 ** 24, -2.0 ** 24, 1.0, 3.0, -1.0, 0.5], np.float32)
    host = [choices[rng.integers(0, choices.size, p)] for _ in range(n)]
    want = _oracle(host, "f32")
    rows = to_device_rows(host)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, want)


def test_non_power_of_two_division():
    # x / 3 differs from x * (1/3) for some x: the kernel must divide
    n, p = 3, 4096
    host = [np.arange(1, p + 1, dtype=np.float32), np.zeros(p, np.float32), np.zeros(p, np.float32)]
    want = _oracle(host, "f32")
    rows = to_device_rows(host)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, want)


def test_special_values():
    # subnormals, signed zeros, large magnitudes whose sums stay finite (the
    # workloads hold no NaN or Inf, and NaN bit patterns are not compared)
    n, p = 4, 257
    rng = np.random.default_rng(3)
    vals = np.array([0.0, -0.0, 1e-45, -1e-45, 1.2e-38, 8e37, -8e37, 1e-40, 7.0], np.float32)
    host = [vals[rng.integers(0, vals.size, p)] for _ in range(n)]
    want = _oracle(host, "f32")
    rows = to_device_rows(host)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, want)


# --------------------------------------------------------------------------
# SGD epilogue


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,p,woff", [(1, 100, 0), (2, 1031, 0), (5, 7777, 0), (32, 4099, 0), (8, 12_345, 1),
                                      (8, 12_345, 2)])
def test_sgd_matches_oracle(n, p, dtype, woff):
    host = _host_rows(n, p, dtype, seed=50 + n)
    w0 = synth.normal_f32(5, 0, 0.05, 0, p)
    want = _oracle(host, dtype)
    w_want = w0.copy()
    oracle.sgd_update_f32(w_want, want, 0.1)
    rows = to_device_rows(host)
    wbase = torch.empty(p + 8, dtype=torch.float32, device="cuda")
    w = wbase[woff:woff + p]
    w.copy_(torch.from_numpy(w0))
    ra.ra_allreduce_sgd(rows, w, 0.1)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, want)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), w_want.view(np.uint32))


def test_resnet18_sgd_n32_f32_full():
    wl = synth.WORKLOADS["resnet18_sgd_n32_f32"]
    host = [wl.row(k) for k in range(wl.n)]
    w0 = wl.weights()
    want = _oracle(host, "f32")
    w_want = w0.copy()
    oracle.sgd_update_f32(w_want, want, wl.sgd_lr)
    rows = to_device_rows(host)
    w = torch.from_numpy(w0).cuda()
    ra.ra_allreduce_sgd(rows, w, wl.sgd_lr)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, want)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), w_want.view(np.uint32))


# --------------------------------------------------------------------------
# staged (literal schedule)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,p,layout", [(1, 50, "separate"), (2, 7, "separate"), (3, 1000, "separate"),
                                        (5, 4099, "offset"), (8, 70_001, "separate"), (16, 1031, "mixed"),
                                        (4, 1_048_579, "packed")])
def test_staged_matches_oracle_and_counts_traffic(n, p, dtype, layout):
    host = _host_rows(n, p, dtype, seed=90 + n)
    rows_o = [r.copy() for r in host]
    if dtype == "f32":
        sent, recv = oracle.ring_allreduce_avg_f32(rows_o)
    else:
        sent, recv = oracle.ring_allreduce_avg_bf16(rows_o)
    rows = to_device_rows(host, layout=layout, pad=3)
    traffic = ra.ra_allreduce_avg_staged(rows)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, rows_o[0])
    assert [t[0] for t in traffic] == sent.tolist()
    assert [t[1] for t in traffic] == recv.tolist()


@pytest.mark.parametrize("n,p,dtype,layout", [(8, 6_000_017, "f32", "separate"), (4, 10_500_013, "bf16", "offset"),
                                              (4, 10_500_013, "f32", "offset")])
def test_staged_large_tiles_match_oracle(n, p, dtype, layout):
    # large enough that each launch fills a wave with 1024-vector tiles (the
    # staged kernel's larger tile instance); also the workspace-free variant
    host = _host_rows(n, p, dtype, seed=190 + n)
    rows_o = [r.copy() for r in host]
    (oracle.ring_allreduce_avg_f32 if dtype == "f32" else oracle.ring_allreduce_avg_bf16)(rows_o)
    rows = to_device_rows(host, layout=layout, pad=3)
    ra.ra_allreduce_avg_staged(rows)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, rows_o[0])
    if dtype == "f32":  # binary32 needs no scratch, so any length works without a workspace
        rows = to_device_rows(host, layout=layout, pad=3)
        ra.ra_allreduce_avg_staged_static(rows)
        torch.cuda.synchronize()
        _assert_rows_equal_oracle(rows, rows_o[0])


def test_staged_equals_fused():
    wl = synth.WORKLOADS["ring4_uneven_1m_f32"]
    host = [wl.row(k) for k in range(wl.n)]
    a = to_device_rows(host)
    b = to_device_rows(host)
    ra.ra_allreduce_avg(a)
    ra.ra_allreduce_avg_staged(b)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


# --------------------------------------------------------------------------
# buckets


def test_bucket_plan_matches_oracle():
    for numel, eb, cap in [([10, 20, 30, 40], 4, 200), ([10, 50], 4, 200), ([], 4, 8), ([5, 100, 5], 2, 100)]:
        assert ra.ra_bucket_plan(numel, eb, cap) == oracle.bucket_plan(numel, eb, cap)
    wl = synth.WORKLOADS["transformer24_buckets_n4_f32"]
    assert ra.ra_bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes) == oracle.bucket_plan(wl.tensors, 4,
                                                                                        wl.bucket_cap_bytes)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_buckets_match_oracle(dtype):
    rng = np.random.default_rng(5)
    numel = rng.integers(0, 3000, 60).tolist()
    n = 5
    p = sum(numel)
    host = _host_rows(n, p, dtype, seed=123)
    plan = oracle.bucket_plan(numel, 4 if dtype == "f32" else 2, 8000)
    rows_o = [r.copy() for r in host]
    for off, cnt in plan:
        sub = [r[off:off + cnt] for r in rows_o]
        if dtype == "f32":
            oracle.ring_allreduce_avg_f32(sub)
        else:
            oracle.ring_allreduce_avg_bf16(sub)
    rows = to_device_rows(host)
    ra.ra_allreduce_avg_buckets(rows, plan)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, rows_o[0])
    # one launch per bucket gives the same bits
    rows2 = to_device_rows(host)
    for off, cnt in plan:
        ra.ra_allreduce_avg([r[off:off + cnt] for r in rows2])
    torch.cuda.synchronize()
    for x, y in zip(rows, rows2):
        assert torch.equal(x, y)


def test_many_buckets_split_over_launches():
    # more (bucket, chunk) pieces than one launch's parameter table holds
    n = 8
    numel = [37] * 400
    p = sum(numel)
    host = _host_rows(n, p, "f32", seed=9)
    plan = oracle.bucket_plan(numel, 4, 37 * 4)
    assert len(plan) * n > 896
    rows_o = [r.copy() for r in host]
    for off, cnt in plan:
        oracle.ring_allreduce_avg_f32([r[off:off + cnt] for r in rows_o])
    rows = to_device_rows(host)
    ra.ra_allreduce_avg_buckets(rows, plan)
    torch.cuda.synchronize()
    _assert_rows_equal_oracle(rows, rows_o[0])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("extra", [-1, 0, 1])
def test_unaligned_pass_boundaries(dtype, extra):
    # Rows that disagree modulo 16 bytes take the unaligned kernel, which
    # runs a tile's passes of J x 256 elements without bounds checks and
    # checks only the last one.  The chunk lengths here put a tile's element
    # count exactly on a pass boundary, and one element either side, for
    # the all-reduce and SGD (J = 2: 512-element passes) and the
    # reduce-scatter (J = 4: 1024-element passes); a chunk's first and last
    # 16 bytes go element by element, so the kernel's part is L - 2V.
    n = 4
    esz = 4 if dtype == "f32" else 2
    V = 16 // esz
    for k in (1, 2, 3, 4, 5, 8, 9):
        L = 2 * V + 512 * k + extra
        p = n * L
        host = _host_rows(n, p, dtype, seed=50 + k)
        want = _oracle(host, dtype)
        rows = to_device_rows(host, layout="mixed", pad=1)
        ra.ra_allreduce_avg(rows)
        torch.cuda.synchronize()
        _assert_rows_equal_oracle(rows, want)

        # SGD on the same rows, weights offset by one element
        rows = to_device_rows(host, layout="mixed", pad=1)
        w0 = synth.normal_f32(60 + k, 0, 0.05, 0, p)
        wbase = torch.empty(p + 4, dtype=torch.float32, device="cuda")
        w = wbase[1:1 + p]
        w.copy_(torch.from_numpy(w0))
        ra.ra_allreduce_sgd(rows, w, 0.1)
        torch.cuda.synchronize()
        _assert_rows_equal_oracle(rows, want)
        wexp = w0.copy()
        oracle.sgd_update_f32(wexp, want, np.float32(0.1))
        np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), wexp.view(np.uint32))

        # reduce-scatter: each chunk's mean on the worker that owns it
        rows = to_device_rows(host, layout="mixed", pad=1)
        ra.ra_reduce_scatter_avg(rows)
        torch.cuda.synchronize()
        owned = oracle.reduce_scatter_avg([h.copy() for h in host])
        for wk, (b, e) in owned.items():
            got = to_host(rows[wk])[b:e]
            bits = np.uint32 if dtype == "f32" else np.uint16
            np.testing.assert_array_equal(got.view(bits), want[b:e].view(bits), err_msg="k=%d worker %d" % (k, wk))
