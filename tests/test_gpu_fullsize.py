"""Full-size workloads on the GPU, launched the way bench.py launches them,
compared with the oracle on EVERY element.

The inputs are generated on the host slice by slice; each slice goes to the
device and, from the same host bytes, the oracle's range evaluation gives
the ring's result for every element of it (the ring is element-wise
independent, so a slice with its chunk indices gives exactly the full run's
values; Gibiansky, "Scatter-Reduce" and "Allgather").  After the call,
worker 0's row is read back whole and compared bit for bit, and every other
worker's row must equal worker 0's on the device.  On a sample the result
is also held to the binary64 mean: for binary32 1e-5 relative in norm, and
per element 1e-5 of the mean absolute input.
"""
from __future__ import annotations

import gc

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth
from gpu_util import assert_row_equals, fill_and_expect, sample_indices

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _alloc_rows(wl):
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    return [torch.empty(wl.p, dtype=dt, device="cuda") for _ in range(wl.n)]


def _check_identical(rows):
    v = (lambda t: t.view(torch.int16)) if rows[0].dtype == torch.bfloat16 else (lambda t: t.view(torch.int32))
    for k, r in enumerate(rows[1:], 1):
        assert torch.equal(v(rows[0]), v(r)), "worker %d differs from worker 0" % k


def _close_to_binary64(wl, want, idx):
    """The ring's mean against the binary64 mean on sampled elements: for
    binary32, 1e-5 relative in norm and, per element, 1e-5 of the mean
    absolute input (the recursive-summation bound); bf16 results also carry
    their one rounding to bf16 (8 significand bits: at most 2^-8 relative)."""
    def wide(bits_or_f32):
        if wl.dtype == "f32":
            return bits_or_f32.astype(np.float64)
        return (bits_or_f32.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    vals = np.stack([wide(wl.values_at(k, idx)) for k in range(wl.n)])
    mean64 = vals.mean(axis=0)
    got = wide(want[idx])
    rnd = 0.0 if wl.dtype == "f32" else 2.0 ** -8
    assert np.linalg.norm(got - mean64) <= (1e-5 + rnd) * np.linalg.norm(mean64)
    fold = 1e-5 * np.abs(vals).mean(axis=0)
    assert np.all(np.abs(got - mean64) <= rnd * (np.abs(mean64) + fold) + fold + 1e-45)


def _release(*objs):
    del objs
    gc.collect()
    torch.cuda.empty_cache()


def test_speech300m_n8_f32():
    wl = synth.WORKLOADS["speech300m_n8_f32"]
    rows = _alloc_rows(wl)
    want = fill_and_expect(wl, rows)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    assert_row_equals(rows[0], want, what="speech300m worker 0")
    _check_identical(rows)
    _close_to_binary64(wl, want, sample_indices(wl.p, wl.n, np.random.default_rng(21), count=3000))
    _release(rows)


def test_transformer24_buckets_n4_f32():
    wl = synth.WORKLOADS["transformer24_buckets_n4_f32"]
    plan = ra.ra_bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes)
    assert plan == oracle.bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes)
    rows = _alloc_rows(wl)
    want = fill_and_expect(wl, rows, rings=plan)  # every bucket is a ring of its own
    ra.ra_allreduce_avg_buckets(rows, plan)
    torch.cuda.synchronize()
    assert_row_equals(rows[0], want, what="transformer24 worker 0")
    _check_identical(rows)
    _release(rows)


def test_transformer24_buckets_n4_f32_one_launch_per_bucket():
    wl = synth.WORKLOADS["transformer24_buckets_n4_f32"]
    plan = ra.ra_bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes)
    rows = _alloc_rows(wl)
    want = fill_and_expect(wl, rows, rings=plan)
    for b in plan:  # the order a backward pass makes them ready: output side first
        ra.ra_allreduce_avg_buckets(rows, [b])
    torch.cuda.synchronize()
    assert_row_equals(rows[0], want, what="transformer24 per-bucket worker 0")
    _check_identical(rows)
    _release(rows)


def test_student_t3_1g_n16_bf16():
    wl = synth.WORKLOADS["student_t3_1g_n16_bf16"]
    rows = _alloc_rows(wl)
    want = fill_and_expect(wl, rows)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    assert_row_equals(rows[0], want, what="student_t3 worker 0")
    _check_identical(rows)
    _close_to_binary64(wl, want, sample_indices(wl.p, wl.n, np.random.default_rng(23), count=3000))
    _release(rows)
