"""Full-size workloads on the GPU, launched the way bench.py launches them.

The oracle cannot simulate these whole in a test's time, so each test checks
(a) a sample of outputs -- random indices plus every chunk (and bucket)
boundary neighbourhood and both ends -- against the oracle's one-element
ring evaluation, fed with the seeded generator's values at those indices,
on every worker; and (b) properties that hold at any size: all workers end
bit-identical, and the result is within 1e-5 relative (norm) of the binary64
mean on the sample.
"""
from __future__ import annotations

import gc

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth
from gpu_util import fill_device_rows, gather, sample_indices

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


def _inputs_at(wl, idx):
    return [wl.values_at(k, idx) for k in range(wl.n)]


def _check_identical(rows):
    for r in rows[1:]:
        assert torch.equal(rows[0].view(torch.int16) if rows[0].dtype == torch.bfloat16 else rows[0].view(torch.int32),
                           r.view(torch.int16) if r.dtype == torch.bfloat16 else r.view(torch.int32))


def _expected_f32(vals, p, idx, local=None, plocal=None):
    out = np.empty(idx.size, np.float32)
    for j in range(idx.size):
        v = np.array([vals[k][j] for k in range(len(vals))], np.float32)
        if local is None:
            out[j] = oracle.ring_avg_point_f32(v, p, int(idx[j]))
        else:
            out[j] = oracle.ring_avg_point_f32(v, int(plocal[j]), int(local[j]))
    return out


def test_speech300m_n8_f32():
    wl = synth.WORKLOADS["speech300m_n8_f32"]
    rows = _alloc_rows(wl)
    fill_device_rows(wl, rows)
    rng = np.random.default_rng(21)
    idx = sample_indices(wl.p, wl.n, rng, count=3000)
    vals = _inputs_at(wl, idx)
    # inputs on the device are the generator's values
    got_in = gather(rows, idx)
    for k in range(wl.n):
        np.testing.assert_array_equal(got_in[k], vals[k])
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    want = _expected_f32(vals, wl.p, idx)
    for k, g in enumerate(gather(rows, idx)):
        np.testing.assert_array_equal(g.view(np.uint32), want.view(np.uint32), err_msg="worker %d" % k)
    _check_identical(rows)
    mean64 = np.mean(np.stack([v.astype(np.float64) for v in vals]), axis=0)
    assert np.linalg.norm(want - mean64) <= 1e-5 * np.linalg.norm(mean64)
    del rows
    gc.collect()
    torch.cuda.empty_cache()


def test_transformer24_buckets_n4_f32():
    wl = synth.WORKLOADS["transformer24_buckets_n4_f32"]
    plan = ra.ra_bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes)
    assert plan == oracle.bucket_plan(wl.tensors, 4, wl.bucket_cap_bytes)
    rows = _alloc_rows(wl)
    fill_device_rows(wl, rows)
    rng = np.random.default_rng(22)
    extra = []
    for off, cnt in plan:  # every bucket's chunk boundaries and ends
        for c in range(wl.n):
            b, e = oracle.chunk_range(cnt, wl.n, c)
            extra += [off + b - 1, off + b, off + b + 1, off + e - 1]
    idx = sample_indices(wl.p, wl.n, rng, count=3000, extra=extra)
    vals = _inputs_at(wl, idx)
    ra.ra_allreduce_avg_buckets(rows, plan)
    torch.cuda.synchronize()
    starts = np.array(sorted(o for o, _ in plan))
    counts = dict(plan)
    bstart = starts[np.searchsorted(starts, idx, side="right") - 1]
    local = idx - bstart
    plocal = np.array([counts[int(s)] for s in bstart])
    want = _expected_f32(vals, wl.p, idx, local, plocal)
    for k, g in enumerate(gather(rows, idx)):
        np.testing.assert_array_equal(g.view(np.uint32), want.view(np.uint32), err_msg="worker %d" % k)
    _check_identical(rows)
    del rows
    gc.collect()
    torch.cuda.empty_cache()


def test_student_t3_1g_n16_bf16():
    wl = synth.WORKLOADS["student_t3_1g_n16_bf16"]
    rows = _alloc_rows(wl)
    fill_device_rows(wl, rows)
    rng = np.random.default_rng(23)
    idx = sample_indices(wl.p, wl.n, rng, count=3000)
    vals = _inputs_at(wl, idx)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    want = np.array([oracle.ring_avg_point_bf16(np.array([vals[k][j] for k in range(wl.n)], np.uint16), wl.p,
                                                int(idx[j])) for j in range(idx.size)], np.uint16)
    for k, g in enumerate(gather(rows, idx)):
        np.testing.assert_array_equal(g, want, err_msg="worker %d" % k)
    _check_identical(rows)
    del rows
    gc.collect()
    torch.cuda.empty_cache()
