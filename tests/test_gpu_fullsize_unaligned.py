"""Full-size workloads with rows that share no 16-byte boundary: the N rows
sit back to back in one allocation with a stride of P + 1 elements, so row k
starts k * (P + 1) elements in and the rows disagree modulo 16 bytes -- the
case the widened-copy kernel handles.

As in the aligned full-size tests, a sample of outputs (random indices, every
chunk boundary neighbourhood, both ends) is checked bit for bit against the
oracle's one-element ring evaluation on every worker, and all workers must
end bit-identical.  The gap element between two rows must be left alone.
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

GAP = 0x5A5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _strided_rows(wl):
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    big = torch.empty(wl.n * (wl.p + 1), dtype=dt, device="cuda")
    big.view(torch.int16).fill_(GAP)
    rows = [big[k * (wl.p + 1):k * (wl.p + 1) + wl.p] for k in range(wl.n)]
    esz = big.element_size()
    shifts = {(r.data_ptr() % 16) // esz for r in rows}
    assert len(shifts) > 1, "the rows must disagree modulo 16 bytes"
    return big, rows


def _gaps_intact(big, wl):
    gaps = torch.arange(1, wl.n + 1, device="cuda") * (wl.p + 1) - 1
    g = big.view(torch.int16).view(-1, big.element_size() // 2)[gaps]
    assert bool((g == GAP).all()), "an element between two rows was written"


def _identical(rows):
    v = (lambda t: t.view(torch.int16)) if rows[0].dtype == torch.bfloat16 else (lambda t: t.view(torch.int32))
    for r in rows[1:]:
        assert torch.equal(v(rows[0]), v(r))


def test_speech300m_n8_f32_rows_without_common_alignment():
    wl = synth.WORKLOADS["speech300m_n8_f32"]
    big, rows = _strided_rows(wl)
    fill_device_rows(wl, rows)
    rng = np.random.default_rng(31)
    idx = sample_indices(wl.p, wl.n, rng, count=3000)
    vals = [wl.values_at(k, idx) for k in range(wl.n)]
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    want = np.array([oracle.ring_avg_point_f32(np.array([vals[k][j] for k in range(wl.n)], np.float32), wl.p,
                                               int(idx[j])) for j in range(idx.size)], np.float32)
    for k, g in enumerate(gather(rows, idx)):
        np.testing.assert_array_equal(g.view(np.uint32), want.view(np.uint32), err_msg="worker %d" % k)
    _identical(rows)
    _gaps_intact(big, wl)
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()


def test_speech300m_n8_f32_reduce_scatter_rows_without_common_alignment():
    wl = synth.WORKLOADS["speech300m_n8_f32"]
    big, rows = _strided_rows(wl)
    fill_device_rows(wl, rows)
    rng = np.random.default_rng(32)
    idx = sample_indices(wl.p, wl.n, rng, count=3000)
    vals = [wl.values_at(k, idx) for k in range(wl.n)]
    ra.ra_reduce_scatter_avg(rows)
    torch.cuda.synchronize()
    want = np.array([oracle.ring_avg_point_f32(np.array([vals[k][j] for k in range(wl.n)], np.float32), wl.p,
                                               int(idx[j])) for j in range(idx.size)], np.float32)
    got = gather(rows, idx)
    # which worker the oracle leaves each chunk on, from a small run
    small = [np.zeros(3 * wl.n, np.float32) for _ in range(wl.n)]
    owned = oracle.reduce_scatter_avg(small)
    chunk_of = {oracle.chunk_range(3 * wl.n, wl.n, c): c for c in range(wl.n)}
    owner_of = {chunk_of[tuple(r)]: w for w, r in owned.items()}
    for c in range(wl.n):
        b, e = oracle.chunk_range(wl.p, wl.n, c)
        sel = (idx >= b) & (idx < e)
        owner = owner_of[c]
        np.testing.assert_array_equal(got[owner][sel].view(np.uint32), want[sel].view(np.uint32),
                                      err_msg="chunk %d" % c)
    _gaps_intact(big, wl)
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()


def test_student_t3_1g_n16_bf16_rows_without_common_alignment():
    wl = synth.WORKLOADS["student_t3_1g_n16_bf16"]
    big, rows = _strided_rows(wl)
    fill_device_rows(wl, rows)
    rng = np.random.default_rng(33)
    idx = sample_indices(wl.p, wl.n, rng, count=3000)
    vals = [wl.values_at(k, idx) for k in range(wl.n)]
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    want = np.array([oracle.ring_avg_point_bf16(np.array([vals[k][j] for k in range(wl.n)], np.uint16), wl.p,
                                                int(idx[j])) for j in range(idx.size)], np.uint16)
    for k, g in enumerate(gather(rows, idx)):
        np.testing.assert_array_equal(g, want, err_msg="worker %d" % k)
    _identical(rows)
    _gaps_intact(big, wl)
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()


def test_more_than_2_pow_31_elements_rows_without_common_alignment():
    # N=2 rows of 2^31 + 1001 fp32 elements at stride P+1 (8.6 GB each):
    # element indices past 2^31 in the widened-copy kernel must not wrap
    n, p = 2, (1 << 31) + 1001
    big = torch.empty(n * (p + 1), dtype=torch.float32, device="cuda")
    rows = [big[k * (p + 1):k * (p + 1) + p] for k in range(n)]
    assert len({r.data_ptr() % 16 for r in rows}) > 1
    piece = 1 << 27
    host = torch.empty(piece, dtype=torch.float32).pin_memory()
    for k, r in enumerate(rows):
        for s in range(0, p, piece):
            c = min(piece, p - s)
            synth.fill_normal_f32(host.data_ptr(), 78, k, 1.0, s, c)
            r[s:s + c].copy_(host[:c])
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    rng = np.random.default_rng(6)
    idx = np.unique(np.concatenate([rng.integers(0, p, 500), np.arange(p - 40, p),
                                    np.arange((1 << 31) - 20, (1 << 31) + 20),
                                    np.arange(p // 2 - 10, p // 2 + 10)])).astype(np.int64)
    vals = [synth.normal_f32_at(78, k, 1.0, idx) for k in range(n)]
    want = np.array([oracle.ring_avg_point_f32(np.array([vals[0][j], vals[1][j]], np.float32), p, int(idx[j]))
                     for j in range(idx.size)], np.float32)
    for g in gather(rows, idx):
        np.testing.assert_array_equal(g.view(np.uint32), want.view(np.uint32))
    assert torch.equal(rows[0].view(torch.int32), rows[1].view(torch.int32))
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()
