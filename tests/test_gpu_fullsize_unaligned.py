"""Full-size workloads with rows that share no 16-byte boundary: the N rows
sit back to back in one allocation with a stride of P + 1 elements, so row k
starts k * (P + 1) elements in and the rows disagree modulo 16 bytes -- the
case the widened-copy kernel handles.

As in the aligned full-size tests, every output element is compared bit for
bit with the oracle's range evaluation over the same host inputs (worker
0's row read back whole; for the reduce-scatter, each chunk on the worker
that owns it), and all workers must end bit-identical.  The gap element
between two rows must be left alone.
"""
from __future__ import annotations

import gc

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth
from gpu_util import assert_row_equals, fill_and_expect

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
    want = fill_and_expect(wl, rows)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    assert_row_equals(rows[0], want, what="speech300m strided worker 0")
    _identical(rows)
    _gaps_intact(big, wl)
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()


def test_speech300m_n8_f32_reduce_scatter_rows_without_common_alignment():
    wl = synth.WORKLOADS["speech300m_n8_f32"]
    big, rows = _strided_rows(wl)
    want = fill_and_expect(wl, rows)
    ra.ra_reduce_scatter_avg(rows)
    torch.cuda.synchronize()
    # which worker the oracle leaves each chunk on, from a small run
    small = [np.zeros(3 * wl.n, np.float32) for _ in range(wl.n)]
    owned = oracle.reduce_scatter_avg(small)
    chunk_of = {oracle.chunk_range(3 * wl.n, wl.n, c): c for c in range(wl.n)}
    owner_of = {chunk_of[tuple(r)]: w for w, r in owned.items()}
    for c in range(wl.n):
        b, e = oracle.chunk_range(wl.p, wl.n, c)
        assert_row_equals(rows[owner_of[c]], want, b, e, what="chunk %d on worker %d" % (c, owner_of[c]))
    _gaps_intact(big, wl)
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()


def test_student_t3_1g_n16_bf16_rows_without_common_alignment():
    wl = synth.WORKLOADS["student_t3_1g_n16_bf16"]
    big, rows = _strided_rows(wl)
    want = fill_and_expect(wl, rows)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    assert_row_equals(rows[0], want, what="student_t3 strided worker 0")
    _identical(rows)
    _gaps_intact(big, wl)
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()


def test_more_than_2_pow_31_elements_rows_without_common_alignment():
    # N=2 rows of 2^31 + 1001 fp32 elements at stride P+1 (8.6 GB each):
    # element indices past 2^31 in the widened-copy kernel must not wrap
    wl = synth.Workload("normal_2g_n2_f32", n=2, p=(1 << 31) + 1001, dtype="f32", dist="normal", scale=1.0, seed=78)
    big = torch.empty(wl.n * (wl.p + 1), dtype=torch.float32, device="cuda")
    rows = [big[k * (wl.p + 1):k * (wl.p + 1) + wl.p] for k in range(wl.n)]
    assert len({r.data_ptr() % 16 for r in rows}) > 1
    want = fill_and_expect(wl, rows)
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    assert_row_equals(rows[0], want, what="2^31+1001 worker 0")
    assert torch.equal(rows[0].view(torch.int32), rows[1].view(torch.int32))
    del rows, big
    gc.collect()
    torch.cuda.empty_cache()
