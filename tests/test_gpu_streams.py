"""Stream semantics and thread safety of the C ABI: calls only queue work on
the caller's stream (they return before the GPU runs it, and they are
ordered after earlier work on that stream), and several host threads may
call concurrently on their own streams (ctypes releases the GIL)."""
from __future__ import annotations

import threading
import time

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


def test_calls_return_before_the_gpu_runs_them_and_keep_stream_order():
    n, p = 4, 2_000_003
    host = [synth.normal_f32(21, k, 1.0, 0, p) for k in range(n)]
    # the oracle applies the same four calls in the same order
    want = [h.copy() for h in host]
    oracle.ring_allreduce_avg_f32(want)
    oracle.ring_allreduce_avg_f32(want)
    oracle.reduce_scatter_avg(want)
    oracle.all_gather(want)
    rows = [torch.zeros(p, device="cuda") for _ in range(n)]
    src = [torch.from_numpy(h).cuda() for h in host]
    s = torch.cuda.Stream()
    # The first launch of a kernel in a process may load its module, and
    # CUDA may synchronise the context while loading (lazy module loading);
    # run the same kernel variants once first, as a training loop's first step
    # would.
    warm = [torch.zeros(p, device="cuda") for _ in range(n)]
    ra.ra_allreduce_avg(warm)
    ra.ra_allreduce_avg_staged(warm)
    ra.ra_reduce_scatter_avg(warm)
    ra.ra_all_gather(warm)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(int(2e9))  # about a second of GPU time ahead of everything below
        for r, x in zip(rows, src):
            r.copy_(x)  # the inputs land only after the sleep
        t0 = time.perf_counter()
        ra.ra_allreduce_avg(rows, s)
        ra.ra_allreduce_avg_staged(rows, stream=s)
        ra.ra_reduce_scatter_avg(rows, None, s)
        ra.ra_all_gather(rows, None, s)
        host_ms = (time.perf_counter() - t0) * 1e3
    assert host_ms < 100, "a call waited for the GPU (%.1f ms)" % host_ms
    assert not s.query()  # the queued work is still pending
    s.synchronize()
    # all four calls ran, in order, after the copies of the real inputs
    for r in rows:
        np.testing.assert_array_equal(r.cpu().numpy().view(np.uint32), want[0].view(np.uint32))


def test_concurrent_host_threads_on_their_own_streams():
    nthreads, n, p = 6, 5, 700_001
    results = [None] * nthreads
    errors = []

    def worker(t):
        try:
            torch.cuda.set_device(0)
            host = [synth.normal_f32(100 + t, k, 1.0, 0, p) for k in range(n)]
            want = [h.copy() for h in host]
            oracle.ring_allreduce_avg_f32(want)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                rows = [torch.from_numpy(h).cuda(non_blocking=False) for h in host]
                for _ in range(20):
                    ra.ra_allreduce_avg(rows, s)
                    ra.ra_allreduce_avg_staged(rows, stream=s)
            s.synchronize()
            ok = all(np.array_equal(r.cpu().numpy().view(np.uint32), want[0].view(np.uint32)) for r in rows)
            results[t] = ok
        except Exception as e:  # surfaced below
            errors.append(repr(e))

    ths = [threading.Thread(target=worker, args=(t,)) for t in range(nthreads)]
    for th in ths:
        th.start()
    for th in ths:
        th.join(timeout=300)
    assert not errors, errors
    assert all(results), results
