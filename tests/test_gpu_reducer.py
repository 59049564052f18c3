"""ra_reducer: per-bucket ring all-reduces queued as the backward pass marks
layer gradients ready, on the reducer's own stream.  Results must equal the
oracle's bucketed all-reduce bit for bit, whatever the marking order, and the
all-reduce of a bucket must see the gradient writes queued before its marks."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth

pytestmark = pytest.mark.gpu

NUMEL = [4096, 64, 64, 16384, 128, 40000, 300, 7, 0, 12345, 2048, 2048]
CAP = 64 * 1024  # bytes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


def _host(n, dtype, seed):
    p = sum(NUMEL)
    if dtype == "f32":
        return [synth.normal_f32(seed, k, 1e-2, 0, p) for k in range(n)]
    return [synth.student_t3_bf16(seed, k, 1e-3, 0, p) for k in range(n)]


def _want(host, dtype):
    rows = [r.copy() for r in host]
    for off, cnt in oracle.bucket_plan(NUMEL, 4 if dtype == "f32" else 2, CAP):
        sub = [r[off:off + cnt] for r in rows]
        (oracle.ring_allreduce_avg_f32 if dtype == "f32" else oracle.ring_allreduce_avg_bf16)(sub)
    return rows[0]


def _dev(host, dtype):
    out = []
    for h in host:
        t = torch.from_numpy(h.view(np.int16) if dtype == "bf16" else h).cuda()
        out.append(t.view(torch.bfloat16) if dtype == "bf16" else t)
    return out


def _host_of(t, dtype):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else t.cpu().numpy()


def _eq(a, b, dtype):
    np.testing.assert_array_equal(a.view(np.uint32) if dtype == "f32" else a, b.view(np.uint32) if dtype == "f32" else b)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("order", ["reverse", "forward", "shuffled"])
@pytest.mark.parametrize("n", [2, 4, 5])
def test_reducer_matches_bucketed_oracle(n, dtype, order):
    host = _host(n, dtype, seed=900 + n)
    want = _want(host, dtype)
    rows = _dev(host, dtype)
    red = ra.Reducer(rows, NUMEL, CAP)
    assert red.buckets() == oracle.bucket_plan(NUMEL, 4 if dtype == "f32" else 2, CAP)
    idx = list(range(len(NUMEL)))
    if order == "reverse":
        idx.reverse()
    elif order == "shuffled":
        np.random.default_rng(n).shuffle(idx)
    for t in idx:
        red.mark_ready(t)
    red.finish()
    torch.cuda.synchronize()
    for r in rows:
        _eq(_host_of(r, dtype), want, dtype)
    red.close()


def test_reducer_waits_for_the_gradient_writes():
    # gradients are written on the compute stream, behind a long matmul,
    # tensor by tensor from the output side; each tensor is marked right after
    # its write is queued.  The reduction must see the written values.
    n, dtype = 4, "f32"
    host = _host(n, dtype, seed=42)
    want = _want(host, dtype)
    src = _dev(host, dtype)
    rows = [torch.zeros_like(s) for s in src]
    red = ra.Reducer(rows, NUMEL, CAP)
    bounds = np.cumsum([0] + NUMEL)
    a = torch.randn(4096, 4096, device="cuda")
    compute = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(compute):
        for t in reversed(range(len(NUMEL))):
            a = a @ a * 1e-3  # a slow kernel ahead of the write
            for k in range(n):
                rows[k][bounds[t]:bounds[t + 1]].copy_(src[k][bounds[t]:bounds[t + 1]])
            red.mark_ready(t, compute)
        red.finish(compute)
    torch.cuda.synchronize()
    for r in rows:
        _eq(_host_of(r, dtype), want, dtype)
    red.close()


def test_finish_reduces_unmarked_buckets_and_resets():
    n, dtype = 3, "f32"
    host = _host(n, dtype, seed=7)
    want = _want(host, dtype)
    rows = _dev(host, dtype)
    red = ra.Reducer(rows, NUMEL, CAP)
    red.mark_ready(len(NUMEL) - 1)
    red.finish()  # everything else reduced here
    torch.cuda.synchronize()
    for r in rows:
        _eq(_host_of(r, dtype), want, dtype)
    # a second step with new gradients works after the reset
    host2 = _host(n, dtype, seed=8)
    want2 = _want(host2, dtype)
    for r, h in zip(rows, host2):
        r.copy_(torch.from_numpy(h))
    for t in reversed(range(len(NUMEL))):
        red.mark_ready(t)
    red.finish()
    torch.cuda.synchronize()
    for r in rows:
        _eq(_host_of(r, dtype), want2, dtype)
    red.close()


def test_marking_a_tensor_twice_is_an_error():
    rows = _dev(_host(2, "f32", seed=1), "f32")
    red = ra.Reducer(rows, NUMEL, CAP)
    red.mark_ready(3)
    with pytest.raises(ra.RaError):
        red.mark_ready(3)
    with pytest.raises(ra.RaError):
        red.mark_ready(len(NUMEL))
    red.finish()
    torch.cuda.synchronize()
    red.close()
