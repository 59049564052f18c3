"""The device calls only queue kernels on the caller's stream (no
allocation, no synchronisation), so a training step can capture them in a
CUDA graph; replaying the graph gives the same bits as eager calls."""
from __future__ import annotations

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


def test_graph_replay_matches_eager_and_oracle():
    n, p = 8, 1_000_003
    host = [synth.normal_f32(11, k, 1.0, 0, p) for k in range(n)]
    want = [h.copy() for h in host]
    oracle.ring_allreduce_avg_f32(want)
    rows = [torch.empty(p, device="cuda") for _ in range(n)]
    src = [torch.from_numpy(h).cuda() for h in host]
    numel = [p // 4, p // 4, p - 2 * (p // 4)]
    plan = ra.ra_bucket_plan(numel, 4, 1 << 20)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # eager warm-up on the capture stream
        for r, x in zip(rows, src):
            r.copy_(x)
        ra.ra_allreduce_avg(rows)
        ra.ra_reduce_scatter_avg(rows)
        ra.ra_all_gather(rows)
        ra.ra_allreduce_avg_buckets(rows, plan)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for r, x in zip(rows, src):
            r.copy_(x)
        ra.ra_allreduce_avg(rows)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for r in rows:
        np.testing.assert_array_equal(r.cpu().numpy().view(np.uint32), want[0].view(np.uint32))
    # reduce-scatter + all-gather and the bucketed call under capture too
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        for r, x in zip(rows, src):
            r.copy_(x)
        ra.ra_reduce_scatter_avg(rows)
        ra.ra_all_gather(rows)
    g2.replay()
    torch.cuda.synchronize()
    for r in rows:
        np.testing.assert_array_equal(r.cpu().numpy().view(np.uint32), want[0].view(np.uint32))
    g3 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g3, stream=s):
        for r, x in zip(rows, src):
            r.copy_(x)
        ra.ra_allreduce_avg_buckets(rows, plan)
    g3.replay()
    torch.cuda.synchronize()
    eager = [x.clone() for x in src]
    ra.ra_allreduce_avg_buckets(eager, plan)
    torch.cuda.synchronize()
    for r, e in zip(rows, eager):
        assert torch.equal(r, e)
