"""ra_reduce_scatter_avg and ra_all_gather (the ring's two phases on their
own) against the CPU oracle, bit for bit.  After the reduce-scatter only the
owned chunks are results: they must equal the oracle's; every other element
must keep its input (the library's documented behaviour)."""
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


def _host_rows(n, p, dtype, seed):
    if dtype == "f32":
        return [synth.normal_f32(seed, k, 1.0, 0, p) for k in range(n)]
    return [synth.student_t3_bf16(seed, k, 1e-3, 0, p) for k in range(n)]


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _shard_tensors(n, p, dtype, pad):
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    out = []
    for m in range(n):
        b, e = oracle.chunk_range(p, n, (m + 1) % n)
        base = torch.empty(e - b + 16, dtype=tdt, device="cuda")
        out.append(base[pad:pad + e - b])
    return out


SHAPES = [(1, 33), (2, 7), (3, 1000), (4, 1_048_579), (5, 4099), (8, 70_001), (16, 12_345), (32, 4096), (64, 200)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["separate", "offset", "mixed"])
@pytest.mark.parametrize("n,p", SHAPES)
def test_reduce_scatter_in_place(n, p, dtype, layout):
    host = _host_rows(n, p, dtype, seed=200 + n)
    want = [r.copy() for r in host]
    owned = oracle.reduce_scatter_avg(want)
    rows = to_device_rows(host, layout=layout, pad=3)
    ra.ra_reduce_scatter_avg(rows)
    torch.cuda.synchronize()
    for w in range(n):
        got = to_host(rows[w])
        b, e = owned[w]
        np.testing.assert_array_equal(_bits(got[b:e]), _bits(want[w][b:e]))
        keep = np.ones(p, bool)
        keep[b:e] = False
        np.testing.assert_array_equal(_bits(got[keep]), _bits(host[w][keep]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pad", [0, 1])
@pytest.mark.parametrize("n,p", [(1, 33), (3, 1000), (4, 1_048_579), (8, 70_001), (16, 12_345)])
def test_reduce_scatter_to_shards(n, p, dtype, pad):
    host = _host_rows(n, p, dtype, seed=300 + n)
    want = [r.copy() for r in host]
    owned = oracle.reduce_scatter_avg(want)
    rows = to_device_rows(host)
    shards = _shard_tensors(n, p, dtype, pad)
    ra.ra_reduce_scatter_avg(rows, shards)
    torch.cuda.synchronize()
    for w in range(n):
        b, e = owned[w]
        np.testing.assert_array_equal(_bits(to_host(shards[w])), _bits(want[w][b:e]))
        np.testing.assert_array_equal(_bits(to_host(rows[w])), _bits(host[w]))  # inputs untouched


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("layout", ["separate", "offset", "mixed"])
@pytest.mark.parametrize("n,p", SHAPES)
def test_all_gather_in_place(n, p, dtype, layout):
    host = _host_rows(n, p, dtype, seed=400 + n)
    want = [r.copy() for r in host]
    oracle.all_gather(want)
    rows = to_device_rows(host, layout=layout, pad=5)
    ra.ra_all_gather(rows)
    torch.cuda.synchronize()
    for w in range(n):
        np.testing.assert_array_equal(_bits(to_host(rows[w])), _bits(want[w]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pad", [0, 3])
@pytest.mark.parametrize("n,p", [(1, 33), (3, 1000), (8, 70_001), (16, 12_345)])
def test_all_gather_from_shards(n, p, dtype, pad):
    host = _host_rows(n, p, dtype, seed=500 + n)
    shards = _shard_tensors(n, p, dtype, pad)
    want = np.empty(p, host[0].dtype)
    for m in range(n):
        b, e = oracle.chunk_range(p, n, (m + 1) % n)
        vals = host[m][:e - b]
        want[b:e] = vals
        t = torch.from_numpy(vals.view(np.int16) if dtype == "bf16" else vals.copy())
        shards[m].copy_(t.view(torch.bfloat16) if dtype == "bf16" else t)
    rows = to_device_rows([np.zeros(p, host[0].dtype) for _ in range(n)])
    ra.ra_all_gather(rows, shards)
    torch.cuda.synchronize()
    for w in range(n):
        np.testing.assert_array_equal(_bits(to_host(rows[w])), _bits(want))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_reduce_scatter_then_all_gather_equals_the_fused_all_reduce(dtype):
    wl_n, p = 8, 1_000_003
    host = _host_rows(wl_n, p, dtype, seed=600)
    a = to_device_rows(host)
    b = to_device_rows(host)
    ra.ra_reduce_scatter_avg(a)
    ra.ra_all_gather(a)
    ra.ra_allreduce_avg(b)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16) if dtype == "bf16" else x.view(torch.int32),
                           y.view(torch.int16) if dtype == "bf16" else y.view(torch.int32))
