"""Guard bands: every device buffer a call writes sits between canary words,
and the canaries must survive every entry point (no write outside
[ptr, ptr + count)).  Also the largest sizes: arrays of more than 2^31
elements, where a 32-bit index would wrap."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth

pytestmark = pytest.mark.gpu

GUARD = 4096  # elements on each side


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


class Guarded:
    """A device tensor of `count` elements at element offset `pad` past a
    16-byte boundary, with GUARD canary elements on both sides."""

    def __init__(self, count, dtype, pad=0, fill=None):
        self.tdt = torch.float32 if dtype == "f32" else torch.bfloat16
        self.base = torch.empty(count + 2 * GUARD + 8, dtype=self.tdt, device="cuda")
        self.base.view(torch.int16 if dtype == "bf16" else torch.int32).fill_(0x5A5A if dtype == "bf16" else 0x5A5A5A5A)
        self.lo = GUARD + pad
        self.t = self.base[self.lo:self.lo + count]
        self.count = count
        self.dtype = dtype
        if fill is not None:
            src = torch.from_numpy(fill.view(np.int16) if dtype == "bf16" else fill)
            self.t.copy_(src.view(torch.bfloat16) if dtype == "bf16" else src)

    def check(self):
        raw = self.base.view(torch.int16 if self.dtype == "bf16" else torch.int32)
        want = 0x5A5A if self.dtype == "bf16" else 0x5A5A5A5A
        before = raw[:self.lo]
        after = raw[self.lo + self.count:]
        assert bool((before == want).all()) and bool((after == want).all()), "a guard band was overwritten"


def _rows(n, p, dtype, seed, pads):
    out = []
    for k in range(n):
        v = synth.normal_f32(seed, k, 1.0, 0, p) if dtype == "f32" else synth.student_t3_bf16(seed, k, 1e-3, 0, p)
        out.append(Guarded(p, dtype, pads[k % len(pads)], v))
    return out


CASES = [(2, 1), (3, 7), (4, 1031), (8, 70_001), (16, 4099), (33, 500)]
PADS = [[0], [1], [3], [0, 1, 2, 3]]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pads", PADS)
@pytest.mark.parametrize("n,p", CASES)
def test_every_entry_point_stays_inside_its_buffers(n, p, dtype, pads):
    g = _rows(n, p, dtype, 1000 + n, pads)
    ts = [x.t for x in g]
    ra.ra_allreduce_avg(ts)
    ra.ra_allreduce_avg_staged(ts)
    ra.ra_allreduce_avg_single_reducer(ts)
    if dtype == "bf16":
        ra.ra_allreduce_avg_bf16_wire(ts)
        if p <= ra.RA_STAGED_STATIC_MAX_P:
            ra.ra_allreduce_avg_staged_static(ts)
    ra.ra_reduce_scatter_avg(ts)
    ra.ra_all_gather(ts)
    shards = []
    for m in range(n):
        b, e = oracle.chunk_range(p, n, (m + 1) % n)
        shards.append(Guarded(e - b, dtype, pads[m % len(pads)]))
    ra.ra_reduce_scatter_avg(ts, [s.t for s in shards])
    ra.ra_all_gather(ts, [s.t for s in shards])
    w = Guarded(p, "f32", pads[0], synth.normal_f32(5, 0, 0.05, 0, p))
    ra.ra_allreduce_sgd(ts, w.t, 0.1)
    plan = oracle.bucket_plan([p // 3, p // 3, p - 2 * (p // 3)], 4 if dtype == "f32" else 2, 64)
    ra.ra_allreduce_avg_buckets(ts, plan)
    torch.cuda.synchronize()
    for x in g + shards + [w]:
        x.check()


def test_more_than_2_pow_31_elements():
    # N=2 workers of 2^31 + 1001 fp32 elements (8.6 GB each): indices past
    # 2^31 must not wrap.  Sampled check against the oracle's point ring.
    n, p = 2, (1 << 31) + 1001
    rows = [torch.empty(p, dtype=torch.float32, device="cuda") for _ in range(n)]
    piece = 1 << 27
    host = torch.empty(piece, dtype=torch.float32).pin_memory()
    for k, r in enumerate(rows):
        for s in range(0, p, piece):
            c = min(piece, p - s)
            synth.fill_normal_f32(host.data_ptr(), 77, k, 1.0, s, c)
            r[s:s + c].copy_(host[:c])
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.integers(0, p, 500), np.arange(p - 40, p),
                                    np.arange((1 << 31) - 20, (1 << 31) + 20),
                                    np.arange(p // 2 - 10, p // 2 + 10)])).astype(np.int64)
    vals = [synth.normal_f32_at(77, k, 1.0, idx) for k in range(n)]
    want = np.array([oracle.ring_avg_point_f32(np.array([vals[0][j], vals[1][j]], np.float32), p, int(idx[j]))
                     for j in range(idx.size)], np.float32)
    it = torch.from_numpy(idx).cuda()
    for r in rows:
        got = r.index_select(0, it).cpu().numpy()
        np.testing.assert_array_equal(got.view(np.uint32), want.view(np.uint32))
    assert torch.equal(rows[0], rows[1])
    del rows
    torch.cuda.empty_cache()


def test_64_workers():
    n, p = 64, 3_000_001
    host = [synth.normal_f32(64, k, 1.0, 0, p) for k in range(n)]
    want = [h.copy() for h in host]
    oracle.ring_allreduce_avg_f32(want)
    rows = [torch.from_numpy(h).cuda() for h in host]
    ra.ra_allreduce_avg(rows)
    torch.cuda.synchronize()
    for r in rows:
        np.testing.assert_array_equal(r.cpu().numpy().view(np.uint32), want[0].view(np.uint32))
