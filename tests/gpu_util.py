"""Helpers for the GPU parity tests: put seeded host rows on the device in
the layouts the tests need, fill full-size workloads with the oracle's
expected result beside them, and compare device rows with it."""
from __future__ import annotations

import numpy as np
import torch


def to_device_rows(host_rows, layout="separate", pad=0):
    """Copy host rows (float32 or uint16 bf16 bits) to CUDA tensors.

    layout "separate": one allocation per worker (16-byte aligned);
    "offset": one allocation per worker, each starting `pad` elements past a
    16-byte boundary (all rows share the misalignment);
    "mixed": row k starts (k * pad) mod 8 elements past a boundary, so the
    rows disagree and the scalar path runs;
    "packed": all rows back to back in one [N, P] allocation (rows start at
    k*P elements, aligned only if P is a multiple of the vector).
    """
    n = len(host_rows)
    p = host_rows[0].shape[0]
    bf16 = host_rows[0].dtype == np.uint16
    tdt = torch.bfloat16 if bf16 else torch.float32

    def dev(a):
        t = torch.from_numpy(a.view(np.int16) if bf16 else a)
        return t.view(torch.bfloat16) if bf16 else t

    if layout == "packed":
        big = torch.empty(n * p + 8, dtype=tdt, device="cuda")
        rows = [big[k * p:(k + 1) * p] for k in range(n)]
    else:
        rows = []
        for k in range(n):
            off = pad if layout == "offset" else ((k * pad) % 8 if layout == "mixed" else 0)
            base = torch.empty(p + 16, dtype=tdt, device="cuda")
            rows.append(base[off:off + p])
    for k in range(n):
        rows[k].copy_(dev(host_rows[k]))
    return rows


def to_host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def sample_indices(p, n, rng, count=2000, extra=()):
    """Random indices plus every chunk boundary neighbourhood and the ends."""
    idx = set(rng.integers(0, p, count).tolist()) if p > 0 else set()
    from oracle import chunk_range  # host-side index arithmetic of the oracle
    for c in range(n):
        b, e = chunk_range(p, n, c)
        for i in range(b - 9, b + 9):
            if 0 <= i < p:
                idx.add(i)
    for i in list(range(16)) + list(range(p - 16, p)) + list(extra):
        if 0 <= i < p:
            idx.add(i)
    return np.array(sorted(idx), dtype=np.int64)


def fill_and_expect(wl, rows, rings=None):
    """Put the workload's inputs in `rows` and compute the ring's result for
    every element on the host: the rows are generated slice by slice, each
    slice goes to the device rows and, from the same host bytes, the oracle's
    range evaluation gives the ring's result for it (bench.fill_workload,
    which the benchmark uses to check the calls it times).  rings:
    [(offset, count)] element ranges that are rings of their own (the
    buckets), or None for one ring over all p elements.  Returns the expected
    result, p elements (float32, or uint16 bf16 bits)."""
    import bench
    mean, _ = bench.fill_workload(wl, rows, None, rings, verify=True)
    return mean


def assert_row_equals(row, expected, begin=0, end=None, what="", slice_elems=1 << 26):
    """Every element of the device row [begin, end) equals `expected`
    [begin, end) bit for bit (read back in slices)."""
    end = expected.shape[0] if end is None else end
    bits = np.uint16 if expected.dtype == np.uint16 else np.uint32
    for s in range(begin, end, slice_elems):
        e = min(end, s + slice_elems)
        got = to_host(row[s:e]).view(bits)
        want = expected[s:e].view(bits)
        if not np.array_equal(got, want):
            bad = np.flatnonzero(got != want)
            raise AssertionError("%s: %d of %d elements differ from the oracle, first at %d (got %#x, want %#x)"
                                 % (what, bad.size, e - s, s + int(bad[0]), int(got[bad[0]]), int(want[bad[0]])))
