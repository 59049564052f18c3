"""Addressing of the unaligned-rows kernel, checked on the CPU.

When the worker rows disagree modulo 16 bytes the fused all-reduce copies
each row's tile widened to 16-byte boundaries (first byte rounded down, end
rounded up), keeps a 16-byte margin at both ends of every segment (those
elements go element by element), writes the mean with scalar stores, and for
SGD copies the weights the same way and bulk-stores their whole 16-byte
granules.  This test walks that plan in Python, for random layouts, worker
counts, bucket tables and staging budgets, and checks what a bulk copy needs
and what the caller's buffers need:

- every bulk copy starts and ends on a 16-byte boundary and fits its slot;
- every widened copy lies inside its own segment of its own row (or of w);
- the bytes of one barrier's copies stay under the mbarrier's 2^20 limit;
- every destination byte is written exactly once.

The tile rule mirrors the library's (ra_internal.h): the staging budget
divided by n, rounded down to 16 bytes, kept between 2 KB and 16 KB per row,
and cut so that no block stages more than 64 KB; the budget is 32 KB per
block for this kernel and 64 KB for the reduce-scatter.
"""
from __future__ import annotations

import random

import pytest

import oracle

UNALIGNED_STAGE = 32768
ONE_DEST_STAGE = 65536
MAX_STAGE = 65536


def tile_bytes(n, one_destination, budget=UNALIGNED_STAGE):
    budget = ONE_DEST_STAGE if one_destination else budget
    b = min(16384, max(2048, (budget // n) & ~15))
    if b * n > MAX_STAGE:
        b = (MAX_STAGE // n) & ~15
    return b


def test_tile_rule_examples():
    # odd worker counts get tiles that fill the budget; n = 64 is cut to 64 KB per block
    assert [tile_bytes(n, False, 16384) for n in (2, 3, 5, 8, 16, 33, 64)] == [8192, 5456, 3264, 2048, 2048, 1984, 1024]
    assert [tile_bytes(n, True) for n in (2, 8, 64)] == [16384, 8192, 1024]


def rup(x):
    return (x + 15) & ~15


def rdn(x):
    return x & ~15


def walk(n, esz, rows, out, segs, w, aux, budget, margin=True):
    """Follow the kernel's plan; return {(dest, byte): times written}."""
    V = 16 // esz if margin else 0
    B = tile_bytes(n, out == "one", budget)
    slot = B + 16
    wslot = (B // esz) * 4 + 16 if out == "sgd" else 0
    assert n * slot + wslot + 16 + 4 * (2 * n + 1) + 8 + 8 * n <= 227 * 1024
    written = {}

    def wr(dest, lo, hi):
        for x in range(lo, hi):
            written[(dest, x)] = written.get((dest, x), 0) + 1

    for b, e, c in segs:
        ab, ae = b + V, e - V
        if ae < ab:
            ab = ae = b
        nt = max(1, ((ae - ab) * esz + B - 1) // B)
        for t in range(nt):
            first = ab + t * (B // esz)
            left = (ae - first) * esz
            nbytes = 0 if left <= 0 else min(left, B)
            ne = nbytes // esz
            if nbytes > 0:
                total = 0
                for k in range(n):
                    a = rows[k] + first * esz
                    d = a & 15
                    size = rup(d + nbytes)
                    assert (a - d) % 16 == 0 and size % 16 == 0 and size <= slot
                    assert rows[k] + b * esz <= a - d and a - d + size <= rows[k] + e * esz
                    total += size
                if out == "sgd":
                    a = w + first * 4
                    d = a & 15
                    size = rup(d + ne * 4)
                    assert (a - d) % 16 == 0 and size <= wslot
                    assert w + b * 4 <= a - d and a - d + size <= w + e * 4
                    total += size
                assert total < (1 << 20)
                for j in range(ne):  # the mean: scalar stores
                    if out == "one":
                        x = aux[c] + (first + j) * esz
                        wr("aux", x, x + esz)
                    else:
                        for k in range(n):
                            x = rows[k] + (first + j) * esz
                            wr(k, x, x + esz)
                if out == "sgd":  # weights: whole granules by bulk copy, the rest by element
                    a = w + first * 4
                    d = a & 15
                    lo, hi = rup(d), rdn(d + ne * 4)
                    if hi > lo:
                        assert (a - d + lo) % 16 == 0
                        wr("w", a - d + lo, a - d + hi)
                    for j in range(ne):
                        pos = d + 4 * j
                        if not lo <= pos < hi:
                            wr("w", a + 4 * j, a + 4 * j + 4)
            edges = (list(range(b, ab)) if t == 0 else []) + (list(range(max(ae, ab), e)) if t == nt - 1 else [])
            for i in edges:
                if out == "one":
                    wr("aux", aux[c] + i * esz, aux[c] + (i + 1) * esz)
                else:
                    for k in range(n):
                        wr(k, rows[k] + i * esz, rows[k] + (i + 1) * esz)
                    if out == "sgd":
                        wr("w", w + 4 * i, w + 4 * i + 4)
    return written


def expected(n, esz, rows, out, segs, w, aux):
    want = {}
    for b, e, c in segs:
        if out == "one":
            for x in range(aux[c] + b * esz, aux[c] + e * esz):
                want[("aux", x)] = 1
            continue
        for k in range(n):
            for x in range(rows[k] + b * esz, rows[k] + e * esz):
                want[(k, x)] = 1
        if out == "sgd":
            for x in range(w + 4 * b, w + 4 * e):
                want[("w", x)] = 1
    return want


def segments(rng, n, p, bucketed):
    segs = []
    if not bucketed:
        bounds = [0, p]
    else:
        bounds = [0] + sorted(rng.randint(0, p) for _ in range(rng.randint(0, 5))) + [p]
    for x, y in zip(bounds, bounds[1:]):
        for c in range(n):
            b, e = oracle.chunk_range(y - x, n, c)
            if e > b:
                segs.append((x + b, x + e, c))
    return segs


@pytest.mark.parametrize("budget", [16384, 32768, 65536])
@pytest.mark.parametrize("seed", range(4))
def test_widened_copies_stay_inside_and_every_byte_is_written_once(seed, budget):
    rng = random.Random(1000 * seed + budget)
    for _ in range(60):
        n = rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 16, 17, 33, 64])
        p = rng.choice([0, 1, 2, 3, 7, 8, 9, 15, 16, 17, 31, 33, 100, 1000, rng.randint(0, 9000)])
        if n >= 32:
            p = min(p, 2500)
        esz = rng.choice([2, 4])
        rows = [rng.randrange(1 << 30) * 16 + rng.randrange(16 // esz) * esz for _ in range(n)]
        out = rng.choice(["all", "all", "sgd", "one"])
        w = rng.randrange(1 << 30) * 16 + rng.randrange(4) * 4
        aux = [rng.randrange(1 << 30) * 16 + rng.randrange(16 // esz) * esz for _ in range(n)]
        segs = segments(rng, n, p, out == "all" and rng.random() < 0.4)
        assert walk(n, esz, rows, out, segs, w, aux, budget) == expected(n, esz, rows, out, segs, w, aux)


def test_without_the_margins_a_widened_copy_leaves_its_segment():
    # the mutation the margins exist for: tiles starting at the segment's
    # first element let the rounded-down copy start before the row
    rows = [16 * 100 + 4, 16 * 900 + 8]
    segs = [(b, e, c) for c in range(2) for b, e in [oracle.chunk_range(1000, 2, c)]]
    walk(2, 4, rows, "all", segs, 0, [0, 0], UNALIGNED_STAGE)
    with pytest.raises(AssertionError):
        walk(2, 4, rows, "all", segs, 0, [0, 0], UNALIGNED_STAGE, margin=False)
