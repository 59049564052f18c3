"""Pins for the CPU oracle: the pages' worked tables, exact arithmetic,
closed forms and invariants (no GPU).

Each test fails for a plausible mistake in the oracle: a wrong chunk index or
direction in the schedule, a dropped or repeated addend, a different fold
start, multiplication by 1/N instead of division, a fused multiply-add in the
SGD step, or a wrong bucket rule.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np
import pytest

import exact_ieee as X
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


def _kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split()
                out[k] = float(v)
    return out


def _int_rows(rng, n, p, lim=1000):
    return [rng.integers(-lim, lim + 1, p).astype(np.float32) for _ in range(n)]


# --------------------------------------------------------------------------
# schedule: the pages' 5-GPU tables


def test_scatter_reduce_first_iteration_table():
    for gpu, sends, recvs in _table("gibiansky_scatter_reduce_first_iteration.txt"):
        assert oracle.scatter_send_chunk(5, gpu, 0) == sends
        assert oracle.scatter_recv_chunk(5, gpu, 0) == recvs


def test_allgather_first_iteration_table():
    for gpu, sends, recvs in _table("gibiansky_allgather_first_iteration.txt"):
        assert oracle.gather_send_chunk(5, gpu, 0) == sends
        assert oracle.gather_recv_chunk(5, gpu, 0) == recvs


@pytest.mark.parametrize("n", [2, 3, 5, 8, 13])
def test_schedule_forwards_what_was_received(n):
    # Both phases: each iteration sends the chunk received in the previous
    # one, and what worker m receives is what worker m-1 sends.
    for t in range(n - 2):
        for w in range(n):
            assert oracle.scatter_send_chunk(n, w, t + 1) == oracle.scatter_recv_chunk(n, w, t)
            assert oracle.gather_send_chunk(n, w, t + 1) == oracle.gather_recv_chunk(n, w, t)
    for t in range(n - 1):
        for w in range(n):
            assert oracle.scatter_recv_chunk(n, w, t) == oracle.scatter_send_chunk(n, (w - 1) % n, t)
            assert oracle.gather_recv_chunk(n, w, t) == oracle.gather_send_chunk(n, (w - 1) % n, t)
        # every chunk is on the wire exactly once per iteration
        assert sorted(oracle.scatter_send_chunk(n, w, t) for w in range(n)) == list(range(n))
        assert sorted(oracle.gather_send_chunk(n, w, t) for w in range(n)) == list(range(n))


# --------------------------------------------------------------------------
# chunks


@pytest.mark.parametrize("p,n", [(0, 1), (0, 4), (3, 4), (4, 4), (5, 4), (1_048_579, 4), (17, 5), (100, 64)])
def test_chunks_partition_in_order(p, n):
    ranges = [oracle.chunk_range(p, n, c) for c in range(n)]
    assert ranges[0][0] == 0 and ranges[-1][1] == p
    for (b0, e0), (b1, e1) in zip(ranges, ranges[1:]):
        assert e0 == b1
    sizes = [e - b for b, e in ranges]
    # N "equal" chunks: sizes differ by at most one, larger ones first
    assert max(sizes) - min(sizes) <= 1
    assert sizes == sorted(sizes, reverse=True)
    assert sum(sizes) == p


def test_chunks_of_the_uneven_4_worker_ring():
    # P = 1,048,579 = 4 * 262,144 + 3: three chunks of 262,145, one of 262,144
    assert [oracle.chunk_range(1_048_579, 4, c) for c in range(4)] == [
        (0, 262_145), (262_145, 524_290), (524_290, 786_435), (786_435, 1_048_579)]


# --------------------------------------------------------------------------
# intermediate states


def test_first_iteration_partial_sum():
    # Scatter-Reduce: after the first iteration the second GPU's first chunk
    # is the sum of the first and second GPUs' values of that chunk.
    rng = np.random.default_rng(1)
    g = _int_rows(rng, 5, 23)
    rows = [r.copy() for r in g]
    oracle.ring_run_f32(rows, 1, False, 0)
    b, e = oracle.chunk_range(23, 5, 0)
    np.testing.assert_array_equal(rows[1][b:e], g[0][b:e] + g[1][b:e])
    # every worker changed exactly the chunk it received
    for m in range(5):
        c = oracle.scatter_recv_chunk(5, m, 0)
        for k in range(5):
            bk, ek = oracle.chunk_range(23, 5, k)
            if k == c:
                np.testing.assert_array_equal(rows[m][bk:ek], g[m][bk:ek] + g[(m - 1) % 5][bk:ek])
            else:
                np.testing.assert_array_equal(rows[m][bk:ek], g[m][bk:ek])


@pytest.mark.parametrize("n,p", [(2, 7), (5, 23), (8, 64), (7, 3)])
def test_after_scatter_each_worker_holds_one_complete_chunk(n, p):
    rng = np.random.default_rng(n * 100 + p)
    g = _int_rows(rng, n, p)
    total = sum(r.astype(np.float64) for r in g)
    rows = [r.copy() for r in g]
    oracle.ring_run_f32(rows, n - 1, False, 0)
    for w in range(n):
        b, e = oracle.chunk_range(p, n, (w + 1) % n)
        np.testing.assert_array_equal(rows[w][b:e].astype(np.float64), total[b:e])


def test_allgather_overwrites_and_ignores_old_values():
    # All-gather replaces the receiver's chunk; what it held before must not
    # matter.  Poison every non-final chunk before the all-gather.
    rng = np.random.default_rng(2)
    n, p = 6, 41
    g = [rng.standard_normal(p).astype(np.float32) for _ in range(n)]
    ref = [r.copy() for r in g]
    oracle.ring_allreduce_avg_f32(ref)
    rows = [r.copy() for r in g]
    oracle.ring_run_f32(rows, n - 1, True, 0)
    for w in range(n):
        for k in range(n):
            if k != (w + 1) % n:
                b, e = oracle.chunk_range(p, n, k)
                rows[w][b:e] = np.float32(12345.0)
    # run only the all-gather
    oracle.ring_run_f32(rows, 0, False, n - 1)
    for w in range(n):
        np.testing.assert_array_equal(rows[w], ref[0])


# --------------------------------------------------------------------------
# exact results


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9, 16, 31])
def test_small_integers_give_the_correctly_rounded_mean(n):
    # Small integers add exactly in any order, so the ring's sum is the exact
    # sum S and its result must be RN(S / N) -- checked with exact rationals.
    rng = np.random.default_rng(n)
    p = 3 * n + 2
    g = _int_rows(rng, n, p, lim=2 ** 10)
    rows = [r.copy() for r in g]
    oracle.ring_allreduce_avg_f32(rows)
    for i in range(p):
        s = sum(int(r[i]) for r in g)
        want = X.rn_f32(Fraction(s, n))
        for r in rows:
            assert Fraction(float(r[i])) == want, (n, i)


def test_division_not_reciprocal_multiplication():
    # For N=3 or 10, x / N and x * (1/N) differ for some x; the oracle must
    # divide.  Search inputs where they differ and check the oracle divides.
    found = 0
    for n in (3, 10):
        for s in range(1, 2000):
            q_div = X.rn_f32(Fraction(s, n))
            q_mul = X.rn_f32(Fraction(s) * X.rn_f32(Fraction(1, n)))
            if q_div != q_mul:
                rows = [np.full(n, np.float32(0.0)) for _ in range(n)]
                rows[0][:] = np.float32(s)
                oracle.ring_allreduce_avg_f32(rows)
                assert Fraction(float(rows[0][0])) == q_div
                found += 1
                break
    assert found == 2


def _fold(vals, start):
    """Left fold from worker `start` around the ring, exact binary32 adds."""
    n = len(vals)
    acc = X.frac(vals[start])
    for k in range(1, n):
        acc = X.add(vals[(start + k) % n], acc)
    return acc


def test_summation_order_is_the_ring_fold_of_each_chunk():
    # Values chosen so that the fold start changes the binary32 result.
    rng = np.random.default_rng(3)
    n, p = 5, 40
    big = np.float32(2.0 ** 24)
    g = [np.zeros(p, np.float32) for _ in range(n)]
    for i in range(p):
        vals = rng.choice([big, -big, np.float32(1.0), np.float32(3.0), np.float32(-1.0)], size=n)
        for w in range(n):
            g[w][i] = vals[w]
    rows = [r.copy() for r in g]
    oracle.ring_allreduce_avg_f32(rows)
    sensitive = 0
    for c in range(n):
        b, e = oracle.chunk_range(p, n, c)
        for i in range(b, e):
            vals = [g[w][i] for w in range(n)]
            want = X.div(_fold(vals, c), n)
            assert Fraction(float(rows[0][i])) == want, (c, i)
            if any(X.div(_fold(vals, s), n) != want for s in range(n) if s != c):
                sensitive += 1
    assert sensitive >= 5  # the data really distinguishes the fold start


def test_point_evaluation_matches_the_full_ring():
    rng = np.random.default_rng(4)
    for n, p in [(1, 5), (2, 9), (4, 1031), (7, 100), (16, 333), (33, 40)]:
        g = [rng.standard_normal(p).astype(np.float32) * np.float32(rng.choice([1e-3, 1, 1e3])) for _ in range(n)]
        rows = [r.copy() for r in g]
        oracle.ring_allreduce_avg_f32(rows)
        for i in range(p):
            v = np.array([r[i] for r in g], np.float32)
            assert oracle.ring_avg_point_f32(v, p, i) == rows[0][i], (n, p, i)


def _ranges(rng, n, p):
    """Sub-ranges of a p-element ring: whole, empty, around every chunk
    boundary, single elements and random spans."""
    out = [(0, p), (0, 0), (p, p)]
    for c in range(n):
        b, e = oracle.chunk_range(p, n, c)
        out += [(max(0, b - 3), min(p, b + 3)), (b, e), (max(0, e - 1), e)]
    for _ in range(12):
        b = int(rng.integers(0, p + 1))
        out.append((b, int(rng.integers(b, p + 1))))
    return out


@pytest.mark.parametrize("bf16", [False, True])
def test_range_evaluation_matches_the_full_ring(bf16):
    # The range form evaluates any slice of the ring from the input slices
    # alone; on every slice it must give the literal simulation's bits.
    # Rows at mixed scales make the result depend on the fold start.
    import synth
    rng = np.random.default_rng(41)
    for n, p in [(1, 5), (2, 9), (3, 2), (4, 1031), (7, 100), (16, 333), (33, 40)]:
        if bf16:
            g = [synth.student_t3_bf16(7, k, float(rng.choice([1e-3, 1, 1e3])), 0, p) for k in range(n)]
            rows = [r.copy() for r in g]
            oracle.ring_allreduce_avg_bf16(rows)
        else:
            g = [rng.standard_normal(p).astype(np.float32) * np.float32(rng.choice([1e-3, 1, 1e3])) for _ in range(n)]
            rows = [r.copy() for r in g]
            oracle.ring_allreduce_avg_f32(rows)
        whole = oracle.ring_avg_range([r.copy() for r in g], p, 0)
        assert np.array_equal(whole.view(np.uint16 if bf16 else np.uint32), rows[0].view(np.uint16 if bf16 else np.uint32))
        for b, e in _ranges(rng, n, p):
            got = oracle.ring_avg_range([np.ascontiguousarray(r[b:e]) for r in g], p, b)
            assert got.shape == (e - b,)
            assert np.array_equal(got.view(np.uint16 if bf16 else np.uint32),
                                  rows[0][b:e].view(np.uint16 if bf16 else np.uint32)), (n, p, b, e)


def test_range_evaluation_rejects_a_slice_outside_the_ring():
    g = [np.zeros(4, np.float32) for _ in range(2)]
    with pytest.raises(ValueError):
        oracle.ring_avg_range(g, 6, 3)  # elements 3..7 of a 6-element ring


# --------------------------------------------------------------------------
# invariants


@pytest.mark.parametrize("n,p", [(2, 1), (3, 2), (4, 1031), (8, 64), (64, 100), (5, 0)])
def test_all_workers_end_identical(n, p):
    rng = np.random.default_rng(n + p)
    rows = [rng.standard_normal(p).astype(np.float32) for _ in range(n)]
    oracle.ring_allreduce_avg_f32(rows)
    for r in rows[1:]:
        np.testing.assert_array_equal(r, rows[0])


def test_one_worker_is_unchanged():
    rng = np.random.default_rng(5)
    g = rng.standard_normal(1000).astype(np.float32)
    rows = [g.copy()]
    sent, recv = oracle.ring_allreduce_avg_f32(rows)
    np.testing.assert_array_equal(rows[0], g)
    assert sent[0] == 0 and recv[0] == 0


@pytest.mark.parametrize("n", [2, 4, 8, 16, 32, 64])
def test_close_to_the_binary64_mean(n):
    # Recursive summation bound (Higham): |fl(sum) - sum| <= (N-1) u sum|g| + O(u^2),
    # plus one rounding of the division.
    rng = np.random.default_rng(n)
    p = 2000
    g = [(rng.standard_normal(p) * rng.choice([1e-3, 1.0, 1e2], size=p)).astype(np.float32) for _ in range(n)]
    mean64 = oracle.mean_f64(g)
    rows = [r.copy() for r in g]
    oracle.ring_allreduce_avg_f32(rows)
    u = 2.0 ** -24
    abs_sum = sum(np.abs(r.astype(np.float64)) for r in g)
    bound = ((n - 1) * u * 1.001) * abs_sum / n + u * np.abs(mean64) + 1e-45
    err = np.abs(rows[0].astype(np.float64) - mean64)
    assert np.all(err <= bound)
    # the tolerance stated for the method: 1e-5 relative in norm
    assert np.linalg.norm(rows[0] - mean64) <= 1e-5 * np.linalg.norm(mean64)


def test_mean_f64_is_the_mean():
    rng = np.random.default_rng(6)
    g = [rng.integers(-50, 50, 11).astype(np.float32) for _ in range(6)]
    m = oracle.mean_f64(g)
    for i in range(11):
        assert Fraction(m[i]) == Fraction(sum(int(r[i]) for r in g), 6) or abs(
            m[i] - sum(int(r[i]) for r in g) / 6) == 0


# --------------------------------------------------------------------------
# traffic


@pytest.mark.parametrize("n,p", [(2, 10), (4, 1_048_576), (5, 100), (8, 4000), (40, 4000)])
def test_traffic_is_2_n_minus_1_over_n_of_the_array(n, p):
    # Allreduce Communication Cost: N-1 sends in each phase, K/N values each:
    # 2(N-1)K/N per GPU, independent of the worker.
    assert p % n == 0
    sent, recv = oracle.ring_traffic(n, p)
    assert np.all(sent == 2 * (n - 1) * p // n)
    assert np.all(recv == 2 * (n - 1) * p // n)


@pytest.mark.parametrize("n,p", [(3, 10), (4, 1_048_579), (7, 5), (8, 3)])
def test_traffic_uneven_chunks(n, p):
    # A worker sends every chunk except (n+1) in the scatter phase and every
    # chunk except (n+2) in the all-gather phase; it receives every chunk
    # except n and (n+1).
    sizes = [oracle.chunk_range(p, n, c)[1] - oracle.chunk_range(p, n, c)[0] for c in range(n)]
    sent, recv = oracle.ring_traffic(n, p)
    for w in range(n):
        assert sent[w] == 2 * p - sizes[(w + 1) % n] - sizes[(w + 2) % n]
        assert recv[w] == 2 * p - sizes[w] - sizes[(w + 1) % n]
    assert sent.sum() == recv.sum()


def test_simulated_traffic_matches_the_schedule_walk():
    rng = np.random.default_rng(7)
    for n, p in [(3, 10), (5, 23), (8, 64)]:
        rows = [rng.standard_normal(p).astype(np.float32) for _ in range(n)]
        s1, r1 = oracle.ring_allreduce_avg_f32(rows)
        s2, r2 = oracle.ring_traffic(n, p)
        np.testing.assert_array_equal(s1, s2)
        np.testing.assert_array_equal(r1, r2)


def test_cost_figures_of_the_pages():
    f = _kv("gibiansky_cost_figures.txt")
    p = int(f["params"])
    nbytes = p * f["bytes_per_param"]
    assert abs(nbytes / 1e9 - f["gradient_gb"]) < 0.05
    # the ring: about 2.4 GB per GPU, about 400 ms at 6 GB/s (40 GPUs)
    n = int(f["ring_gpus"])
    sent, recv = oracle.ring_traffic(n, p - p % n)
    gb = sent[0] * f["bytes_per_param"] / 1e9
    assert abs(gb - f["ring_gb_per_gpu"]) / f["ring_gb_per_gpu"] < 0.05
    assert abs(gb / f["ring_link_gbps"] * 1e3 - f["ring_comm_ms"]) / f["ring_comm_ms"] < 0.05
    # the single reducer's extra time grows with N-1 (1.2 s at 2 GPUs, 10.8 s at 10)
    for gpus, key in ((2, "single_reducer_extra_s_2gpu"), (10, "single_reducer_extra_s_10gpu")):
        t = (gpus - 1) * nbytes / 1e9 / f["single_reducer_link_gbps"]
        assert abs(t - f[key]) < 1e-6


# --------------------------------------------------------------------------
# data-parallel identity ([AI System] Training With Multiple GPUs, Comparison
# With Centralized Training; GPipe page section 7)


def _linreg_case(rng, n, b, d):
    x = rng.integers(-3, 4, (b, d)).astype(np.float32)
    y = rng.integers(-3, 4, b).astype(np.float32)
    w = rng.integers(-2, 3, d).astype(np.float32)
    return x, y, w


@pytest.mark.parametrize("n", [1, 2, 4, 8])
def test_ring_average_equals_full_batch_gradient(n):
    # Equal contiguous shards (DistributedSampler-style); per-worker mean-loss
    # gradient (2/(B/N)) X_n^T (X_n w - y_n).  With small integers and
    # power-of-two shard sizes every quantity is exact, so the ring average
    # must equal the full-batch gradient (2/B) X^T (X w - y) bit for bit.
    rng = np.random.default_rng(n)
    b, d = 32, 7
    x, y, w = _linreg_case(rng, n, b, d)
    sh = b // n
    grads = []
    for k in range(n):
        xs, ys = x[k * sh:(k + 1) * sh], y[k * sh:(k + 1) * sh]
        grads.append((np.float32(2.0 / sh) * (xs.T @ (xs @ w - ys))).astype(np.float32))
    rows = [g.copy() for g in grads]
    oracle.ring_allreduce_avg_f32(rows)
    full = (np.float32(2.0 / b) * (x.T @ (x @ w - y))).astype(np.float32)
    np.testing.assert_array_equal(rows[0], full)


def test_model_averaging_equals_gradient_averaging():
    # Each worker takes one local step with its own gradient; averaging the
    # models equals stepping with the averaged gradient (exact data).
    rng = np.random.default_rng(9)
    n, b, d, lr = 4, 16, 5, np.float32(0.125)
    x, y, w = _linreg_case(rng, n, b, d)
    sh = b // n
    grads = []
    for k in range(n):
        xs, ys = x[k * sh:(k + 1) * sh], y[k * sh:(k + 1) * sh]
        grads.append((np.float32(2.0 / sh) * (xs.T @ (xs @ w - ys))).astype(np.float32))
    models = [(w - lr * g).astype(np.float32) for g in grads]
    oracle.ring_allreduce_avg_f32(models)
    rows = [g.copy() for g in grads]
    oracle.ring_allreduce_avg_f32(rows)
    w2 = w.copy()
    oracle.sgd_update_f32(w2, rows[0], lr)
    np.testing.assert_array_equal(models[0], w2)


# --------------------------------------------------------------------------
# bf16


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(10)
    x = np.concatenate([
        rng.standard_normal(5000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormal range
        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2 ** -133, 3.0e38, 0.0, -0.0],
                 np.float32),                                    # exact ties and edges
    ])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle.f32_to_bf16_bits(v) for v in x], np.uint16)
    np.testing.assert_array_equal(got, want)


def test_bf16_rounding_exact_model():
    rng = np.random.default_rng(11)
    for v in rng.standard_normal(500).astype(np.float32):
        assert X.bf16_value(oracle.f32_to_bf16_bits(v)) == X.rn_bf16(X.frac(v))


def _bf16_rows_from_ints(rng, n, p, lim):
    # small integers are exact bf16 values when |v| <= 256
    vals = [rng.integers(-lim, lim + 1, p).astype(np.float32) for _ in range(n)]
    return vals, [(v.view(np.uint32) >> 16).astype(np.uint16) for v in vals]


@pytest.mark.parametrize("n", [2, 3, 5, 16])
def test_bf16_ring_rounds_the_exact_mean_once(n):
    rng = np.random.default_rng(12 + n)
    p = 4 * n + 3
    vals, rows = _bf16_rows_from_ints(rng, n, p, 256)
    oracle.ring_allreduce_avg_bf16(rows)
    for i in range(p):
        s = sum(int(v[i]) for v in vals)
        want = X.rn_bf16(X.rn_f32(Fraction(s, n)))
        for r in rows:
            assert X.bf16_value(r[i]) == want


def test_bf16_point_evaluation_matches_the_full_ring():
    import synth
    for n, p in [(2, 9), (5, 101), (16, 333)]:
        rows = [synth.student_t3_bf16(3, w, 1e-3, 0, p) for w in range(n)]
        g = [r.copy() for r in rows]
        oracle.ring_allreduce_avg_bf16(rows)
        for i in range(p):
            assert oracle.ring_avg_point_bf16(np.array([r[i] for r in g], np.uint16), p, i) == rows[0][i]


def test_bf16_partials_stay_binary32():
    # With bf16 partials the sum 256 + 1 + 1 would lose the ones (bf16 keeps
    # 8 significand bits); with binary32 partials the mean is (258)/3 = 86.
    rows = [np.array([v], np.float32) for v in (256.0, 1.0, 1.0)]
    b = [(r.view(np.uint32) >> 16).astype(np.uint16) for r in rows]
    oracle.ring_allreduce_avg_bf16(b)
    assert X.bf16_value(b[0][0]) == X.rn_bf16(X.rn_f32(Fraction(258, 3)))


# --------------------------------------------------------------------------
# SGD


def test_sgd_is_two_roundings_not_fma():
    rng = np.random.default_rng(13)
    lr = np.float32(0.1)
    w = rng.standard_normal(4000).astype(np.float32)
    avg = rng.standard_normal(4000).astype(np.float32)
    got = w.copy()
    oracle.sgd_update_f32(got, avg, lr)
    differs_from_fma = 0
    for i in range(4000):
        want = X.sub(w[i], X.mul(lr, avg[i]))
        assert Fraction(float(got[i])) == want
        if X.rn_f32(X.frac(w[i]) - X.frac(lr) * X.frac(avg[i])) != want:
            differs_from_fma += 1
    assert differs_from_fma > 0


def test_sgd_with_bf16_gradients_uses_the_bf16_mean():
    # bf16 gradients: every replica holds the bf16-rounded mean after the
    # all-reduce, and that is what it applies (The Communication Problem:
    # the averaged gradient updates the weights; DDP: every replica applies
    # the same one).  Expected values come from the exact-rational model:
    # the ring's binary32 fold and division, one bf16 rounding, then
    # w - RN(lr * mean) rounded twice.  The data is chosen so that three
    # wrong readings give other bits on some elements: updating with the
    # binary32 mean before its bf16 rounding, a fused multiply-add, and a
    # step lr * mean rounded to bf16.
    import synth
    n, p = 4, 3000
    lr = np.float32(0.1)
    g = [synth.student_t3_bf16(3, k, 1e-3, 0, p) for k in range(n)]
    w = synth.normal_f32(5, 0, 0.05, 0, p)
    rows = [r.copy() for r in g]
    oracle.ring_allreduce_avg_bf16(rows)
    got = w.copy()
    oracle.sgd_update_f32(got, rows[0], lr)
    wrong = {"binary32 mean": 0, "fma": 0, "bf16 step": 0}
    for i in range(p):
        c = next(k for k in range(n) if oracle.chunk_range(p, n, k)[0] <= i < oracle.chunk_range(p, n, k)[1])
        acc = X.bf16_value(g[c][i])
        for t in range(1, n):
            acc = X.add(X.bf16_value(g[(c + t) % n][i]), acc)
        m32 = X.div(acc, n)
        m16 = X.rn_bf16(m32)
        assert X.bf16_value(rows[0][i]) == m16
        want = X.sub(w[i], X.mul(lr, m16))
        assert Fraction(float(got[i])) == want, i
        wrong["binary32 mean"] += X.sub(w[i], X.mul(lr, m32)) != want
        wrong["fma"] += X.rn_f32(X.frac(w[i]) - X.frac(lr) * m16) != want
        wrong["bf16 step"] += X.sub(w[i], X.rn_bf16(X.mul(lr, m16))) != want
    assert all(v > 0 for v in wrong.values()), wrong


# --------------------------------------------------------------------------
# buckets (Applying the Allreduce to Deep Learning: subsets, output layer first)


def test_bucket_plan_hand_example():
    # tensors (forward order) of 10, 20, 30, 40 elements, 4-byte elements,
    # cap 200 bytes = 50 elements; the tensors start at 0, 10, 30, 60.
    # Reverse walk: 40 (<50), +30 = 70 -> close [30, 100); 20 (<50),
    # +10 = 30 -> end: last bucket [0, 30).
    assert oracle.bucket_plan([10, 20, 30, 40], 4, 200) == [(30, 70), (0, 30)]
    # a single tensor above the cap closes a bucket on its own
    assert oracle.bucket_plan([5, 100, 5], 4, 200) == [(5, 105), (0, 5)]
    # a bucket that reaches the cap exactly is closed (">= cap")
    assert oracle.bucket_plan([10, 50], 4, 200) == [(10, 50), (0, 10)]
    assert oracle.bucket_plan([], 4, 200) == []
    assert oracle.bucket_plan([3], 4, 4) == [(0, 3)]


def test_bucket_plan_invariants_on_the_transformer():
    import synth
    numel = synth.shapes.numels(synth.transformer_shapes())
    cap = 25 * 1024 * 1024
    plan = oracle.bucket_plan(numel, 4, cap)
    bounds = np.cumsum([0] + numel)
    # contiguous, reverse order, covering everything
    assert plan[0][0] + plan[0][1] == sum(numel)
    for (o0, c0), (o1, c1) in zip(plan, plan[1:]):
        assert o1 + c1 == o0
    assert plan[-1][0] == 0
    for k, (o, c) in enumerate(plan):
        assert o in bounds and o + c in bounds  # whole tensors only
        if k < len(plan) - 1:
            assert c * 4 >= cap
            # minimal: without its first (lowest-offset) tensor it is below the cap
            j = int(np.searchsorted(bounds, o))
            assert (o + c - bounds[j + 1]) * 4 < cap
    # the output projection (32000 x 2048 fp32 = 262 MB) is the first bucket
    assert plan[0] == (sum(numel) - 32000 * 2048, 32000 * 2048)


def test_buckets_are_rings_of_their_own():
    rng = np.random.default_rng(14)
    n, numel = 3, [7, 5, 11, 9]
    p = sum(numel)
    g = [(rng.standard_normal(p) * 1e3).astype(np.float32) for _ in range(n)]
    plan = oracle.bucket_plan(numel, 4, 40)
    rows = [r.copy() for r in g]
    oracle.ring_allreduce_avg_buckets_f32(rows, plan)
    for o, c in plan:
        sub = [r[o:o + c].copy() for r in g]
        oracle.ring_allreduce_avg_f32(sub)
        np.testing.assert_array_equal(rows[0][o:o + c], sub[0])


# --------------------------------------------------------------------------
# workload shapes against the pages' parameter counts


def test_transformer_parameter_count():
    import synth
    f = _kv("gpipe_transformer_params.txt")
    numel = synth.shapes.numels(synth.transformer_shapes())
    assert len(numel) == 2 + 24 * 16
    one = synth.shapes.numels(synth.transformer_shapes(layers=1))
    fixed = 2 * int(f["vocab"]) * int(f["d"])
    per_layer = sum(one) - fixed
    assert abs(per_layer / 1e6 - f["per_layer_millions"]) < 0.005
    assert abs(fixed / 1e6 - f["fixed_millions"]) < 0.5
    assert abs((fixed + 3 * per_layer) / 1e6 - f["layers3_millions"]) < 0.05
    assert abs((fixed + 1663 * per_layer) / 1e9 - f["layers1663_billions"]) < 0.005
    assert sum(numel) == fixed + 24 * per_layer


def test_resnet18_parameter_count():
    import synth
    f = _kv("resnet18_params.txt")
    numel = synth.shapes.numels(synth.resnet18_shapes())
    assert abs(sum(numel) / 1e6 - f["params_millions"]) < 0.05
    assert abs(sum(numel) * 4 / 1e6 - f["fp32_mb"]) < 0.1


# --------------------------------------------------------------------------
# the two phases on their own ([D] FSDP reduce-scatter / all-gather)


@pytest.mark.parametrize("n,p", [(1, 9), (2, 7), (5, 23), (8, 64), (7, 3)])
def test_reduce_scatter_leaves_each_worker_its_chunk_of_the_mean(n, p):
    rng = np.random.default_rng(n + 7 * p)
    g = _int_rows(rng, n, p, lim=2 ** 10)
    rows = [r.copy() for r in g]
    owned = oracle.reduce_scatter_avg(rows)
    for w, (b, e) in owned.items():
        assert (b, e) == oracle.chunk_range(p, n, (w + 1) % n)
        for i in range(b, e):
            assert Fraction(float(rows[w][i])) == X.rn_f32(Fraction(sum(int(r[i]) for r in g), n))
    # the owners' chunks tile the array exactly once
    cover = sorted(owned.values())
    assert sum(e - b for b, e in cover) == p


@pytest.mark.parametrize("n", [2, 3, 5, 16])
def test_reduce_scatter_bf16_owned_chunks_match_the_full_ring(n):
    import synth
    p = 4 * n + 3
    g = [synth.student_t3_bf16(3, w, 1e-3, 0, p) for w in range(n)]
    full = [r.copy() for r in g]
    oracle.ring_allreduce_avg_bf16(full)
    rs = [r.copy() for r in g]
    owned = oracle.reduce_scatter_avg(rs)
    for w, (b, e) in owned.items():
        np.testing.assert_array_equal(rs[w][b:e], full[0][b:e])
        # outside its chunk a worker keeps its input
        mask = np.ones(p, bool)
        mask[b:e] = False
        np.testing.assert_array_equal(rs[w][mask], g[w][mask])


@pytest.mark.parametrize("dtype", [np.float32, np.uint16])
@pytest.mark.parametrize("n,p", [(1, 4), (2, 5), (5, 23), (8, 3)])
def test_all_gather_spreads_every_owned_chunk(n, p, dtype):
    # worker (c-1) mod N holds chunk c (marked c+1); everything else is junk
    rows = [np.full(p, 999, dtype) for _ in range(n)]
    for c in range(n):
        b, e = oracle.chunk_range(p, n, c)
        rows[(c - 1) % n][b:e] = c + 1
    oracle.all_gather(rows)
    want = np.empty(p, dtype)
    for c in range(n):
        b, e = oracle.chunk_range(p, n, c)
        want[b:e] = c + 1
    for r in rows:
        np.testing.assert_array_equal(r, want)


def test_reduce_scatter_then_all_gather_is_the_all_reduce():
    rng = np.random.default_rng(17)
    n, p = 6, 1001
    g = [rng.standard_normal(p).astype(np.float32) for _ in range(n)]
    full = [r.copy() for r in g]
    oracle.ring_allreduce_avg_f32(full)
    rows = [r.copy() for r in g]
    oracle.reduce_scatter_avg(rows)
    oracle.all_gather(rows)
    for r in rows:
        np.testing.assert_array_equal(r, full[0])


# --------------------------------------------------------------------------
# bf16 on the wire


def _bf16_fold(vals, start):
    """Left fold from `start` with every partial rounded: fp32 add, then bf16."""
    n = len(vals)
    acc = X.bf16_value(vals[start])
    for k in range(1, n):
        acc = X.rn_bf16(X.rn_f32(X.bf16_value(vals[(start + k) % n]) + acc))
    return acc


@pytest.mark.parametrize("n,p", [(2, 9), (3, 20), (5, 101), (16, 333)])
def test_bf16_wire_rounds_every_partial(n, p):
    import synth
    g = [synth.student_t3_bf16(3, w, 1e-3, 0, p) for w in range(n)]
    rows = [r.copy() for r in g]
    oracle.ring_allreduce_avg_bf16_wire(rows)
    for c in range(n):
        b, e = oracle.chunk_range(p, n, c)
        for i in range(b, e):
            want = X.rn_bf16(X.rn_f32(_bf16_fold([r[i] for r in g], c) / n))
            for r in rows:
                assert X.bf16_value(r[i]) == want


def test_bf16_wire_loses_what_binary32_partials_keep():
    # 256 + 1 + 1 over 3 workers: with bf16 partials 256 + 1 rounds back to
    # 256 (ties to even), so the mean is bf16(256 / 3) = 85.5; binary32
    # partials give 258 / 3 = 86.
    b = [np.array([np.float32(v).view(np.uint32) >> 16], np.uint16) for v in (256.0, 1.0, 1.0)]
    wire = [r.copy() for r in b]
    oracle.ring_allreduce_avg_bf16_wire(wire)
    assert X.bf16_value(wire[0][0]) == Fraction(171, 2)
    f32 = [r.copy() for r in b]
    oracle.ring_allreduce_avg_bf16(f32)
    assert X.bf16_value(f32[0][0]) == 86


@pytest.mark.parametrize("n", [2, 4, 7])
def test_bf16_wire_exact_when_partials_fit(n):
    # integers |v| <= 16 over at most 7 workers: every partial fits bf16
    rng = np.random.default_rng(n)
    p = 3 * n + 1
    vals, rows = _bf16_rows_from_ints(rng, n, p, 16)
    oracle.ring_allreduce_avg_bf16_wire(rows)
    for i in range(p):
        s = sum(int(v[i]) for v in vals)
        assert X.bf16_value(rows[0][i]) == X.rn_bf16(X.rn_f32(Fraction(s, n)))


# --------------------------------------------------------------------------
# single reducer ([G] The Communication Problem)


@pytest.mark.parametrize("n", [1, 2, 3, 8, 13])
def test_single_reducer_folds_in_worker_order(n):
    rng = np.random.default_rng(40 + n)
    p = 50
    choices = np.array([2.0 ** 24, -2.0 ** 24, 1.0, 3.0, -1.0, 0.5], np.float32)
    g = [choices[rng.integers(0, choices.size, p)] for _ in range(n)]
    rows = [r.copy() for r in g]
    sent, recv = oracle.single_reducer_avg(rows)
    for i in range(p):
        want = X.div(_fold([r[i] for r in g], 0), n)
        for r in rows:
            assert Fraction(float(r[i])) == want
    # the reducer receives and sends (N-1)P; every other worker P each way
    assert recv[0] == sent[0] == (n - 1) * p
    assert all(sent[m] == recv[m] == p for m in range(1, n))


def test_single_reducer_cost_figures_of_the_pages():
    f = _kv("gibiansky_cost_figures.txt")
    p = 1000
    for gpus, key in ((2, "single_reducer_extra_s_2gpu"), (10, "single_reducer_extra_s_10gpu")):
        rows = [np.zeros(p, np.float32) for _ in range(gpus)]
        sent, recv = oracle.single_reducer_avg(rows)
        # the reducer's link carries its received elements: scale to 300M fp32
        gb = recv[0] / p * f["params"] * f["bytes_per_param"] / 1e9
        assert abs(gb / f["single_reducer_link_gbps"] - f[key]) < 1e-6


def test_single_reducer_bf16_small_integers():
    rng = np.random.default_rng(41)
    n, p = 5, 17
    vals, rows = _bf16_rows_from_ints(rng, n, p, 256)
    oracle.single_reducer_avg(rows)
    for i in range(p):
        s = sum(int(v[i]) for v in vals)
        assert X.bf16_value(rows[2][i]) == X.rn_bf16(X.rn_f32(Fraction(s, n)))
