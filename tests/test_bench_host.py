"""Host-side helpers of bench.py (no GPU): the source hash that keys the
committed ncu traffic figures follows the code, not its comments (the bench
reports the traffic only while the hash matches); the two arms print the
same config object; call_bytes follows each call's design."""
from __future__ import annotations

import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _copy_csrc(tag):
    d = os.path.join(ROOT, "tests", ".scratch", "csrc_" + tag)
    shutil.rmtree(d, ignore_errors=True)
    shutil.copytree(os.path.join(ROOT, "gradient_ring_all_gb300", "csrc"), d)
    return d


def test_source_hash_ignores_comments_but_not_code():
    base = bench._source_hash()
    d = _copy_csrc("comments")
    try:
        assert bench._source_hash(d) == base
        f = os.path.join(d, "ra_kernels.cuh")
        src = open(f).read()
        open(f, "w").write("// a new comment\n/* and a block\n comment */\n" + src.replace("\n", "\n  ", 3))
        assert bench._source_hash(d) == base  # comments and indentation only
        open(f, "w").write(src.replace("kWaitLimitNs = 2000000000ull", "kWaitLimitNs = 1000000000ull"))
        assert bench._source_hash(d) != base  # a code change
    finally:
        shutil.rmtree(d, ignore_errors=True)


def test_both_arms_print_one_config():
    wl = synth.WORKLOADS["speech300m_n8_f32"]
    c = bench._config(wl, wl.n, wl.p, 1)
    assert c["workload"] == "speech300m_n8_f32" and c["workers"] == 8 and c["elements_per_worker"] == 300_000_000
    assert c["bytes_per_step"] == 19_200_000_000 and c["parallelism"] == "single GPU"
    assert bench._config(wl, wl.n, wl.p, 4)["parallelism"] == "replicas"


def test_call_bytes():
    n, p = 8, 300_000_000
    assert bench.call_bytes("allreduce", n, p, 4) == 2 * n * p * 4
    assert bench.call_bytes("sgd", n, p, 4) == 2 * n * p * 4 + 2 * p * 4
    assert bench.call_bytes("reduce_scatter", n, p, 4) == (n + 1) * p * 4
    assert bench.call_bytes("all_gather", n, p, 4) == n * p * 4
    assert bench.call_bytes("staged", n, p, 4) == 44_400_000_000  # (5(N-1)+2) P s


def test_bucket_tensors_cut_to_the_rows():
    # a reduced --elements run plans buckets only over the tensors that fit,
    # so that no bucket reaches past the rows it is given
    wl = synth.WORKLOADS["transformer24_buckets_n4_f32"]
    for p in (1, 65_536_000, 100_000_000, wl.p):
        t = bench.tensors_within(wl.tensors, p)
        assert sum(t) == p and all(x > 0 for x in t)
        assert t[:-1] == list(wl.tensors[:len(t) - 1])
    assert bench.tensors_within(wl.tensors, wl.p) == list(wl.tensors)


def test_result_check_finds_any_wrong_element():
    # bench.py's check of the call it timed: worker 0's row against the
    # oracle's result on every element, the other workers against worker 0,
    # the SGD weights against theirs.  Host tensors stand in for device rows.
    import numpy as np
    import torch
    rng = np.random.default_rng(5)
    for bf16 in (False, True):
        p = 1000
        mean = rng.standard_normal(p).astype(np.float32)
        if bf16:
            mean = (mean.view(np.uint32) >> 16).astype(np.uint16)
            rows = [torch.from_numpy(mean.view(np.int16).copy()).view(torch.bfloat16) for _ in range(3)]
        else:
            rows = [torch.from_numpy(mean.copy()) for _ in range(3)]
        w = torch.from_numpy(rng.standard_normal(p).astype(np.float32))
        wexp = w.numpy().copy()
        assert bench.check_result(rows, mean, w, wexp, slice_elems=256) == {"bit_exact": True, "first_mismatch": None}
        bits = torch.int16 if bf16 else torch.int32
        for who, idx in ((0, 777), (2, 3)):  # one flipped low bit in worker 0, then in worker 2
            rows[who].view(bits)[idx] ^= 1
            r = bench.check_result(rows, mean, w, wexp, slice_elems=256)
            assert r["bit_exact"] is False and str(who if who else idx) in r["first_mismatch"], r
            rows[who].view(bits)[idx] ^= 1
        w.view(torch.int32)[999] ^= 1
        r = bench.check_result(rows, mean, w, wexp, slice_elems=256)
        assert r["bit_exact"] is False and r["first_mismatch"] == "weights, element 999"


def test_per_config_covers_every_other_workload():
    # the recorded benchmark line measures and verifies every configuration:
    # the headline, plus each other workload (the bucketed one both ways)
    names = {w for w, _ in bench.PER_CONFIG}
    assert names | {bench.WORKLOAD} == set(synth.WORKLOADS)
    assert ("transformer24_buckets_n4_f32", "buckets") in bench.PER_CONFIG
    assert ("transformer24_buckets_n4_f32", "buckets_each") in bench.PER_CONFIG
    assert ("resnet18_sgd_n32_f32", "sgd") in bench.PER_CONFIG
    for _, call in bench.PER_CONFIG:
        assert call in bench.CALLS
