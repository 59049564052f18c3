"""Seeded random sweep over every entry point: worker counts 1..64, lengths
spread log-uniformly from 0 to 40,000, both dtypes, four pointer layouts,
random bucket plans -- each result bit-exact against the CPU oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth
from gpu_util import to_device_rows, to_host

pytestmark = pytest.mark.gpu

CALLS = ["avg", "staged", "staged_static", "sgd", "reduce_scatter", "all_gather", "bf16_wire", "single_reducer",
         "buckets"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _case(seed):
    rng = np.random.default_rng(seed)
    call = CALLS[seed % len(CALLS)]
    n = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 9, 12, 16, 17, 31, 32, 33, 48, 64]))
    p = int(np.exp(rng.uniform(0, np.log(40_000)))) if rng.random() > 0.05 else 0
    dtype = "bf16" if call == "bf16_wire" else str(rng.choice(["f32", "bf16"]))
    layout = str(rng.choice(["separate", "offset", "mixed", "packed"]))
    pad = int(rng.integers(0, 8))
    return rng, call, n, p, dtype, layout, pad


@pytest.mark.parametrize("seed", range(180))
def test_random_case(seed):
    rng, call, n, p, dtype, layout, pad = _case(seed)
    if dtype == "f32":
        host = [(synth.normal_f32(seed, k, 1.0, 0, p) * np.float32(rng.choice([1e-3, 1.0, 1e3]))).astype(np.float32)
                for k in range(n)]
    else:
        host = [synth.student_t3_bf16(seed, k, float(rng.choice([1e-3, 1.0])), 0, p) for k in range(n)]
    rows = to_device_rows(host, layout=layout, pad=pad)
    want = [h.copy() for h in host]
    rs_owned = None
    if call in ("avg", "staged", "staged_static"):
        (oracle.ring_allreduce_avg_f32 if dtype == "f32" else oracle.ring_allreduce_avg_bf16)(want)
        {"avg": lambda: ra.ra_allreduce_avg(rows), "staged": lambda: ra.ra_allreduce_avg_staged(rows),
         "staged_static": lambda: ra.ra_allreduce_avg_staged_static(rows)}[call]()
    elif call == "sgd":
        (oracle.ring_allreduce_avg_f32 if dtype == "f32" else oracle.ring_allreduce_avg_bf16)(want)
        w0 = synth.normal_f32(seed + 1, 0, 0.05, 0, p)
        w_want = w0.copy()
        oracle.sgd_update_f32(w_want, want[0], 0.1)
        wbase = torch.empty(p + 8, dtype=torch.float32, device="cuda")
        woff = int(rng.integers(0, 4))
        w = wbase[woff:woff + p]
        w.copy_(torch.from_numpy(w0))
        ra.ra_allreduce_sgd(rows, w, 0.1)
    elif call == "reduce_scatter":
        rs_owned = oracle.reduce_scatter_avg(want)
        ra.ra_reduce_scatter_avg(rows)
    elif call == "all_gather":
        oracle.all_gather(want)
        ra.ra_all_gather(rows)
    elif call == "bf16_wire":
        oracle.ring_allreduce_avg_bf16_wire(want)
        ra.ra_allreduce_avg_bf16_wire(rows)
    elif call == "single_reducer":
        oracle.single_reducer_avg(want)
        ra.ra_allreduce_avg_single_reducer(rows)
    else:  # buckets
        cuts = np.sort(rng.integers(0, p + 1, int(rng.integers(0, 12))))
        numel = np.diff(np.concatenate([[0], cuts, [p]])).tolist()
        plan = oracle.bucket_plan(numel, 4 if dtype == "f32" else 2, int(rng.integers(16, 4096)))
        for off, cnt in plan:
            sub = [r[off:off + cnt] for r in want]
            (oracle.ring_allreduce_avg_f32 if dtype == "f32" else oracle.ring_allreduce_avg_bf16)(sub)
        ra.ra_allreduce_avg_buckets(rows, plan)
    torch.cuda.synchronize()
    for k, r in enumerate(rows):
        got = to_host(r)
        if rs_owned is not None:
            b, e = rs_owned[k]
            np.testing.assert_array_equal(_bits(got[b:e]), _bits(want[k][b:e]), err_msg=str((call, n, p, dtype, layout)))
        else:
            np.testing.assert_array_equal(_bits(got), _bits(want[k]), err_msg=str((call, n, p, dtype, layout)))
    if call == "sgd":
        np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), w_want.view(np.uint32))
