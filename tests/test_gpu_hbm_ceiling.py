"""The fused all-reduce against bare data movement on the same GPU.

tests/hbm_patterns.cu moves bytes with the same TMA bulk copies as the fused
kernel and no arithmetic: read only, write only, a 1:1 copy, and the
all-reduce's own in-place pattern (8 rows, one 2 KB tile of each per block,
loaded and stored back), plus two write-grouping schedules and smaller
blocks.  The all-reduce of the benchmark workload (N=8 x P=300M fp32) must
move its bytes at least at 0.97 x the in-place pattern's rate: the fold, the
division and the ring bookkeeping must cost (almost) nothing on top of the
traffic.  The measured table goes to tests/.scratch/hbm_ceiling.json.
"""
from __future__ import annotations

import json
import os
import subprocess

import pytest
import torch

import gradient_ring_all_gb300 as ra

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HERE = os.path.dirname(os.path.abspath(__file__))
SCRATCH = os.path.join(HERE, ".scratch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()


def _patterns(p, reps):
    os.makedirs(SCRATCH, exist_ok=True)
    exe = os.path.join(SCRATCH, "hbm_patterns")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    os.path.join(HERE, "hbm_patterns.cu"), "-o", exe], check=True, capture_output=True, timeout=300)
    r = subprocess.run([exe, str(p), str(reps)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


def _allreduce_gbs(n, p, steps):
    rows = [torch.zeros(p, dtype=torch.float32, device="cuda") for _ in range(n)]
    stream = torch.cuda.current_stream()
    for _ in range(3):
        ra.ra_allreduce_avg(rows, stream)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        ra.ra_allreduce_avg(rows, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del rows
    torch.cuda.empty_cache()
    return 2 * n * p * 4 / (ms / 1e3) / 1e9


def test_allreduce_moves_its_bytes_as_fast_as_a_bare_tma_copy():
    n, p = 8, 300_000_000
    ours = _allreduce_gbs(n, p, 20)
    pat = _patterns(p, 10)
    pat["fused_allreduce"] = ours
    with open(os.path.join(SCRATCH, "hbm_ceiling.json"), "w") as f:
        json.dump(pat, f, indent=1)
    assert pat["waits_expired"] == 0
    # the patterns are ordered as expected of HBM: a 1:1 mix is slower than either direction alone
    assert pat["copy"] < pat["read_only"] and pat["copy"] < pat["write_only"]
    assert ours >= 0.97 * pat["in_place"], pat
