"""bench.py's multi-process path on CPU (gloo, world size 2): the barrier +
max-over-ranks timing of independent replicas, the whole-job aggregate, and
the reference arm under torchrun (rank 0 alone prints)."""
from __future__ import annotations

import json
import os
import shutil
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _WallTimer:
    def sync(self):
        pass

    def start(self):
        self.t0 = time.perf_counter()

    def stop(self):
        self.t1 = time.perf_counter()

    def elapsed_ms(self):
        return (self.t1 - self.t0) * 1e3


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank 1 is the slow replica: 4 steps of 30 ms against rank 0's 4 x 5 ms
    delay = 0.005 if rank == 0 else 0.030
    mine, slowest = bench.timed_region(lambda k: time.sleep(delay), 4, dist, _WallTimer())
    q.put((rank, mine, slowest, bench.aggregate_gbs(1e9, world, slowest / 4)))
    dist.destroy_process_group()


def test_replica_timing_takes_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, mine0, max0, val0), (r1, mine1, max1, val1) = res
    assert max0 == max1 == max(mine0, mine1)
    assert mine1 >= 120.0 and mine0 < mine1
    # both replicas' bytes over the slowest replica's time
    assert abs(val0 - 2 * 1e9 / (max0 / 4 / 1e3) / 1e9) < 1e-9


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    scratch = os.path.join(ROOT, "tests", ".scratch")  # torchrun's own files stay in the repo (git-ignored)
    os.makedirs(scratch, exist_ok=True)
    env = dict(os.environ, OMP_NUM_THREADS="1", TMPDIR=scratch)
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    finally:
        shutil.rmtree(scratch, ignore_errors=True)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def _failing_rank_main(rank, world, port, mode, q):
    # rank 1 fails between steps: it exits, or stops answering; rank 0 must
    # get an error from its next barrier instead of waiting for it forever
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      RA_BENCH_PG_TIMEOUT_S="5")
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_replicas()
    bench.timed_region(lambda k: None, 1, dist, _WallTimer())  # one good step together
    if rank == 1:
        if mode == "exit":
            os._exit(3)
        time.sleep(40)  # stops answering
        os._exit(0)
    t0 = time.perf_counter()
    try:
        bench.timed_region(lambda k: None, 1, dist, _WallTimer())
        q.put((rank, "no error", time.perf_counter() - t0))
    except Exception as e:  # the failure surfaces as an exception
        q.put((rank, type(e).__name__, time.perf_counter() - t0))


@pytest.mark.parametrize("mode", ["exit", "hang"])
def test_a_failed_replica_surfaces_as_an_error_not_a_hang(mode):
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_failing_rank_main, args=(r, 2, port, mode, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        rank, outcome, waited = q.get(timeout=120)
    finally:
        for p in procs:
            p.join(timeout=10)
            if p.is_alive():
                p.kill()  # our own child (the rank that stopped answering)
                p.join()
    assert rank == 0
    assert outcome != "no error"
    assert waited < 30, waited  # the 5 s timeout, not the default 30 minutes
