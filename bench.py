#!/usr/bin/env python3
"""Benchmark: fused ring all-reduce-average, N=8 workers x P=300M fp32.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one ra_allreduce_avg over the 8 workers' 1.2 GB fp32 gradient
arrays (the 300M-parameter speech model of Gibiansky, "The Communication
Problem"), inputs resident in HBM.  The metric is HBM GB/s over the minimum
traffic of the all-reduce, 2*N*P*4 bytes per step (every input read once,
the mean written to every worker once).  One JSON line is printed by rank 0.

--gpus N > 1 runs under torchrun as N independent replicas (the path has no
exchange between GPUs: all workers live in one GPU's memory); value sums the
replicas' bytes over the slowest replica's time.

--impl reference times the CPU oracle (a literal, single-threaded
simulation of the ring) on a bounded sample of the same workload.

The CPU leg is the only part of this file that runs the oracle: it times it
on a bounded sample (cpu_baseline, and the reference arm), and it computes
the result each verified call must produce, from host copies of that call's
inputs (fill_workload with verify, then check_result).  The GPU path never
reads anything the oracle produced.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "all-reduce-avg HBM GB/s and % of GB300 peak at N=8, P=300M fp32"
WORKLOAD = "speech300m_n8_f32"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
CPU_SAMPLE_P = 25_000_000  # elements per worker in the oracle's bounded sample


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# A replica that dies or stops between steps must not hold the others (and
# their GPUs) for the default 30-minute collective timeout: their next
# barrier fails after this many seconds instead.
PG_TIMEOUT_S = float(os.environ.get("RA_BENCH_PG_TIMEOUT_S", "600"))


def init_replicas():
    """The replicas' gloo group, with the bounded timeout above."""
    import datetime
    import torch.distributed as dist
    dist.init_process_group("gloo", timeout=datetime.timedelta(seconds=PG_TIMEOUT_S))
    return dist


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class _ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in (out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        loaded = [x for x in sm if smax and x >= 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


def _code_only(src: str) -> str:
    """C/CUDA source without comments and with whitespace collapsed, so that
    the hash changes with the code and not with its comments."""
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return " ".join(src.split())


def _source_hash(csrc_dir: str | None = None) -> str:
    h = hashlib.sha256()
    d = csrc_dir or os.path.join(ROOT, "gradient_ring_all_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(d, f), encoding="utf-8") as fh:
                h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def _traffic_from_profile(kernel_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_hash") == _source_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def max_over_ranks(x: float, dist) -> float:
    """The largest value of x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0])


def aggregate_gbs(bytes_per_step: float, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every replica's bytes over the slowest replica's time."""
    return bytes_per_step * world / (ms_per_step / 1e3) / 1e9


def timed_region(step, steps: int, dist, timer):
    """Barrier, `steps` calls of step(k), barrier; returns (this rank's ms,
    the max over ranks).  `timer` brackets the region: start(), stop(),
    sync(), elapsed_ms()."""
    if dist is not None:
        dist.barrier()
    timer.sync()
    timer.start()
    for k in range(steps):
        step(k)
    timer.stop()
    timer.sync()
    if dist is not None:
        dist.barrier()
    ms = timer.elapsed_ms()
    return ms, max_over_ranks(ms, dist)


class _CudaEventTimer:
    def __init__(self, stream):
        import torch
        self.torch = torch
        self.stream = stream
        self.a = torch.cuda.Event(enable_timing=True)
        self.b = torch.cuda.Event(enable_timing=True)

    def sync(self):
        self.torch.cuda.synchronize()

    def start(self):
        self.a.record(self.stream)

    def stop(self):
        self.b.record(self.stream)

    def elapsed_ms(self):
        return self.a.elapsed_time(self.b)


def _cpu_oracle_sample(n: int, p: int, reps: int):
    """Time the oracle (as it stands) on a bounded sample: a ring of n workers
    x p elements of the workload's distribution.  Returns (GB/s, seconds)."""
    import oracle
    import synth
    wl = synth.WORKLOADS[WORKLOAD]
    rows = [synth.normal_f32(wl.seed, k, wl.scale, 0, p) for k in range(n)]
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.ring_allreduce_avg_f32(rows)
    dt = time.perf_counter() - t0
    return 2.0 * n * p * 4 * reps / dt / 1e9, dt


def _oracle_step(wl, rows, w, plan):
    """One oracle run of the workload's call on host rows, in place."""
    import oracle
    if plan:
        for off, cnt in plan:
            sub = [r[off:off + cnt] for r in rows]
            (oracle.ring_allreduce_avg_f32 if wl.dtype == "f32" else oracle.ring_allreduce_avg_bf16)(sub)
    elif wl.dtype == "f32":
        oracle.ring_allreduce_avg_f32(rows)
    else:
        oracle.ring_allreduce_avg_bf16(rows)
    if w is not None:
        oracle.sgd_update_f32(w, rows[0], wl.sgd_lr)


def _config(wl, n, p, ws):
    """The `config` object of the bench line (both arms print the same one)."""
    esz = 4 if wl.dtype == "f32" else 2
    return {"workload": wl.name, "workers": n, "elements_per_worker": p,
            "distribution": "N(0, %g), seed %d, worker n = generator stream n" % (wl.scale, wl.seed),
            "bytes_per_step": 2 * n * p * esz, "parallelism": "replicas" if ws > 1 else "single GPU",
            "l2": "inputs of %.1f GB per GPU, larger than the 129 MB L2; no flush" % (n * p * esz / 1e9)}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    import oracle
    import synth
    oracle.build()
    synth.build()
    wl = synth.WORKLOADS[args.workload]
    esz = 4 if wl.dtype == "f32" else 2
    # per-step sample: at most 8 x 25M values (about 0.6 s of one core), fewer
    # when W + K steps would otherwise take more than about a minute
    values = min(8 * CPU_SAMPLE_P, 8 * CPU_SAMPLE_P * 100 // (args.steps + args.warmup))
    p = int(min(wl.p, max(1_000_000 // wl.n, values // wl.n)))
    rows = [wl.row(k, 0, p) for k in range(wl.n)]
    w = wl.weights(0, p) if wl.sgd_lr > 0 else None
    plan = None
    if wl.bucket_cap_bytes:
        # the workload's reverse-order buckets over the first p elements
        plan = oracle.bucket_plan(tensors_within(wl.tensors, p), esz, wl.bucket_cap_bytes)
    for _ in range(args.warmup):
        _oracle_step(wl, rows, w, plan)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _oracle_step(wl, rows, w, plan)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    nbytes = 2 * wl.n * p * esz + (2 * p * 4 if w is not None else 0)
    value = nbytes * args.steps / total / 1e9
    sample = ("N=%d workers x P=%d %s elements of %s per step (a bounded sample of its P=%d), in place, "
              "one core" % (wl.n, p, wl.dtype, wl.name, wl.p))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic", "config": _config(wl, wl.n, wl.p, ws),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# inputs, and the check of what a call produced


def fill_workload(wl, rows, w=None, rings=None, verify=False, slice_elems=1 << 24, sub_elems=1 << 15):
    """Generate the workload's rows (and its SGD weights) on the host, slice
    by slice, and copy them to the device tensors `rows` (and `w`).

    With `verify`, the CPU oracle's range evaluation runs on the same host
    slices, so the result of the workload's call is known for every element:
    returns (mean row, weights after the SGD step or None) as host arrays
    (float32, or uint16 bf16 bits).  Without it, returns (None, None).
    rings: [(offset, count)] element ranges reduced as rings of their own
    (the buckets), or None for one ring of all p elements.  The oracle only
    reads the host copies of the inputs: it checks the GPU's result and is
    never on the path that produces it."""
    import numpy as np
    import torch
    from concurrent.futures import ThreadPoolExecutor
    n, p = wl.n, wl.p
    bf16 = wl.dtype == "bf16"
    hdt = np.uint16 if bf16 else np.float32
    s_el = min(slice_elems, max(1, p))
    host = torch.empty((n, s_el), dtype=torch.int16 if bf16 else torch.float32).pin_memory()
    hnp = host.numpy().view(hdt)
    hw = torch.empty(s_el, dtype=torch.float32).pin_memory() if w is not None else None
    mean = wexp = None
    if verify:
        import oracle
        mean = np.empty(p, hdt)
        wexp = np.empty(p, np.float32) if w is not None else None
    stream = torch.cuda.current_stream()
    with ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
        for off, cnt in ([(0, p)] if rings is None else rings):
            for s in range(0, cnt, s_el):
                c, g = min(s_el, cnt - s), off + s
                for k in range(n):
                    wl.fill_row(host[k].data_ptr(), k, g, c)
                    rows[k][g:g + c].copy_(host[k, :c].view(torch.bfloat16) if bf16 else host[k, :c],
                                           non_blocking=True)
                if w is not None:
                    wl.fill_weights(hw.data_ptr(), g, c)
                    w[g:g + c].copy_(hw[:c], non_blocking=True)
                if verify:
                    def part(a, s=s, c=c, g=g, cnt=cnt):
                        b = min(c, a + sub_elems)
                        oracle.ring_avg_range([hnp[k, a:b] for k in range(n)], cnt, s + a, out=mean[g + a:g + b])
                        if wexp is not None:
                            wexp[g + a:g + b] = hw.numpy()[a:b]
                            oracle.sgd_update_f32(wexp[g + a:g + b], mean[g + a:g + b], wl.sgd_lr)

                    list(ex.map(part, range(0, c, sub_elems)))
                stream.synchronize()  # the copies are done with the host slice
    return mean, wexp


def _bits(a):
    """Integer view of a host array of float32 or bf16 bits, for bitwise comparison."""
    import numpy as np
    return a.view(np.uint16) if a.dtype == np.uint16 else a.view(np.uint32)


def _host_bits(t):
    """A device tensor's values as host integers (bf16 -> uint16, float32 -> uint32)."""
    import numpy as np
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint32)


def check_result(rows, mean, w=None, wexp=None, slice_elems=1 << 26):
    """Compare a call's result with the oracle's on every element: worker
    0's row read back whole against `mean`, every other worker's row against
    worker 0's on the device, and the SGD weights against `wexp`.  Returns
    {"bit_exact": bool, "first_mismatch": None or where}."""
    import numpy as np
    import torch

    def first_diff(dev, want):
        for s in range(0, want.shape[0], slice_elems):
            e = min(want.shape[0], s + slice_elems)
            d = np.flatnonzero(_host_bits(dev[s:e]) != _bits(want[s:e]))
            if d.size:
                return s + int(d[0])
        return None

    i = first_diff(rows[0], mean)
    if i is not None:
        return {"bit_exact": False, "first_mismatch": "worker 0, element %d" % i}
    iv = torch.int16 if rows[0].dtype == torch.bfloat16 else torch.int32
    for k, r in enumerate(rows[1:], 1):
        if not torch.equal(rows[0].view(iv), r.view(iv)):
            return {"bit_exact": False, "first_mismatch": "worker %d differs from worker 0" % k}
    if wexp is not None:
        i = first_diff(w, wexp)
        if i is not None:
            return {"bit_exact": False, "first_mismatch": "weights, element %d" % i}
    return {"bit_exact": True, "first_mismatch": None}


def error_vs_binary64(wl, mean, count=200_000, seed=11):
    """The binary32 ring mean against the binary64 mean of the inputs, on
    `count` random elements (regenerated from the seeded generator): the
    norm-relative error, and the largest element error in units of the mean
    absolute input (the recursive-summation bound makes that (N-1)u at
    most; the stated tolerance is 1e-5)."""
    import numpy as np
    idx = np.unique(np.random.default_rng(seed).integers(0, wl.p, count)).astype(np.int64)
    vals = np.stack([wl.values_at(k, idx).astype(np.float64) for k in range(wl.n)])
    m64 = vals.mean(axis=0)
    err = mean[idx].astype(np.float64) - m64
    return {"norm": float(np.linalg.norm(err) / np.linalg.norm(m64)),
            "max_elementwise": float(np.max(np.abs(err) / np.abs(vals).mean(axis=0))),
            "sample": "%d random elements" % idx.size}


def _time_steps(step, steps, stream, dist=None):
    """CUDA events around each call on the launch stream, inside the
    barrier-bracketed timed region; returns (total ms max over ranks, mean
    ms per call)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]

    def one(k):
        starts[k].record(stream)
        step()
        ends[k].record(stream)

    _, total_ms = timed_region(one, steps, dist, _CudaEventTimer(stream))
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return total_ms, sum(per) / len(per)


# the other configurations of the benchmark, each measured the way the
# headline is: inputs filled from the seeded generator, the first call
# compared with the oracle on every element, then timed
PER_CONFIG = (("ring4_uneven_1m_f32", "allreduce"), ("transformer24_buckets_n4_f32", "buckets"),
              ("transformer24_buckets_n4_f32", "buckets_each"), ("student_t3_1g_n16_bf16", "allreduce"),
              ("resnet18_sgd_n32_f32", "sgd"))


def graph_rate(ra, rows, nbytes, peak, calls=100, replays=10):
    """The same all-reduce captured `calls` times in one CUDA graph and
    replayed: the GPU's own time per call, without the host's per-call cost
    (which bounds a call this small when it is issued from Python)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ra.ra_allreduce_avg(rows, torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            ra.ra_allreduce_avg(rows, torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    ms, _ = timed_region(lambda k: g.replay(), replays, None, _CudaEventTimer(torch.cuda.current_stream()))
    per = ms / replays / calls
    gbs = nbytes / (per / 1e3) / 1e9
    return {"calls_per_graph": calls, "replays": replays, "ms_per_call": per, "gbs": gbs, "frac": gbs / peak}


def measure_config(ra, wl, calls, steps, warmup, peak):
    """One workload, one or more calls on it: verified first call, then
    `warmup` more and `steps` timed.  Returns one result dict per call."""
    import torch
    stream = torch.cuda.current_stream()
    bf16 = wl.dtype == "bf16"
    esz = 2 if bf16 else 4
    rows = [torch.empty(wl.p, dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda") for _ in range(wl.n)]
    w = torch.empty(wl.p, dtype=torch.float32, device="cuda") if wl.sgd_lr > 0 else None
    plan = ra.ra_bucket_plan(wl.tensors, esz, wl.bucket_cap_bytes) if wl.bucket_cap_bytes else None
    mean, wexp = fill_workload(wl, rows, w, rings=plan, verify=True)
    # every call starts from the same inputs: a device copy to restore them
    keep = [r.clone() for r in rows] + ([w.clone()] if w is not None else []) if len(calls) > 1 else None
    out = []
    for j, call in enumerate(calls):
        if j > 0:
            for r, k in zip(rows + ([w] if w is not None else []), keep):
                r.copy_(k)
        if call == "allreduce":
            step = lambda: ra.ra_allreduce_avg(rows, stream)
        elif call == "sgd":
            step = lambda: ra.ra_allreduce_sgd(rows, w, wl.sgd_lr, stream)
        elif call == "buckets":
            step = lambda: ra.ra_allreduce_avg_buckets(rows, plan, stream)
        else:  # buckets_each: one call, and so one launch, per bucket, output side first
            def step():
                for b in plan:
                    ra.ra_allreduce_avg_buckets(rows, [b], stream)
        step()
        torch.cuda.synchronize()
        chk = check_result(rows, mean, w, wexp)
        for _ in range(warmup - 1):
            step()
        # the whole region over the calls (no event between two calls, which
        # would keep the next launch from overlapping the current one's tail);
        # more calls for a workload that fits the L2 and takes microseconds
        small = wl.n * wl.p * esz < 129e6
        k_steps = max(steps, 200) if small else steps
        ms, _ = timed_region(lambda k: step(), k_steps, None, _CudaEventTimer(stream))
        ms /= k_steps
        nbytes = call_bytes(call, wl.n, wl.p, esz)
        graph = graph_rate(ra, rows, nbytes, peak) if small and call == "allreduce" else None
        torch.cuda.synchronize()
        st = ra.ra_check_device_errors()
        gbs = nbytes / (ms / 1e3) / 1e9
        res = {"workload": wl.name, "call": call, "workers": wl.n, "elements_per_worker": wl.p, "dtype": wl.dtype,
               "bytes_per_call": nbytes, "ms_per_call": ms, "gbs": gbs, "frac": gbs / peak,
               "pct_of_nominal_hbm": 100.0 * gbs / NOMINAL_HBM_GBS, "steps": k_steps,
               "bit_exact": chk["bit_exact"] and st == ra.RA_OK,
               "device_errors": ra.ra_status_str(st)}
        if chk["first_mismatch"]:
            res["first_mismatch"] = chk["first_mismatch"]
        if plan:
            res["buckets"] = len(plan)
            res["launches_per_call"] = len(plan) if call == "buckets_each" else 1
        if small:
            res["note"] = ("inputs of %.1f MB fit the 129 MB L2; issued from Python the call is bound by the host's "
                           "per-call cost (cuda_graph: the same calls replayed from a graph)" % (wl.n * wl.p * esz / 1e6))
        if graph:
            res["cuda_graph"] = graph
        out.append(res)
    del rows, w, keep
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import dataclasses

    import torch
    ws, rank, local = _dist()
    if args.gpus > 1 and ws == 1:
        print("bench.py: --gpus %d needs torchrun (one process per GPU)" % args.gpus, file=sys.stderr)
        return 2
    torch.cuda.set_device(local)
    dist = None
    if ws > 1:
        dist = init_replicas()
    from gradient_ring_all_gb300 import build
    build.build()
    import gradient_ring_all_gb300 as ra
    import synth
    ra.load()
    wl = synth.WORKLOADS[WORKLOAD]
    if args.elements:
        wl = dataclasses.replace(wl, p=args.elements)
    n, p = wl.n, wl.p
    nbytes = 2 * n * p * 4  # every input read once, the mean written to every worker once
    verify = args.legs == "all"

    # inputs: each worker's row generated on the host, copied to its own
    # allocation; the oracle's result for every element computed beside it
    rows = [torch.empty(p, dtype=torch.float32, device="cuda") for _ in range(n)]
    mean, _ = fill_workload(wl, rows, verify=verify)
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    # the first warm-up call runs on the fresh inputs: its result is compared
    # with the oracle's on every element (the timed calls then re-average
    # rows that are already identical, which moves the same bytes)
    ra.ra_allreduce_avg(rows, stream)
    torch.cuda.synchronize()
    check = check_result(rows, mean) if verify else None
    err64 = error_vs_binary64(wl, mean) if verify and check["bit_exact"] else None
    del mean
    for _ in range(args.warmup - 1):
        ra.ra_allreduce_avg(rows, stream)
    torch.cuda.synchronize()

    # timed region: K launches, an event pair around each on the launch stream
    clocks = _ClockSampler(local).start()
    time.sleep(0.3)
    w0 = time.time()
    total_ms, avg_kernel_ms = _time_steps(lambda: ra.ra_allreduce_avg(rows, stream), args.steps, stream, dist)
    w1 = time.time()
    clk = clocks.stop(w0, w1)
    # a bounded wait that gave up inside the timed region would have skipped
    # its block's stores: the device's error word must be clean
    torch.cuda.synchronize()
    dev_status = ra.ra_check_device_errors()
    ms_per_step = total_ms / args.steps
    value = aggregate_gbs(nbytes, ws, ms_per_step)

    if args.legs == "device":
        # profiling runs (e.g. a smaller --elements under ncu): device loop only
        if rank == 0:
            print(json.dumps({"profile_run": True, "workload": WORKLOAD, "workers": n, "elements_per_worker": p,
                              "ms_per_step": total_ms / args.steps,
                              "gbs": nbytes / (total_ms / args.steps / 1e3) / 1e9,
                              "device_errors": ra.ra_status_str(dev_status)}), flush=True)
        if dist:
            dist.destroy_process_group()
        return 0 if dev_status == ra.RA_OK else 3

    # end to end through the host-buffer entry point: every step the fused
    # kernel reads the 8 pinned host rows and writes the mean back to all of
    # them over NVLink-C2C (the direct path); the staged path (copy in,
    # reduce, copy out on the copy engines) is timed beside it for context
    e2e_steps = max(1, min(args.steps, 10))
    hrows = [torch.empty(p, dtype=torch.float32).pin_memory() for _ in range(n)]
    for k in range(n):
        hrows[k].copy_(rows[k])

    def time_host(mode, steps):
        ra.ra_allreduce_avg_host(hrows, rows, mode, stream)  # warm-up
        _, ms = timed_region(lambda k: ra.ra_allreduce_avg_host(hrows, rows, mode, stream), steps, dist,
                             _CudaEventTimer(stream))
        return ms / steps

    e2e_ms = time_host(ra.RA_HOST_DIRECT, e2e_steps)
    staged_ms = time_host(ra.RA_HOST_STAGED, max(1, e2e_steps // 2))
    del hrows
    torch.cuda.synchronize()
    host_status = ra.ra_check_device_errors()
    del rows
    torch.cuda.empty_cache()

    peak, peak_kind = _peaks()
    per_config = None
    if ws == 1 and not args.elements and args.per_config:
        per_config = []
        done = {}
        for name, call in PER_CONFIG:
            done.setdefault(name, []).append(call)
        for name, calls in done.items():
            per_config += measure_config(ra, synth.WORKLOADS[name], calls, args.config_steps, 3, peak)

    # every replica verified its own first call and timed region
    mine = bool(check and check["bit_exact"]) and dev_status == ra.RA_OK and host_status == ra.RA_OK
    bit_exact = max_over_ranks(0.0 if mine else 1.0, dist) == 0.0
    if rank != 0:
        dist.destroy_process_group()
        return 0 if mine or not verify else 3

    achieved = nbytes / (avg_kernel_ms / 1e3) / 1e9
    cpu_gbs, cpu_s, reps = None, None, 16
    if ws == 1:
        cpu_gbs, cpu_s = _cpu_oracle_sample(n, CPU_SAMPLE_P, reps)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": _config(wl, n, p, ws),
        "bit_exact": bit_exact,
        "max_rel_err_vs_f64": err64,
        "verification": {"first_call": "every element of worker 0's row against the CPU oracle's ring over the same "
                                       "inputs; every other worker's row against worker 0's",
                         "first_mismatch": check and check["first_mismatch"],
                         "device_errors_after_timed_region": ra.ra_status_str(dev_status),
                         "device_errors_after_e2e": ra.ra_status_str(host_status)},
        "pct_of_measured_hbm": 100.0 * value / ws / peak,
        "pct_of_nominal_hbm": 100.0 * value / ws / NOMINAL_HBM_GBS,
        "elements_per_s": n * p * ws / (ms_per_step / 1e3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": "%s copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" % peak_kind
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "kernel": "fused_tma_kernel<F32, N=8, kOutAll>", "avg_launch_ms": avg_kernel_ms,
                     "traffic": _traffic_from_profile("fused_f32_n8_speech300m")},
        "e2e": {"value": aggregate_gbs(nbytes, ws, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": n * p * 4, "d2h_bytes_per_step": n * p * 4,
                "path": "ra_allreduce_avg_host, direct: the fused kernel reads the pinned host rows and "
                        "writes the mean back to every host row over NVLink-C2C"},
        "e2e_staged": {"value": aggregate_gbs(nbytes, ws, staged_ms), "unit": "GB/s", "ms_per_step": staged_ms,
                       "path": "ra_allreduce_avg_host, staged: cudaMemcpyAsync in, fused kernel, cudaMemcpyAsync out"},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if per_config is not None:
        line["per_config"] = per_config
    if args.elements:
        line["config"]["note"] = "reduced --elements: not the benchmark configuration"
    if cpu_gbs is not None:
        line["cpu_baseline"] = {"value": cpu_gbs, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": "%d in-place runs of a ring of N=%d x P=%d fp32 elements (%.1f s)"
                                          % (reps, n, CPU_SAMPLE_P, cpu_s),
                                "host_cpus": os.cpu_count()}
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    ok = bit_exact and all(c["bit_exact"] for c in (per_config or []))
    return 0 if ok or not verify else 3


CALLS = ("allreduce", "staged", "sgd", "buckets", "buckets_each", "reduce_scatter", "all_gather", "single_reducer",
         "bf16_wire", "host", "host_link")


def call_bytes(call: str, n: int, p: int, esz: int) -> int:
    """Algorithmic bytes one call moves: every byte its design must read or
    write once (the staged ring's own schedule for `staged`)."""
    if call in ("allreduce", "buckets", "buckets_each", "single_reducer", "bf16_wire", "host"):
        return 2 * n * p * esz
    if call == "sgd":
        return 2 * n * p * esz + 2 * p * 4
    if call == "reduce_scatter":
        return (n + 1) * p * esz
    if call == "all_gather":
        return n * p * esz
    if call == "staged":
        if esz == 4:  # in place: 3P per scatter step, 2P divide, 2P per gather step
            return (5 * (n - 1) + 2) * p * 4
        # bf16: binary32 partials -- 2+2+4 (first step), 2+4+4 (others), 4+2 divide, 2+2 per gather
        return (8 + 10 * (n - 2) + 6 + 4 * (n - 1)) * p
    raise ValueError(call)


def tensors_within(numel, p):
    """The leading layer tensors that fit p elements (the last one cut), so
    that a bucket plan over them stays inside rows of p elements."""
    out, left = [], p
    for t in numel:
        if left <= 0:
            break
        out.append(min(int(t), left))
        left -= out[-1]
    return out


def run_profile_call(args):
    """Device-only timing of one entry point on one workload (the launch
    configuration profiled under ncu); inputs from a seeded torch generator
    on the device, since only the traffic matters here."""
    import torch
    from gradient_ring_all_gb300 import build
    build.build()
    import gradient_ring_all_gb300 as ra
    import synth
    wl = synth.WORKLOADS[args.workload]
    n, p = (args.workers or wl.n), (args.elements or wl.p)
    bf16 = wl.dtype == "bf16"
    esz = 2 if bf16 else 4
    g = torch.Generator(device="cuda")
    g.manual_seed(wl.seed)
    rows = []
    dt = torch.bfloat16 if bf16 else torch.float32
    if args.layout == "strided":
        # rows back to back with a stride of p + 1 elements: they disagree
        # modulo 16 bytes, the case of the unaligned kernel
        big = torch.empty(n * (p + 1), dtype=dt, device="cuda")
        rows = [big[k * (p + 1):k * (p + 1) + p] for k in range(n)]
    else:
        rows = [torch.empty(p, dtype=dt, device="cuda") for _ in range(n)]
    for r in rows:
        tmp = torch.randn(p, generator=g, device="cuda") * wl.scale
        r.copy_(tmp)
        del tmp
    stream = torch.cuda.current_stream()
    c = args.call
    if c == "allreduce":
        step = lambda: ra.ra_allreduce_avg(rows, stream)
    elif c == "staged":
        ws = torch.empty(max(1, ra.ra_staged_workspace_bytes(n, p, 1 if bf16 else 0)), dtype=torch.uint8,
                         device="cuda")
        step = lambda: ra.ra_allreduce_avg_staged(rows, ws, stream)
    elif c == "sgd":
        w = torch.randn(p, generator=g, device="cuda")
        step = lambda: ra.ra_allreduce_sgd(rows, w, wl.sgd_lr or 0.1, stream)
    elif c == "buckets":
        plan = ra.ra_bucket_plan(tensors_within(wl.tensors or (p,), p), esz, wl.bucket_cap_bytes or 25 * 1024 * 1024)
        step = lambda: ra.ra_allreduce_avg_buckets(rows, plan, stream)
    elif c == "buckets_each":  # one call, and so one launch, per bucket
        plan = ra.ra_bucket_plan(tensors_within(wl.tensors or (p,), p), esz, wl.bucket_cap_bytes or 25 * 1024 * 1024)

        def step():
            for b in plan:
                ra.ra_allreduce_avg_buckets(rows, [b], stream)
    elif c == "reduce_scatter":
        step = lambda: ra.ra_reduce_scatter_avg(rows, None, stream)
    elif c == "all_gather":
        step = lambda: ra.ra_all_gather(rows, None, stream)
    elif c == "single_reducer":
        step = lambda: ra.ra_allreduce_avg_single_reducer(rows, stream)
    elif c == "bf16_wire":
        step = lambda: ra.ra_allreduce_avg_bf16_wire(rows, stream)
    else:  # host: the rows live in pinned host memory, the kernel works on them directly
        hrows = [torch.empty(p, dtype=rows[0].dtype).pin_memory() for _ in range(n)]
        for h, r in zip(hrows, rows):
            h.copy_(r)
        del rows
        step = lambda: ra.ra_allreduce_avg_host(hrows, None, ra.RA_HOST_DIRECT, stream)
    for _ in range(args.warmup):
        step()
    _, ms = timed_region(lambda k: step(), args.steps, None, _CudaEventTimer(stream))
    ms /= args.steps
    nbytes = call_bytes(c, n, p, esz)
    print(json.dumps({"profile_run": True, "workload": args.workload, "call": c, "layout": args.layout, "workers": n,
                      "elements_per_worker": p, "ms_per_step": ms, "algorithmic_bytes": nbytes,
                      "gbs": nbytes / (ms / 1e3) / 1e9}), flush=True)
    return 0


def run_host_link(args):
    """What the host link delivers, as the ceiling of the end-to-end number:
    N rows of P fp32 in pinned host memory (the bench workload's shape),
    moved by the copy engines (one cudaMemcpyAsync per row: host to device,
    device to host, and both at once on two streams) and by this library's
    kernels working on the host rows directly over NVLink-C2C (the
    reduce-scatter reads N*P and writes P elements, the all-gather reads P
    and writes (N-1)*P, the all-reduce reads and writes N*P).  One JSON line,
    GB/s of host-side bytes for each."""
    import ctypes

    import torch
    from gradient_ring_all_gb300 import build
    build.build()
    import gradient_ring_all_gb300 as ra
    import synth
    lib = ra.load()
    wl = synth.WORKLOADS[args.workload]
    n, p = (args.workers or wl.n), (args.elements or wl.p)
    esz = 2 if wl.dtype == "bf16" else 4
    dt = torch.bfloat16 if esz == 2 else torch.float32
    code = ra.RA_BF16 if esz == 2 else ra.RA_F32
    h = [torch.zeros(p, dtype=dt).pin_memory() for _ in range(n)]
    d = [torch.empty(p, dtype=dt, device="cuda") for _ in range(n)]
    s0 = torch.cuda.current_stream()
    s1 = torch.cuda.Stream()
    arr = (ctypes.c_void_p * n)(*[x.data_ptr() for x in h])  # pinned host memory is device-addressable
    st = ctypes.c_void_p(s0.cuda_stream)

    def h2d():
        for a, b in zip(d, h):
            a.copy_(b, non_blocking=True)

    def d2h():
        for a, b in zip(h, d):
            a.copy_(b, non_blocking=True)

    def both():
        # half the rows in, the other half out, on two streams at once
        half = n // 2
        s1.wait_stream(s0)  # only the work queued before this step
        for a, b in zip(d[:half], h[:half]):
            a.copy_(b, non_blocking=True)
        with torch.cuda.stream(s1):
            for a, b in zip(h[half:], d[half:]):
                a.copy_(b, non_blocking=True)
        s0.wait_stream(s1)

    def call(fn, what):
        def run():
            rc = fn()
            if rc != 0:
                raise RuntimeError("%s: %s" % (what, ra.ra_status_str(rc)))
        return run

    legs = [
        ("copy_h2d", h2d, n * p * esz),
        ("copy_d2h", d2h, n * p * esz),
        ("copy_h2d_and_d2h_concurrent", both, n * p * esz),
        ("kernel_reduce_scatter_on_host_rows", call(lambda: lib.ra_reduce_scatter_avg(arr, n, p, code, None, st),
                                                    "ra_reduce_scatter_avg"), (n + 1) * p * esz),
        ("kernel_all_gather_on_host_rows", call(lambda: lib.ra_all_gather(arr, n, p, code, None, st),
                                                "ra_all_gather"), n * p * esz),
        ("kernel_allreduce_on_host_rows", call(lambda: lib.ra_allreduce_avg(arr, n, p, code, st), "ra_allreduce_avg"),
         2 * n * p * esz),
    ]
    out = {"profile_run": True, "call": "host_link", "workload": args.workload, "workers": n,
           "elements_per_worker": p, "host_memory": "pinned (cudaHostAlloc through torch)"}
    steps = max(1, min(args.steps, 10))
    for name, fn, nbytes in legs:
        fn()
        _, ms = timed_region(lambda k: fn(), steps, None, _CudaEventTimer(s0))
        ms /= steps
        out[name] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms / 1e3) / 1e9}
    torch.cuda.synchronize()
    out["device_errors"] = ra.ra_status_str(ra.ra_check_device_errors())
    print(json.dumps(out), flush=True)
    return 0


def run_overlap(args):
    """Overlap of the bucketed all-reduce with a synthetic backward pass
    (Gibiansky, "Applying the Allreduce to Deep Learning").  The backward of
    the 24-layer Transformer is stood in for by bf16 tensor-core GEMMs, layer
    by layer from the output side, sized at 4 * tokens * params FLOPs per
    layer (weight and input gradients); as each layer's GEMMs are queued its
    tensors are marked ready on the reducer, whose bucket all-reduces run on
    their own stream.  Prints one JSON line with the four timings."""
    import torch
    from gradient_ring_all_gb300 import build
    build.build()
    import gradient_ring_all_gb300 as ra
    import synth
    wl = synth.WORKLOADS["transformer24_buckets_n4_f32"]
    n, p, numel = wl.n, wl.p, list(wl.tensors)
    rows = [torch.zeros(p, dtype=torch.float32, device="cuda") for _ in range(n)]
    tokens = args.tokens
    # GEMM unit: [tokens x 2048] @ [2048 x 8192] bf16
    a = torch.randn(tokens, 2048, device="cuda", dtype=torch.bfloat16)
    b = torch.randn(2048, 8192, device="cuda", dtype=torch.bfloat16)
    unit_flops = 2.0 * tokens * 2048 * 8192
    # layers: embed, 24 x 16 tensors, softmax -> groups of tensor indices
    groups = [[0]] + [list(range(1 + 16 * l, 17 + 16 * l)) for l in range(24)] + [[len(numel) - 1]]
    reps = [max(1, round(4.0 * tokens * sum(numel[t] for t in g) / unit_flops)) for g in groups]
    stream = torch.cuda.current_stream()
    red = ra.Reducer(rows, numel, wl.bucket_cap_bytes)

    def backward(mark):
        for g, r in zip(reversed(groups), reversed(reps)):
            for _ in range(r):
                torch.mm(a, b)
            if mark:
                for t in reversed(g):
                    red.mark_ready(t, stream)

    def t_of(fn, steps):
        fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    plan = red.buckets()
    steps = max(3, min(args.steps, 10))
    t_bwd = t_of(lambda: backward(False), steps)
    t_ar = t_of(lambda: ra.ra_allreduce_avg_buckets(rows, plan, stream), steps)
    t_seq = t_of(lambda: (backward(False), ra.ra_allreduce_avg_buckets(rows, plan, stream)), steps)
    t_ovl = t_of(lambda: (backward(True), red.finish(stream)), steps)
    red.close()
    line = {"experiment": "overlap of the bucketed all-reduce with a synthetic backward",
            "workload": "transformer24_buckets_n4_f32", "buckets": len(plan), "tokens": tokens,
            "backward_tflop": sum(reps) * unit_flops / 1e12,
            "ms": {"backward": t_bwd, "allreduce": t_ar, "sequential": t_seq, "overlapped": t_ovl},
            "exposed_allreduce_ms": t_ovl - t_bwd,
            "hidden_fraction": (t_seq - t_ovl) / t_ar if t_ar > 0 else None}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--elements", type=int, default=0,
                    help="profiling only: elements per worker instead of the workload's 300M")
    ap.add_argument("--legs", choices=["all", "device"], default="all",
                    help="profiling only: 'device' skips the end-to-end and CPU legs")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="profiling only (with --call): the synthetic workload to run")
    ap.add_argument("--call", choices=CALLS, default=None,
                    help="profiling only: time one entry point on --workload, device loop only")
    ap.add_argument("--workers", type=int, default=0,
                    help="--call: worker count instead of the workload's (with --elements for the length)")
    ap.add_argument("--layout", choices=["separate", "strided"], default="separate",
                    help="--call: one allocation per worker, or rows back to back with stride P+1 elements")
    ap.add_argument("--per-config", dest="per_config", action=argparse.BooleanOptionalAction, default=True,
                    help="after the headline (N=1, full size): also measure and verify every other configuration")
    ap.add_argument("--config-steps", type=int, default=20, help="timed calls per configuration in per_config")
    ap.add_argument("--overlap", action="store_true",
                    help="experiment: bucketed all-reduce overlapped with a synthetic backward")
    ap.add_argument("--tokens", type=int, default=8192, help="--overlap: tokens per backward step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.overlap:
        return run_overlap(args)
    if args.call == "host_link":
        return run_host_link(args)
    if args.call:
        return run_profile_call(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
