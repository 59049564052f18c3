"""bench.py's JSON line on the GPU: a reduced run (20M elements per worker)
must print one line with every key of the benchmark contract, consistent
values, the roofline and CPU-baseline objects, and the check of what it
timed (bit-exact first call, clean device error word).  The host-link leg
prints its copy-engine and kernel figures."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _line(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def test_bench_line_has_the_contract_keys():
    d = _line("--elements", "20000000", "--steps", "5", "--warmup", "3")
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "cpu_baseline", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # value is the algorithmic bytes over the measured step time
    cfg = d["config"]
    assert cfg["workload"] == "speech300m_n8_f32" and cfg["elements_per_worker"] == 20_000_000
    assert abs(d["value"] - cfg["bytes_per_step"] / (d["ms_per_step"] / 1e3) / 1e9) < 1e-6 * d["value"]
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 8 * 20_000_000 * 4
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0 and c["sample"]
    assert d["gpu_launches"] == 5
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["bit_exact"] is True
    v = d["verification"]
    assert v["first_mismatch"] is None and v["device_errors_after_timed_region"] == "RA_OK"
    m = d["max_rel_err_vs_f64"]
    assert 0 <= m["norm"] <= 1e-5 and 0 <= m["max_elementwise"] <= 1e-5
    assert "per_config" not in d  # reduced runs measure the headline only


def test_host_link_leg():
    d = _line("--call", "host_link", "--elements", "4000000", "--steps", "2", "--warmup", "3")
    for k in ("copy_h2d", "copy_d2h", "copy_h2d_and_d2h_concurrent", "kernel_reduce_scatter_on_host_rows",
              "kernel_all_gather_on_host_rows", "kernel_allreduce_on_host_rows"):
        assert d[k]["gbs"] > 0 and d[k]["bytes"] > 0, k
    assert d["device_errors"] == "RA_OK"
