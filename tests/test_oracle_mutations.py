"""Mutation check of the oracle's pins: each case plants one plausible
mistake in a copy of ``oracle/ring_oracle.c`` -- a wrong chunk offset, a
schedule index off by one or in the wrong direction, a dropped iteration,
multiplication by 1/N instead of division, the wrong owner of a chunk, a
rounding that is not ties-to-even, a wrong bucket rule, a wrong traffic
count -- and runs ``tests/test_oracle_pins.py`` against that copy.  Every
mistake must make at least one pin fail; an unmutated copy must pass.

Mutants that cannot change a result are not listed: IEEE addition is
commutative, so swapping the operands of an add is not a mistake; and in the
bf16-wire mean the dividend is a bf16 value, for which the bf16-rounded
quotient x / N equals the bf16-rounded x * (1/N) for every normal x and every
N up to 64 (checked exhaustively in binary32), so that replacement cannot
show either.

The copies live under tests/.scratch (git-ignored) and are removed
afterwards.  CPU only.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SCRATCH = os.path.join(ROOT, "tests", ".scratch", "oracle_mutants")

# (name, exact text in ring_oracle.c, replacement); each text occurs once
MUTANTS = [
    ("chunk offset ignores the extra elements",
     "int64_t b = (int64_t)c * q + (c < r ? c : r);", "int64_t b = (int64_t)c * q + (c < r ? c : 0);"),
    ("extra element on one chunk too many",
     "*end = b + q + (c < r ? 1 : 0);", "*end = b + q + (c <= r ? 1 : 0);"),
    ("scatter-reduce sends in the wrong direction",
     "int oracle_scatter_send_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n - t, n_workers); }",
     "int oracle_scatter_send_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n + t, n_workers); }"),
    ("scatter-reduce receives the wrong chunk",
     "int oracle_scatter_recv_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n - 1 - t, n_workers); }",
     "int oracle_scatter_recv_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n - t, n_workers); }"),
    ("all-gather sends the wrong chunk",
     "int oracle_gather_send_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n + 1 - t, n_workers); }",
     "int oracle_gather_send_chunk(int n_workers, int n, int t) { return mod_n((int64_t)n - t, n_workers); }"),
    ("one scatter-reduce iteration dropped",
     "    for (int t = 0; t < n_scatter; ++t) {", "    for (int t = 1; t < n_scatter; ++t) {"),
    ("average by multiplying with 1/N",
     "float avg = rows[n][i] / fn;", "float avg = rows[n][i] * (1.0f / fn);"),
    ("the wrong worker divides",
     "            int c = mod_n((int64_t)n + 1, N);\n", "            int c = mod_n((int64_t)n, N);\n"),
    ("bf16 ties rounded away from zero",
     "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))", "if (lower >= 0x8000u)"),
    ("bf16 truncated",
     "        upper += 1u;", "        upper += 0u;"),
    ("SGD step added instead of subtracted",
     "        float step = lr * avg[i];\n        w[i] = w[i] - step;",
     "        float step = lr * avg[i];\n        w[i] = w[i] + step;"),
    ("bf16-mean SGD step added instead of subtracted",
     "        float step = lr * bf16_to_f32(avg[i]);\n        w[i] = w[i] - step;",
     "        float step = lr * bf16_to_f32(avg[i]);\n        w[i] = w[i] + step;"),
    ("bf16-mean SGD as one fused multiply-add",
     "        float step = lr * bf16_to_f32(avg[i]);\n        w[i] = w[i] - step;",
     "        w[i] = __builtin_fmaf(-lr, bf16_to_f32(avg[i]), w[i]);"),
    ("bf16-mean SGD step rounded to bf16",
     "        float step = lr * bf16_to_f32(avg[i]);",
     "        float step = bf16_to_f32(oracle_f32_to_bf16(lr * bf16_to_f32(avg[i])));"),
    ("bucket closes only above the cap",
     "if ((end - start) * elem_bytes >= cap_bytes) {", "if ((end - start) * elem_bytes > cap_bytes) {"),
    ("point evaluation folds from the wrong worker",
     "int receiver = mod_n((int64_t)c + 1 + t, N);", "int receiver = mod_n((int64_t)c + t, N);"),
    ("range evaluation folds from the wrong worker",
     "const float *recv = rows[mod_n((int64_t)c + 1 + t, N)];", "const float *recv = rows[mod_n((int64_t)c + t, N)];"),
    ("bf16 range evaluation skips a worker",
     "const uint16_t *recv = rows[mod_n((int64_t)c + 1 + t, N)];",
     "const uint16_t *recv = rows[mod_n((int64_t)c + 2 + t, N)];"),
    ("range evaluation multiplies with 1/N",
     "out[i - begin] = out[i - begin] / fn;", "out[i - begin] = out[i - begin] * (1.0f / fn);"),
    ("traffic credited to the sender",
     "received[mod_n((int64_t)n + 1, N)] += e - b;", "received[n] += e - b;"),
    ("all-gather copies into the wrong chunk",
     "oracle_chunk_range(p, N, oracle_gather_recv_chunk(N, m, t), &b, &e);\n            memcpy(",
     "oracle_chunk_range(p, N, oracle_gather_send_chunk(N, m, t), &b, &e);\n            memcpy("),
    ("single reducer adds the workers in reverse order",
     "    for (int m = 1; m < N; ++m) {\n        for (int64_t i = 0; i < p; ++i)\n            rows[0][i] = rows[0][i] + rows[m][i];",
     "    for (int m = N - 1; m >= 1; --m) {\n        for (int64_t i = 0; i < p; ++i)\n            rows[0][i] = rows[0][i] + rows[m][i];"),
    ("single reducer mean by multiplying with 1/N",
     "        rows[0][i] = rows[0][i] / fn;", "        rows[0][i] = rows[0][i] * (1.0f / fn);"),
    ("binary64 mean over N - 1",
     "out[i] = s / (double)n_workers;", "out[i] = s / (double)(n_workers - 1);"),
]


def _copy_tree(dst, src_c):
    for d in ("oracle", "synth"):
        os.makedirs(os.path.join(dst, d))
        for f in os.listdir(os.path.join(ROOT, d)):
            if f.endswith((".py", ".c", ".h")):
                shutil.copy(os.path.join(ROOT, d, f), os.path.join(dst, d, f))
    with open(os.path.join(dst, "oracle", "ring_oracle.c"), "w") as f:
        f.write(src_c)
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "exact_ieee.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _pins_pass(dst) -> bool:
    env = dict(os.environ, PYTHONPATH=dst, PYTHONDONTWRITEBYTECODE="1")
    # the copy must build: a mutant that does not compile would fail the pins
    # for the wrong reason
    b = subprocess.run([sys.executable, "-c", "import oracle, synth; oracle.build(); synth.build(); "
                        "assert oracle.__file__.startswith(%r)" % dst],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=300)
    assert b.returncode == 0, "the copy in %s did not build: %s" % (dst, b.stderr[-1000:])
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(dst, "tests", "test_oracle_pins.py")],
                       cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode == 0


def test_every_planted_mistake_fails_a_pin():
    with open(os.path.join(ROOT, "oracle", "ring_oracle.c")) as f:
        src = f.read()
    shutil.rmtree(SCRATCH, ignore_errors=True)
    jobs = [("control", src)]
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, "mutation site not unique: %s" % name
        jobs.append((name, src.replace(old, new)))
    dirs = []
    for k, (_, text) in enumerate(jobs):
        d = os.path.join(SCRATCH, "m%02d" % k)
        _copy_tree(d, text)
        dirs.append(d)
    try:
        with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
            passed = list(ex.map(_pins_pass, dirs))
    finally:
        shutil.rmtree(SCRATCH, ignore_errors=True)
    assert passed[0], "the unmutated oracle copy must pass its pins"
    survivors = [jobs[k][0] for k in range(1, len(jobs)) if passed[k]]
    assert not survivors, "planted mistakes no pin catches: %s" % survivors
