"""CPU oracle for the ring all-reduce -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU leg of
``bench.py`` (its timed CPU baseline, and its check of the GPU's result
against host copies of the same inputs) may import this package.  The
product library never imports or links it, and it shares no code with the
CUDA path.

This module is a thin ctypes wrapper around ``ring_oracle.c`` (a plain,
single-threaded C simulation of the ring's scatter-reduce, average and
all-gather steps; see that file's header for the pages it follows and the
readings it takes).  Arrays are numpy arrays on the host.

``build()`` compiles the C file with ``-ffp-contract=off`` so that no fused
multiply-add enters the binary32 arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ring_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compile ring_oracle.c into liboracle.so (in this directory)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    pi64 = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_chunk_range.argtypes = [i64, i32, i32, pi64, pi64]
    lib.oracle_chunk_range.restype = None
    for nm in ("oracle_scatter_send_chunk", "oracle_scatter_recv_chunk",
               "oracle_gather_send_chunk", "oracle_gather_recv_chunk"):
        getattr(lib, nm).argtypes = [i32, i32, i32]
        getattr(lib, nm).restype = i32
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_ring_run_f32.argtypes = [vp, i32, i64, i32, i32, i32, i32, vp, vp]
    lib.oracle_ring_run_f32.restype = i32
    lib.oracle_ring_allreduce_avg_f32.argtypes = [vp, i32, i64, vp, vp]
    lib.oracle_ring_allreduce_avg_f32.restype = i32
    lib.oracle_ring_allreduce_avg_bf16.argtypes = [vp, i32, i64, vp, vp]
    lib.oracle_ring_allreduce_avg_bf16.restype = i32
    lib.oracle_sgd_update_f32.argtypes = [vp, vp, i64, ctypes.c_float]
    lib.oracle_sgd_update_f32.restype = None
    lib.oracle_sgd_update_bf16avg.argtypes = [vp, vp, i64, ctypes.c_float]
    lib.oracle_sgd_update_bf16avg.restype = None
    lib.oracle_ring_avg_point_f32.argtypes = [vp, i32, i64, i64]
    lib.oracle_ring_avg_point_f32.restype = ctypes.c_float
    lib.oracle_ring_avg_point_bf16.argtypes = [vp, i32, i64, i64]
    lib.oracle_ring_avg_point_bf16.restype = ctypes.c_uint16
    for nm in ("oracle_ring_avg_range_f32", "oracle_ring_avg_range_bf16"):
        getattr(lib, nm).argtypes = [vp, i32, i64, i64, i64, vp]
        getattr(lib, nm).restype = i32
    lib.oracle_mean_f64.argtypes = [vp, i32, i64, vp]
    lib.oracle_mean_f64.restype = None
    lib.oracle_bucket_plan.argtypes = [vp, i32, i64, i64, vp, vp, i32]
    lib.oracle_bucket_plan.restype = i32
    lib.oracle_reduce_scatter_avg_bf16.argtypes = [vp, i32, i64]
    lib.oracle_reduce_scatter_avg_bf16.restype = i32
    lib.oracle_all_gather.argtypes = [vp, i32, i64, i32]
    lib.oracle_all_gather.restype = i32
    lib.oracle_ring_allreduce_avg_bf16_wire.argtypes = [vp, i32, i64]
    lib.oracle_ring_allreduce_avg_bf16_wire.restype = i32
    for nm in ("oracle_single_reducer_avg_f32", "oracle_single_reducer_avg_bf16"):
        getattr(lib, nm).argtypes = [vp, i32, i64, vp, vp]
        getattr(lib, nm).restype = i32
    lib.oracle_ring_traffic.argtypes = [i32, i64, vp, vp]
    lib.oracle_ring_traffic.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _row_ptrs(rows):
    arr = (ctypes.c_void_p * len(rows))(*[_ptr(r) for r in rows])
    return arr


def _check_rows(rows, dtype):
    if len(rows) < 1:
        raise ValueError("need at least one worker row")
    p = rows[0].shape[0]
    for r in rows:
        if r.dtype != dtype or r.ndim != 1 or r.shape[0] != p or not r.flags.c_contiguous:
            raise ValueError("rows must be contiguous 1-D %s arrays of one length" % dtype)
    return p


# --------------------------------------------------------------------------
# schedule and chunks


def chunk_range(p: int, n: int, c: int) -> tuple[int, int]:
    lib = _load()
    b, e = ctypes.c_int64(), ctypes.c_int64()
    lib.oracle_chunk_range(p, n, c, ctypes.byref(b), ctypes.byref(e))
    return b.value, e.value


def scatter_send_chunk(n_workers: int, n: int, t: int) -> int:
    return _load().oracle_scatter_send_chunk(n_workers, n, t)


def scatter_recv_chunk(n_workers: int, n: int, t: int) -> int:
    return _load().oracle_scatter_recv_chunk(n_workers, n, t)


def gather_send_chunk(n_workers: int, n: int, t: int) -> int:
    return _load().oracle_gather_send_chunk(n_workers, n, t)


def gather_recv_chunk(n_workers: int, n: int, t: int) -> int:
    return _load().oracle_gather_recv_chunk(n_workers, n, t)


def f32_to_bf16_bits(x: float) -> int:
    return int(_load().oracle_f32_to_bf16(float(np.float32(x))))


# --------------------------------------------------------------------------
# the ring


def ring_run_f32(rows, n_scatter, do_avg, n_gather, bf16_out=False):
    """Run part of the ring in place on binary32 rows; returns (sent, received)."""
    p = _check_rows(rows, np.float32)
    n = len(rows)
    sent = np.zeros(n, np.int64)
    recv = np.zeros(n, np.int64)
    rc = _load().oracle_ring_run_f32(_row_ptrs(rows), n, p, n_scatter, int(do_avg), int(bf16_out),
                                     n_gather, _ptr(sent), _ptr(recv))
    if rc != 0:
        raise ValueError("oracle_ring_run_f32 rejected its arguments")
    return sent, recv


def ring_allreduce_avg_f32(rows):
    """Full ring all-reduce-average of binary32 rows, in place; returns (sent, received)."""
    p = _check_rows(rows, np.float32)
    n = len(rows)
    sent = np.zeros(n, np.int64)
    recv = np.zeros(n, np.int64)
    if _load().oracle_ring_allreduce_avg_f32(_row_ptrs(rows), n, p, _ptr(sent), _ptr(recv)) != 0:
        raise ValueError("oracle_ring_allreduce_avg_f32 rejected its arguments")
    return sent, recv


def ring_allreduce_avg_bf16(rows):
    """Full ring all-reduce-average of bf16 rows (uint16 bit patterns), in place."""
    p = _check_rows(rows, np.uint16)
    n = len(rows)
    sent = np.zeros(n, np.int64)
    recv = np.zeros(n, np.int64)
    if _load().oracle_ring_allreduce_avg_bf16(_row_ptrs(rows), n, p, _ptr(sent), _ptr(recv)) != 0:
        raise ValueError("oracle_ring_allreduce_avg_bf16 rejected its arguments")
    return sent, recv


def sgd_update_f32(w, avg, lr):
    """w <- w - lr*avg in place (two roundings); avg binary32 or bf16 bits."""
    if w.dtype != np.float32 or not w.flags.c_contiguous or avg.shape[0] != w.shape[0]:
        raise ValueError("w must be contiguous float32 of avg's length")
    if avg.dtype == np.float32:
        _load().oracle_sgd_update_f32(_ptr(w), _ptr(avg), w.shape[0], float(lr))
    elif avg.dtype == np.uint16:
        _load().oracle_sgd_update_bf16avg(_ptr(w), _ptr(avg), w.shape[0], float(lr))
    else:
        raise ValueError("avg must be float32 or bf16 bits")


def ring_avg_point_f32(vals, p: int, i: int) -> np.float32:
    """Ring result at element i of a p-element ring, from the N inputs at i."""
    v = np.ascontiguousarray(vals, dtype=np.float32)
    return np.float32(_load().oracle_ring_avg_point_f32(_ptr(v), v.shape[0], p, i))


def ring_avg_point_bf16(vals, p: int, i: int) -> int:
    """bf16 ring result (bit pattern) at element i, from the N bf16 inputs at i."""
    v = np.ascontiguousarray(vals, dtype=np.uint16)
    return int(_load().oracle_ring_avg_point_bf16(_ptr(v), v.shape[0], p, i))


def ring_avg_range(rows, p: int, begin: int, out=None):
    """Ring results at elements [begin, begin + len) of a p-element ring.

    rows: the N workers' input slices at those elements (contiguous 1-D
    float32, or uint16 bf16 bits), all of one length; out (optional): where
    to write them.  Returns out.  Each call runs on the calling thread and
    releases the interpreter lock, so slices can be evaluated in parallel."""
    dt = rows[0].dtype
    if dt not in (np.float32, np.uint16):
        raise ValueError("rows must be float32 or bf16 bits")
    cnt = _check_rows(rows, dt)
    if out is None:
        out = np.empty(cnt, dt)
    if out.dtype != dt or out.shape != (cnt,) or not out.flags.c_contiguous:
        raise ValueError("out must be a contiguous array of the rows' dtype and length")
    fn = _load().oracle_ring_avg_range_f32 if dt == np.float32 else _load().oracle_ring_avg_range_bf16
    if fn(_row_ptrs(rows), len(rows), p, begin, begin + cnt, _ptr(out)) != 0:
        raise ValueError("ring_avg_range rejected its arguments")
    return out


def mean_f64(rows):
    p = _check_rows(rows, np.float32)
    out = np.empty(p, np.float64)
    _load().oracle_mean_f64(_row_ptrs(rows), len(rows), p, _ptr(out))
    return out


def ring_traffic(n: int, p: int):
    """Per-worker (sent, received) element counts of one full ring all-reduce."""
    sent = np.zeros(n, np.int64)
    recv = np.zeros(n, np.int64)
    _load().oracle_ring_traffic(n, p, _ptr(sent), _ptr(recv))
    return sent, recv


def bucket_plan(numel, elem_bytes: int, cap_bytes: int):
    """Reverse-order bucket plan; returns a list of (offset, count)."""
    nm = np.ascontiguousarray(numel, dtype=np.int64)
    mx = max(1, nm.shape[0] + 1)
    off = np.zeros(mx, np.int64)
    cnt = np.zeros(mx, np.int64)
    nb = _load().oracle_bucket_plan(_ptr(nm), nm.shape[0], elem_bytes, cap_bytes, _ptr(off), _ptr(cnt), mx)
    if nb < 0:
        raise ValueError("oracle_bucket_plan rejected its arguments")
    return [(int(off[k]), int(cnt[k])) for k in range(nb)]


def ring_allreduce_avg_buckets_f32(rows, buckets):
    """Each bucket (offset, count) of the rows is its own ring."""
    for off, cnt in buckets:
        ring_allreduce_avg_f32([r[off:off + cnt] for r in rows])


# --------------------------------------------------------------------------
# the two phases on their own


def owned_chunk(n_workers: int, w: int) -> int:
    """After the scatter-reduce worker w holds the complete chunk w+1."""
    return (w + 1) % n_workers


def reduce_scatter_avg(rows):
    """Scatter-reduce + owner's division in place; returns {worker: (begin,
    end)} of the chunk each worker now owns (its only defined result)."""
    n = len(rows)
    if rows[0].dtype == np.float32:
        ring_run_f32(rows, n - 1, True, 0)
    elif rows[0].dtype == np.uint16:
        p = _check_rows(rows, np.uint16)
        if _load().oracle_reduce_scatter_avg_bf16(_row_ptrs(rows), n, p) != 0:
            raise ValueError("oracle_reduce_scatter_avg_bf16 rejected its arguments")
    else:
        raise ValueError("rows must be float32 or bf16 bits")
    p = rows[0].shape[0]
    return {w: chunk_range(p, n, owned_chunk(n, w)) for w in range(n)}


def all_gather(rows):
    """Literal all-gather in place (any dtype): worker (c-1) mod N's chunk c
    reaches every worker."""
    p = rows[0].shape[0]
    for r in rows:
        if r.dtype != rows[0].dtype or r.shape[0] != p or not r.flags.c_contiguous:
            raise ValueError("rows must be contiguous arrays of one dtype and length")
    if _load().oracle_all_gather(_row_ptrs(rows), len(rows), p, rows[0].itemsize) != 0:
        raise ValueError("oracle_all_gather rejected its arguments")


# --------------------------------------------------------------------------
# variants: bf16 partials on the wire, and the single reducer


def ring_allreduce_avg_bf16_wire(rows):
    """The ring over bf16 arrays: every partial sum rounded to bf16 (in place)."""
    p = _check_rows(rows, np.uint16)
    if _load().oracle_ring_allreduce_avg_bf16_wire(_row_ptrs(rows), len(rows), p) != 0:
        raise ValueError("oracle_ring_allreduce_avg_bf16_wire rejected its arguments")


def single_reducer_avg(rows):
    """Worker 0 sums the others' arrays in worker order, divides, broadcasts
    (in place); returns per-worker (sent, received) element counts."""
    n = len(rows)
    sent = np.zeros(n, np.int64)
    recv = np.zeros(n, np.int64)
    if rows[0].dtype == np.float32:
        p = _check_rows(rows, np.float32)
        rc = _load().oracle_single_reducer_avg_f32(_row_ptrs(rows), n, p, _ptr(sent), _ptr(recv))
    else:
        p = _check_rows(rows, np.uint16)
        rc = _load().oracle_single_reducer_avg_bf16(_row_ptrs(rows), n, p, _ptr(sent), _ptr(recv))
    if rc != 0:
        raise ValueError("oracle single reducer rejected its arguments")
    return sent, recv
