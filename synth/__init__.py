"""Seeded synthetic inputs for the ring all-reduce (tests, oracle side, bench).

This module only draws random numbers and lists tensor shapes; it contains
none of the all-reduce's arithmetic.  Values depend on (seed, stream, index)
only (counter-based SplitMix64 + Box-Muller, see ``synth.c``), so any element
can be regenerated alone -- which is how the tests check sampled outputs of
runs too large for the oracle to simulate whole.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .shapes import resnet18_shapes, transformer_shapes  # noqa: F401
from .workloads import WORKLOADS, Workload  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"],
                       check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, d, vp, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        for nm in ("synth_normal_f32", "synth_student_t3_bf16", "synth_student_t3_f32"):
            getattr(lib, nm).argtypes = [u64, u64, d, i64, i64, vp, i32]
            getattr(lib, nm).restype = None
        for nm in ("synth_normal_f32_at", "synth_student_t3_bf16_at"):
            getattr(lib, nm).argtypes = [u64, u64, d, vp, i64, vp]
            getattr(lib, nm).restype = None
        lib.synth_raw_u64.argtypes = [u64, u64, i64, i64, vp]
        lib.synth_raw_u64.restype = None
        lib.synth_splitmix64.argtypes = [u64, i64, i64, vp]
        lib.synth_splitmix64.restype = None
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def fill_normal_f32(ptr: int, seed: int, stream: int, sigma: float, start: int, count: int, threads=None):
    """Write float(sigma*Z) for indices [start, start+count) to host memory at ptr."""
    _load().synth_normal_f32(seed, stream, sigma, start, count, ptr, threads or default_threads())


def fill_student_t3_bf16(ptr: int, seed: int, stream: int, scale: float, start: int, count: int, threads=None):
    """Write bf16_rne(float(scale*T3)) bit patterns (uint16) to host memory at ptr."""
    _load().synth_student_t3_bf16(seed, stream, scale, start, count, ptr, threads or default_threads())


def normal_f32(seed: int, stream: int, sigma: float, start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.float32)
    fill_normal_f32(out.ctypes.data, seed, stream, sigma, start, count)
    return out


def student_t3_bf16(seed: int, stream: int, scale: float, start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint16)
    fill_student_t3_bf16(out.ctypes.data, seed, stream, scale, start, count)
    return out


def student_t3_f32(seed: int, stream: int, scale: float, start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.float32)
    _load().synth_student_t3_f32(seed, stream, scale, start, count, out.ctypes.data, default_threads())
    return out


def normal_f32_at(seed: int, stream: int, sigma: float, idx) -> np.ndarray:
    ix = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(ix.shape[0], np.float32)
    _load().synth_normal_f32_at(seed, stream, sigma, ix.ctypes.data, ix.shape[0], out.ctypes.data)
    return out


def student_t3_bf16_at(seed: int, stream: int, scale: float, idx) -> np.ndarray:
    ix = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.empty(ix.shape[0], np.uint16)
    _load().synth_student_t3_bf16_at(seed, stream, scale, ix.ctypes.data, ix.shape[0], out.ctypes.data)
    return out


def raw_u64(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint64)
    _load().synth_raw_u64(seed, stream, start, count, out.ctypes.data)
    return out


def splitmix64(key: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, np.uint64)
    _load().synth_splitmix64(key, start, count, out.ctypes.data)
    return out
