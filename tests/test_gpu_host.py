"""ra_allreduce_avg_host: gradients in host memory, direct (the kernel on the
host arrays over the coherent link) and staged (copies through device
buffers), against the CPU oracle bit for bit."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import gradient_ring_all_gb300 as ra
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from gradient_ring_all_gb300 import build
    build.build()
    ra.load()
    torch.cuda.init()


def _pageable_access() -> bool:
    return bool(torch.cuda.get_device_properties(0).major >= 9 and _attr(88))


def _attr(a: int) -> int:
    import os
    for c in ("/usr/local/cuda/lib64/libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
        if os.path.exists(c):
            lib = ctypes.CDLL(c)
            v = ctypes.c_int(0)
            lib.cudaDeviceGetAttribute(ctypes.byref(v), a, torch.cuda.current_device())
            return v.value
    return 0


def _host_rows(n, p, dtype, seed, pinned, pad=0):
    rows = []
    for k in range(n):
        if dtype == "f32":
            a = synth.normal_f32(seed, k, 1.0, 0, p)
            base = torch.empty(p + 8, dtype=torch.float32)
            src = torch.from_numpy(a)
        else:
            a = synth.student_t3_bf16(seed, k, 1e-3, 0, p)
            base = torch.empty(p + 8, dtype=torch.bfloat16)
            src = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
        if pinned:
            base = base.pin_memory()
        t = base[pad:pad + p]
        t.copy_(src)
        rows.append(t)
    return rows


def _want(rows, dtype):
    if dtype == "f32":
        g = [r.numpy().copy() for r in rows]
        oracle.ring_allreduce_avg_f32(g)
    else:
        g = [r.view(torch.int16).numpy().view(np.uint16).copy() for r in rows]
        oracle.ring_allreduce_avg_bf16(g)
    return g[0]


def _got(t, dtype):
    return t.numpy() if dtype == "f32" else t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("mode", [ra.RA_HOST_AUTO, ra.RA_HOST_DIRECT, ra.RA_HOST_STAGED])
@pytest.mark.parametrize("n,p,pad", [(4, 1_048_579, 0), (8, 70_001, 1), (3, 5, 0)])
def test_host_path_matches_oracle(dtype, pinned, mode, n, p, pad):
    if mode == ra.RA_HOST_DIRECT and not pinned and not _pageable_access():
        pytest.skip("device cannot address pageable host memory")
    rows = _host_rows(n, p, dtype, seed=31 + n, pinned=pinned, pad=pad)
    want = _want(rows, dtype)
    dev = None
    if mode != ra.RA_HOST_DIRECT:
        dev = [torch.empty(p, dtype=rows[0].dtype, device="cuda") for _ in range(n)]
    ra.ra_allreduce_avg_host(rows, dev, mode)
    torch.cuda.synchronize()
    for r in rows:
        np.testing.assert_array_equal(_got(r, dtype), want)


def test_staged_without_device_buffers_is_unsupported():
    rows = _host_rows(2, 100, "f32", seed=1, pinned=True)
    with pytest.raises(ra.RaError) as e:
        ra.ra_allreduce_avg_host(rows, None, ra.RA_HOST_STAGED)
    assert e.value.status == 2  # RA_ERR_UNSUPPORTED


def test_bad_mode_is_rejected():
    rows = _host_rows(2, 100, "f32", seed=1, pinned=True)
    with pytest.raises(ra.RaError) as e:
        ra.ra_allreduce_avg_host(rows, None, 7)
    assert e.value.status == 1  # RA_ERR_INVALID_ARG
