"""The Python binding: no CPU fallback -- without the shared library every
call fails loudly; argument checks happen before the C call."""
from __future__ import annotations

import importlib

import pytest


def test_missing_library_raises(monkeypatch):
    import gradient_ring_all_gb300 as ra
    monkeypatch.setattr(ra, "_lib", None)
    monkeypatch.setattr(ra, "_LIB_PATH", "/nonexistent/libgradient_ring_all.so")
    with pytest.raises(RuntimeError, match="not built"):
        ra.load()
    with pytest.raises(RuntimeError, match="not built"):
        ra.ra_chunk_range(10, 2, 0)
    monkeypatch.undo()
    importlib.reload(ra)


def test_binding_checks_tensors_before_calling():
    torch = pytest.importorskip("torch")
    import gradient_ring_all_gb300 as ra
    with pytest.raises(ValueError):
        ra.ra_allreduce_avg([])
    with pytest.raises(ValueError):  # CPU tensors are not device buffers
        ra.ra_allreduce_avg([torch.zeros(4), torch.zeros(4)])
    with pytest.raises(TypeError):
        ra.ra_allreduce_avg([torch.zeros(4, dtype=torch.float64)])
