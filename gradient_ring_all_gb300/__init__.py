"""Python binding of the GB300 ring all-reduce library (C ABI in
``include/ring_allreduce.h``).

The functions carry the C names and only marshal arguments: every step of
the all-reduce runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams.  Tensors must be contiguous CUDA tensors of one dtype
(float32 or bfloat16) and one length; the current torch stream is used
unless ``stream`` (a cudaStream_t as int, or a torch.cuda.Stream) is given.

There is no CPU fallback: if the shared library is missing this module
raises on first use.

With GRADIENT_RING_ALL_CHECKED=1 in the environment the bounds-checked build
(libgradient_ring_all_checked.so, ``build.build(checked=True)``) is loaded
instead: its kernels verify every global range they touch and report a
violation as RA_ERR_BOUNDS through ra_check_device_errors.  The tests use it.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "RA_F32", "RA_BF16", "RA_MAX_N", "RaError", "library_path", "load",
    "ra_allreduce_avg", "ra_allreduce_sgd", "ra_allreduce_avg_staged", "ra_staged_workspace_bytes",
    "ra_bucket_plan", "ra_allreduce_avg_buckets", "ra_allreduce_avg_host", "ra_allreduce_avg_staged_static",
    "RA_STAGED_STATIC_MAX_P", "RA_HOST_AUTO", "RA_HOST_DIRECT", "RA_HOST_STAGED", "ra_reduce_scatter_avg",
    "ra_all_gather", "ra_allreduce_avg_bf16_wire", "ra_allreduce_avg_single_reducer", "Reducer", "ra_check_device_errors", "ra_selftest_wait_timeout", "ra_selftest_bounds_check", "ra_chunk_range", "ra_status_str",
    "ra_last_cuda_error", "RA_OK", "RA_ERR_TIMEOUT", "RA_ERR_BOUNDS", "CHECKED",
]

RA_F32 = 0
RA_BF16 = 1
RA_MAX_N = 64
RA_STAGED_STATIC_MAX_P = 4194304
RA_HOST_AUTO, RA_HOST_DIRECT, RA_HOST_STAGED = 0, 1, 2
RA_OK, RA_ERR_TIMEOUT, RA_ERR_BOUNDS = 0, 5, 6

_HERE = os.path.dirname(os.path.abspath(__file__))
CHECKED = os.environ.get("GRADIENT_RING_ALL_CHECKED") == "1"
_LIB_PATH = os.path.join(_HERE, "lib", "libgradient_ring_all_checked.so" if CHECKED else "libgradient_ring_all.so")
_lib = None


class RaError(RuntimeError):
    def __init__(self, status: int, what: str):
        lib = load()
        name = lib.ra_status_str(status).decode()
        msg = "%s failed: %s" % (what, name)
        if name == "RA_ERR_CUDA":
            msg += " (cudaError %d)" % lib.ra_last_cuda_error()
        super().__init__(msg)
        self.status = status


class _Bucket(ctypes.Structure):
    _fields_ = [("offset", ctypes.c_int64), ("count", ctypes.c_int64)]


class _Traffic(ctypes.Structure):
    _fields_ = [("sent", ctypes.c_int64), ("received", ctypes.c_int64)]


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libgradient_ring_all.so (build it with gradient_ring_all_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError("%s is not built; run `python -m gradient_ring_all_gb300.build%s` first"
                           % (_LIB_PATH, " --checked" if CHECKED else ""))
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    pvp = ctypes.POINTER(ctypes.c_void_p)
    lib.ra_allreduce_avg.argtypes = [pvp, i32, i64, i32, vp]
    lib.ra_allreduce_sgd.argtypes = [pvp, i32, i64, i32, vp, f32, vp]
    lib.ra_staged_workspace_bytes.argtypes = [i32, i64, i32]
    lib.ra_staged_workspace_bytes.restype = ctypes.c_size_t
    lib.ra_allreduce_avg_staged.argtypes = [pvp, i32, i64, i32, vp, ctypes.c_size_t, ctypes.POINTER(_Traffic), vp]
    lib.ra_bucket_plan.argtypes = [ctypes.POINTER(ctypes.c_int64), i32, i32, i64, ctypes.POINTER(_Bucket), i32,
                                   ctypes.POINTER(i32)]
    lib.ra_allreduce_avg_buckets.argtypes = [pvp, i32, i32, ctypes.POINTER(_Bucket), i32, vp]
    lib.ra_allreduce_avg_host.argtypes = [pvp, pvp, i32, i64, i32, i32, vp]
    lib.ra_allreduce_avg_staged_static.argtypes = [pvp, i32, i64, i32, ctypes.POINTER(_Traffic), vp]
    lib.ra_reduce_scatter_avg.argtypes = [pvp, i32, i64, i32, pvp, vp]
    lib.ra_all_gather.argtypes = [pvp, i32, i64, i32, pvp, vp]
    lib.ra_allreduce_avg_bf16_wire.argtypes = [pvp, i32, i64, vp]
    lib.ra_allreduce_avg_single_reducer.argtypes = [pvp, i32, i64, i32, ctypes.POINTER(_Traffic), vp]
    lib.ra_reducer_create.argtypes = [pvp, i32, i32, ctypes.POINTER(ctypes.c_int64), i32, i64,
                                      ctypes.POINTER(ctypes.c_void_p)]
    lib.ra_reducer_buckets.argtypes = [vp, ctypes.POINTER(_Bucket), i32, ctypes.POINTER(i32)]
    lib.ra_reducer_mark_ready.argtypes = [vp, i32, vp]
    lib.ra_reducer_finish.argtypes = [vp, vp]
    lib.ra_reducer_destroy.argtypes = [vp]
    lib.ra_check_device_errors.argtypes = []
    lib.ra_selftest_wait_timeout.argtypes = [i32, vp]
    lib.ra_selftest_bounds_check.argtypes = [pvp, i32, i64, i32, vp]
    lib.ra_chunk_range.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    lib.ra_chunk_range.restype = None
    lib.ra_status_str.argtypes = [i32]
    lib.ra_status_str.restype = ctypes.c_char_p
    lib.ra_last_cuda_error.argtypes = []
    for nm in ("ra_allreduce_avg", "ra_allreduce_sgd", "ra_allreduce_avg_staged", "ra_bucket_plan",
               "ra_allreduce_avg_buckets", "ra_allreduce_avg_host", "ra_allreduce_avg_staged_static",
               "ra_reduce_scatter_avg", "ra_all_gather", "ra_allreduce_avg_bf16_wire",
               "ra_allreduce_avg_single_reducer", "ra_reducer_create", "ra_reducer_buckets",
               "ra_reducer_mark_ready", "ra_reducer_finish", "ra_reducer_destroy", "ra_check_device_errors",
               "ra_selftest_wait_timeout", "ra_selftest_bounds_check", "ra_last_cuda_error"):
        getattr(lib, nm).restype = i32
    _lib = lib
    return lib


# ---------------------------------------------------------------------------
# marshalling


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return RA_F32
    if t.dtype == torch.bfloat16:
        return RA_BF16
    raise TypeError("gradients must be float32 or bfloat16, got %s" % t.dtype)


def _rows(tensors):
    """(pointer array, n, p, dtype code, device) for a list of worker tensors."""
    if not isinstance(tensors, (list, tuple)):
        tensors = list(tensors)
    if not tensors:
        raise ValueError("need at least one worker buffer")
    n = len(tensors)
    t0 = tensors[0]
    dt = _dtype_code(t0)
    dtype, p, dev = t0.dtype, t0.numel(), t0.get_device()
    ptrs = [0] * n
    for k, t in enumerate(tensors):
        # one pass, integer device ids: this runs on every call
        if t.get_device() != dev or dev < 0:
            raise ValueError("worker buffers must be CUDA tensors on one device")
        if t.dtype != dtype or t.numel() != p:
            raise ValueError("worker buffers must share dtype, length and device")
        if not t.is_contiguous():
            raise ValueError("worker buffers must be contiguous")
        ptrs[k] = t.data_ptr()
    return (ctypes.c_void_p * n)(*ptrs), n, p, dt, t0.device


def _stream(stream, device):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, what: str):
    if status != 0:
        raise RaError(status, what)


# ---------------------------------------------------------------------------
# the calls


def ra_allreduce_avg(tensors, stream=None) -> None:
    """Every worker tensor becomes the element-wise mean of all of them."""
    arr, n, p, dt, dev = _rows(tensors)
    _check(load().ra_allreduce_avg(arr, n, p, dt, _stream(stream, dev)), "ra_allreduce_avg")


def ra_allreduce_sgd(tensors, w, lr: float, stream=None) -> None:
    """ra_allreduce_avg plus w -= lr * mean in the same pass (w: float32 CUDA tensor)."""
    import torch
    arr, n, p, dt, dev = _rows(tensors)
    if w.dtype != torch.float32 or w.numel() != p or not w.is_contiguous() or w.device != dev:
        raise ValueError("w must be a contiguous float32 tensor of the gradients' length and device")
    _check(load().ra_allreduce_sgd(arr, n, p, dt, ctypes.c_void_p(w.data_ptr()), float(lr), _stream(stream, dev)),
           "ra_allreduce_sgd")


def ra_staged_workspace_bytes(n: int, p: int, dtype: int) -> int:
    return int(load().ra_staged_workspace_bytes(n, p, dtype))


def ra_allreduce_avg_staged(tensors, workspace=None, stream=None):
    """The literal 2(N-1)+1-launch ring; returns [(sent, received)] per worker.
    `workspace` is a CUDA tensor of at least ra_staged_workspace_bytes bytes
    (allocated here with torch when None and needed)."""
    import torch
    arr, n, p, dt, dev = _rows(tensors)
    need = ra_staged_workspace_bytes(n, p, dt)
    ws_ptr, ws_bytes = None, 0
    if need > 0:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    traffic = (_Traffic * n)()
    _check(load().ra_allreduce_avg_staged(arr, n, p, dt, ctypes.c_void_p(ws_ptr), ws_bytes, traffic,
                                          _stream(stream, dev)), "ra_allreduce_avg_staged")
    return [(traffic[k].sent, traffic[k].received) for k in range(n)]


def ra_allreduce_avg_staged_static(tensors, stream=None):
    """The staged ring without a workspace argument, for callers that cannot
    allocate device memory: the bf16 partial sums use a scratch array built
    into the library (at most RA_STAGED_STATIC_MAX_P elements per worker for
    bf16).  Returns [(sent, received)] per worker."""
    arr, n, p, dt, dev = _rows(tensors)
    traffic = (_Traffic * n)()
    _check(load().ra_allreduce_avg_staged_static(arr, n, p, dt, traffic, _stream(stream, dev)),
           "ra_allreduce_avg_staged_static")
    return [(traffic[k].sent, traffic[k].received) for k in range(n)]


def ra_bucket_plan(numel, elem_bytes: int, cap_bytes: int):
    """Reverse-order buckets of whole tensors, each >= cap_bytes but the last;
    returns [(offset, count)] in elements of the forward-ordered flat array."""
    numel = [int(x) for x in numel]
    nt = len(numel)
    arr = (ctypes.c_int64 * max(1, nt))(*numel)
    out = (_Bucket * (nt + 1))()
    nb = ctypes.c_int(0)
    _check(load().ra_bucket_plan(arr, nt, elem_bytes, cap_bytes, out, nt + 1, ctypes.byref(nb)), "ra_bucket_plan")
    return [(out[k].offset, out[k].count) for k in range(nb.value)]


def ra_allreduce_avg_buckets(tensors, buckets, stream=None) -> None:
    """Each (offset, count) bucket of the worker tensors is its own ring."""
    arr, n, p, dt, dev = _rows(tensors)
    for off, cnt in buckets:
        if off < 0 or cnt < 0 or off + cnt > p:
            raise ValueError("bucket (%d, %d) outside the %d-element buffers" % (off, cnt, p))
    nb = len(buckets)
    b = (_Bucket * max(1, nb))(*[_Bucket(int(o), int(c)) for o, c in buckets])
    _check(load().ra_allreduce_avg_buckets(arr, n, dt, b, nb, _stream(stream, dev)), "ra_allreduce_avg_buckets")


def ra_allreduce_avg_host(host_tensors, dev_tensors=None, mode=RA_HOST_AUTO, stream=None) -> None:
    """Every host (CPU) worker tensor becomes the mean.  The fused kernel works
    on the host memory directly when the device can address it (pinned
    memory, or any memory on a device that walks the host page tables);
    otherwise -- or with mode=RA_HOST_STAGED -- through the device staging
    tensors."""
    import torch
    host_tensors = list(host_tensors)
    if not host_tensors:
        raise ValueError("need at least one worker buffer")
    n = len(host_tensors)
    h0 = host_tensors[0]
    dt = _dtype_code(h0)
    p = h0.numel()
    for h in host_tensors:
        if h.is_cuda or h.numel() != p or h.dtype != h0.dtype or not h.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors of one dtype and length")
    harr = (ctypes.c_void_p * n)(*[h.data_ptr() for h in host_tensors])
    if dev_tensors is not None:
        darr, dn, dp, ddt, dev = _rows(dev_tensors)
        if dn != n or dp != p or ddt != dt:
            raise ValueError("device staging tensors must match the host tensors")
    else:
        darr, dev = None, torch.device("cuda", torch.cuda.current_device())
    _check(load().ra_allreduce_avg_host(harr, darr, n, p, dt, int(mode), _stream(stream, dev)),
           "ra_allreduce_avg_host")


def _shards(shards, tensors, n, p):
    if shards is None:
        return None
    shards = list(shards)
    if len(shards) != n:
        raise ValueError("need one shard per worker")
    for m, sh in enumerate(shards):
        b, e = ra_chunk_range(p, n, (m + 1) % n)
        if not sh.is_cuda or sh.dtype != tensors[0].dtype or sh.numel() != e - b or not sh.is_contiguous():
            raise ValueError("shard %d must be a contiguous CUDA tensor of chunk %d's %d elements"
                             % (m, (m + 1) % n, e - b))
    return (ctypes.c_void_p * n)(*[sh.data_ptr() for sh in shards])


def ra_reduce_scatter_avg(tensors, shards=None, stream=None) -> None:
    """Worker (c-1) mod N ends with the mean of chunk c: in place in its own
    tensor, or in shards[(c-1) mod N] when shards are given."""
    tensors = list(tensors)
    arr, n, p, dt, dev = _rows(tensors)
    sh = _shards(shards, tensors, n, p)
    _check(load().ra_reduce_scatter_avg(arr, n, p, dt, sh, _stream(stream, dev)), "ra_reduce_scatter_avg")


def ra_all_gather(tensors, shards=None, stream=None) -> None:
    """Chunk c of worker (c-1) mod N (or shards[(c-1) mod N]) is copied into
    every worker's tensor."""
    tensors = list(tensors)
    arr, n, p, dt, dev = _rows(tensors)
    sh = _shards(shards, tensors, n, p)
    _check(load().ra_all_gather(arr, n, p, dt, sh, _stream(stream, dev)), "ra_all_gather")


def ra_allreduce_avg_bf16_wire(tensors, stream=None) -> None:
    """bf16 all-reduce with every partial sum rounded to bf16 (a bf16 ring)."""
    arr, n, p, dt, dev = _rows(tensors)
    if dt != RA_BF16:
        raise TypeError("ra_allreduce_avg_bf16_wire takes bfloat16 tensors")
    _check(load().ra_allreduce_avg_bf16_wire(arr, n, p, _stream(stream, dev)), "ra_allreduce_avg_bf16_wire")


def ra_allreduce_avg_single_reducer(tensors, stream=None):
    """Mean by the single-reducer scheme (worker 0 sums in worker order);
    returns that scheme's [(sent, received)] per worker."""
    arr, n, p, dt, dev = _rows(tensors)
    traffic = (_Traffic * n)()
    _check(load().ra_allreduce_avg_single_reducer(arr, n, p, dt, traffic, _stream(stream, dev)),
           "ra_allreduce_avg_single_reducer")
    return [(traffic[k].sent, traffic[k].received) for k in range(n)]


class Reducer:
    """ra_reducer: buckets of layer tensors all-reduced as their gradients
    become ready (output layer first), on a stream of the reducer's own.

    flat_tensors: one contiguous CUDA tensor per worker holding the layer
    gradients back to back in forward order; numel: the layer sizes."""

    def __init__(self, flat_tensors, numel, cap_bytes: int):
        flat_tensors = list(flat_tensors)
        arr, n, p, dt, dev = _rows(flat_tensors)
        numel = [int(x) for x in numel]
        if sum(numel) != p:
            raise ValueError("the layer sizes must add up to the flat length")
        self._keep = flat_tensors
        self.device = dev
        cnt = (ctypes.c_int64 * max(1, len(numel)))(*numel)
        h = ctypes.c_void_p()
        _check(load().ra_reducer_create(arr, n, dt, cnt, len(numel), int(cap_bytes), ctypes.byref(h)),
               "ra_reducer_create")
        self._h = h
        self.ntensors = len(numel)

    def buckets(self):
        out = (_Bucket * (self.ntensors + 1))()
        nb = ctypes.c_int(0)
        _check(load().ra_reducer_buckets(self._h, out, self.ntensors + 1, ctypes.byref(nb)), "ra_reducer_buckets")
        return [(out[k].offset, out[k].count) for k in range(nb.value)]

    def mark_ready(self, tensor: int, stream=None) -> None:
        _check(load().ra_reducer_mark_ready(self._h, int(tensor), _stream(stream, self.device)),
               "ra_reducer_mark_ready")

    def finish(self, stream=None) -> None:
        _check(load().ra_reducer_finish(self._h, _stream(stream, self.device)), "ra_reducer_finish")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _check(load().ra_reducer_destroy(self._h), "ra_reducer_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ra_check_device_errors() -> int:
    """What the kernels on the current device recorded since the last check:
    0 (RA_OK), 5 (RA_ERR_TIMEOUT: a bounded wait gave up) or, in the
    bounds-checked build, 6 (RA_ERR_BOUNDS); clears the record."""
    return int(load().ra_check_device_errors())


def ra_selftest_bounds_check(tensors, stream=None) -> None:
    """Bounds-checked build: run the fused all-reduce while telling the kernel
    the rows are one element shorter than they are, so that the check must
    report RA_ERR_BOUNDS (rows' contents afterwards unspecified).  The
    product build raises RaError(RA_ERR_UNSUPPORTED)."""
    arr, n, p, dt, dev = _rows(tensors)
    _check(load().ra_selftest_bounds_check(arr, n, p, dt, _stream(stream, dev)), "ra_selftest_bounds_check")


def ra_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    """Queue a kernel whose bounded wait is made to expire (a timeout test)."""
    import torch
    _check(load().ra_selftest_wait_timeout(int(timeout_us), _stream(stream, torch.device("cuda", torch.cuda.current_device()))),
           "ra_selftest_wait_timeout")


def ra_chunk_range(p: int, n: int, c: int):
    b, e = ctypes.c_int64(), ctypes.c_int64()
    load().ra_chunk_range(p, n, c, ctypes.byref(b), ctypes.byref(e))
    return b.value, e.value


def ra_status_str(status: int) -> str:
    return load().ra_status_str(status).decode()


def ra_last_cuda_error() -> int:
    return load().ra_last_cuda_error()
