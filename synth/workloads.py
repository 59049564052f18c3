"""The five synthetic workloads, named by what they are.

Each worker n's gradient row is generator stream n of the workload's seed.
Sizes and distributions follow the pages' models:
  - the 300M-parameter speech model with a 1.2 GB fp32 gradient
    (Gibiansky, "The Communication Problem"),
  - the 24-layer Transformer of the GPipe page (section 1),
  - ResNet-18 with about 11.7M parameters ("[AI System] Training With
    Multiple GPUs", section Memory).
The second number of "N(0, s)" is the standard deviation.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from .shapes import numels, resnet18_shapes, transformer_shapes

BUCKET_CAP_BYTES = 25 * 1024 * 1024  # 25 MiB


@dataclass(frozen=True)
class Workload:
    name: str
    n: int                 # workers
    p: int                 # elements per worker
    dtype: str             # "f32" or "bf16"
    dist: str              # "normal" or "student_t3"
    scale: float           # sigma of the normal, or the factor on Student-t
    seed: int
    tensors: tuple = field(default=())      # layer numels (forward order) if layer-shaped
    bucket_cap_bytes: int = 0               # >0: reduce in reverse-order buckets
    sgd_lr: float = 0.0                     # >0: fused SGD update
    w_sigma: float = 0.0
    w_seed: int = 0

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def min_bytes(self) -> int:
        """N*P reads + N*P writes (+ read and write of the fp32 weights for SGD)."""
        b = 2 * self.n * self.p * self.elem_bytes
        if self.sgd_lr > 0:
            b += 2 * self.p * 4
        return b

    def fill_row(self, ptr: int, worker: int, start: int = 0, count: int | None = None, threads=None):
        from . import fill_normal_f32, fill_student_t3_bf16
        count = self.p - start if count is None else count
        if self.dist == "normal":
            fill_normal_f32(ptr, self.seed, worker, self.scale, start, count, threads)
        else:
            fill_student_t3_bf16(ptr, self.seed, worker, self.scale, start, count, threads)

    def row(self, worker: int, start: int = 0, count: int | None = None):
        from . import normal_f32, student_t3_bf16
        count = self.p - start if count is None else count
        if self.dist == "normal":
            return normal_f32(self.seed, worker, self.scale, start, count)
        return student_t3_bf16(self.seed, worker, self.scale, start, count)

    def values_at(self, worker: int, idx):
        from . import normal_f32_at, student_t3_bf16_at
        if self.dist == "normal":
            return normal_f32_at(self.seed, worker, self.scale, idx)
        return student_t3_bf16_at(self.seed, worker, self.scale, idx)

    def weights(self, start: int = 0, count: int | None = None):
        from . import normal_f32
        count = self.p - start if count is None else count
        return normal_f32(self.w_seed, 0, self.w_sigma, start, count)

    def fill_weights(self, ptr: int, start: int = 0, count: int | None = None, threads=None):
        from . import fill_normal_f32
        count = self.p - start if count is None else count
        fill_normal_f32(ptr, self.w_seed, 0, self.w_sigma, start, count, threads)

    def weights_at(self, idx):
        from . import normal_f32_at
        return normal_f32_at(self.w_seed, 0, self.w_sigma, idx)


_TF = tuple(numels(transformer_shapes()))
_RN = tuple(numels(resnet18_shapes()))

WORKLOADS = {
    w.name: w
    for w in (
        Workload("ring4_uneven_1m_f32", n=4, p=1_048_579, dtype="f32", dist="normal", scale=1.0, seed=0),
        Workload("speech300m_n8_f32", n=8, p=300_000_000, dtype="f32", dist="normal", scale=1e-3, seed=1),
        Workload("transformer24_buckets_n4_f32", n=4, p=sum(_TF), dtype="f32", dist="normal", scale=1e-2,
                 seed=2, tensors=_TF, bucket_cap_bytes=BUCKET_CAP_BYTES),
        Workload("student_t3_1g_n16_bf16", n=16, p=1_000_000_000, dtype="bf16", dist="student_t3", scale=1e-3,
                 seed=3),
        Workload("resnet18_sgd_n32_f32", n=32, p=sum(_RN), dtype="f32", dist="normal", scale=1e-2, seed=4,
                 tensors=_RN, sgd_lr=0.1, w_sigma=0.05, w_seed=5),
    )
}
