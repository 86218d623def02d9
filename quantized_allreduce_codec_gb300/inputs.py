"""Seeded synthetic rank messages for the quick-allreduce workloads.

This module only draws random numbers and rounds them to fp16/bf16 with
library casts; it holds none of the codec's or the reduction's arithmetic.
Both the CUDA path's tests and benchmark and the CPU oracle's tests take
their inputs from here.

Recipe (numpy PCG64 ``default_rng``; rank r of workload k uses seed
1000*k + r; values are drawn in binary32 and rounded to the message dtype
with a round-half-to-even library cast):

* ``normal``   N(0, sigma)                                    (workloads 1, 2)
* ``outliers`` N(0, 1); each element independently, with probability 0.001,
  multiplied by 50 (the mask is drawn after the normals)     (workloads 3, 5)
* ``rowscale`` N(0, 0.5) times a per-row factor drawn log-uniform on
  [0.1, 10]; the factors are drawn once, from seed 1000*k + 999, and
  shared by every rank (a per-token magnitude)                (workload 4)

The pages measure the allreduce on a tp2 size sweep of fp16 messages
(4k .. 64M, the timing table of vLLM PR #18473); no dataset is involved.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

F16, BF16 = 0, 1
FP, Q8, Q6, Q4, FP8, Q8A, Q4A = 0, 1, 2, 3, 4, 5, 6
FORMAT_NAMES = {FP: "FP", Q8: "Q8", Q6: "Q6", Q4: "Q4", FP8: "FP8", Q8A: "Q8A", Q4A: "Q4A"}
DTYPE_NAMES = {F16: "fp16", BF16: "bf16"}
ALL_FORMATS = (FP, FP8, Q8, Q6, Q4, Q8A, Q4A)


def to_bits(values_f32: np.ndarray, dtype: int) -> np.ndarray:
    """Round binary32 values to fp16/bf16 (library RNE cast); uint16 bits."""
    v = np.ascontiguousarray(values_f32, dtype=np.float32)
    if dtype == F16:
        return v.astype(np.float16).view(np.uint16)
    t = torch.from_numpy(v).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def from_bits(bits: np.ndarray, dtype: int) -> np.ndarray:
    """fp16/bf16 bit patterns to binary32 values (exact widening)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == F16:
        return b.view(np.float16).astype(np.float32)
    return (b.astype(np.uint32) << 16).view(np.float32)


def rank_values(kind: str, seed: int, n: int, *, sigma: float = 1.0,
                rows: int | None = None, row_seed: int | None = None) -> np.ndarray:
    """binary32 values of one rank's message (before rounding to dtype)."""
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return (rng.standard_normal(n, dtype=np.float32) * np.float32(sigma)).astype(np.float32)
    if kind == "outliers":
        x = rng.standard_normal(n, dtype=np.float32)
        mask = rng.random(n, dtype=np.float32) < np.float32(0.001)
        x[mask] *= np.float32(50.0)
        return x
    if kind == "rowscale":
        assert rows and n % rows == 0
        x = rng.standard_normal(n, dtype=np.float32) * np.float32(0.5)
        rrng = np.random.default_rng(row_seed)
        factors = np.exp(rrng.uniform(np.log(0.1), np.log(10.0), rows)).astype(np.float32)
        x = x.reshape(rows, n // rows) * factors[:, None]
        return x.reshape(-1).astype(np.float32)
    raise ValueError(kind)


@dataclass(frozen=True)
class Workload:
    """One emulated allreduce workload: W ranks of n elements each."""
    key: int
    name: str
    W: int
    dtype: int
    n: int
    kind: str
    formats: tuple
    stages: tuple = (2,)
    rows: int | None = None
    sigma: float = 1.0
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def bytes_per_rank(self) -> int:
        return self.n * 2

    def rank_bits(self, r: int) -> np.ndarray:
        vals = rank_values(self.kind, 1000 * self.key + r, self.n, sigma=self.sigma,
                           rows=self.rows, row_seed=1000 * self.key + 999)
        return to_bits(vals, self.dtype)

    def inputs(self) -> list:
        return [self.rank_bits(r) for r in range(self.W)]


def sweep_sizes_bytes():
    """Per-rank message sizes of the tp2 table: 4 KiB .. 64 MiB, powers of two."""
    return [4096 << k for k in range(15)]


def workloads() -> dict:
    """The five workloads (sizes in elements per rank)."""
    w = {}
    w[1] = Workload(1, "W2-fp16-8KiB-Q8", 2, F16, 4096, "normal", (Q8,), (2,))
    w[2] = Workload(2, "W2-fp16-sweep", 2, F16, (64 << 20) // 2, "normal",
                    (FP, FP8, Q8, Q6, Q4), (1, 2))
    w[3] = Workload(3, "W4-bf16-2048x4096-Q4A", 4, BF16, 2048 * 4096, "outliers", (Q4A,), (2,),
                    rows=2048)
    w[4] = Workload(4, "W8-bf16-4096x8192-Q6-Q8A", 8, BF16, 4096 * 8192, "rowscale",
                    (Q6, Q8A), (2,), rows=4096, sigma=0.5)
    w[5] = Workload(5, "W8-fp16-8192x8192-all", 8, F16, 8192 * 8192, "outliers",
                    ALL_FORMATS, (1, 2), rows=8192)
    return w


def sweep_workload(size_bytes: int) -> Workload:
    """One point of the tp2 size sweep (W=2, fp16, N(0,1))."""
    return Workload(2, f"W2-fp16-{size_bytes}B", 2, F16, size_bytes // 2, "normal",
                    (FP, FP8, Q8, Q6, Q4), (1, 2))


def long_message_bits(seed: int, n: int, dtype: int, tile: int = 1 << 20) -> np.ndarray:
    """A message of n values too long to draw value by value in a test (for
    checks of 64-bit offsets past 2^31 elements): one N(0, 1) tile of `tile`
    values drawn with `seed`, repeated, tile i scaled by 2^((5*i mod 13) - 6)
    before the rounding to dtype.  Tiles whose indices differ by a
    power of two never share a scale (13 is prime), so a 32-bit offset that
    wrapped would read different values."""
    base = np.random.default_rng(seed).standard_normal(tile, dtype=np.float32)
    variants = [to_bits(base * np.float32(2.0 ** (s - 6)), dtype) for s in range(13)]
    out = np.empty(n, np.uint16)
    for i, start in enumerate(range(0, n, tile)):
        stop = min(start + tile, n)
        out[start:stop] = variants[(5 * i) % 13][:stop - start]
    return out
