"""Seeded synthetic inputs for the dense half-precision GEMM workloads.

This module only draws random numbers and lays them out in memory; it holds
none of the GEMM's arithmetic.  Both the oracle-side tests and the CUDA-side
tests and benchmark take their inputs from here, so both sides see the same
bit patterns.

The workloads are the ones the pages measure or describe, made synthetic
(the pages name no dataset):

* ``pr1``      -- 256^3, fp16 row-major A and B, U[-1,1], fp32 acc/out.
* ``sq4096``   -- 4096^3, fp16 row-major A and B, U[-1,1], fp32 acc/out
  (the size the WMMA page benchmarks).
* ``sq4096h``  -- 4096^3, A row-major, B column-major, U[-0.5,0.5],
  fp16 accumulate and fp16 output (the m16n8k16 f16.f16.f16.f16 variant).
* ``ragged``   -- M=4097, N=2055, K=1000, A row-major, B column-major,
  N(0,1); C fp32 N(0,1); alpha=0.5, beta=1; fp32 acc/out.
* ``bf16_<n>`` -- bf16 square sweep n in {1024, 2048, 8192, 16384}, row-major,
  U[-1,1], fp32 accumulate, bf16 output.
* ``skinny``   -- bf16 M=16, N=K=8192, same recipe (memory-bound).
* ``sq8192``   -- 8192^3 with the ``sq4096`` recipe (the second size of the
  throughput target).
* ``e4m3_8192``, ``e5m2_8192``, ``tf32_4096`` -- the other tensor-core input
  types (8-bit floats, TF32), A row-major and B column-major, U[-1,1], fp32
  accumulate, bf16 (8-bit) or fp32 (TF32) output.  TF32 operands are fp32
  values whose 13 low fraction bits are cleared, so the tensor cores read
  them exactly.

Every workload also has an integer twin: entries drawn uniformly from
{-2,-1,0,1,2} (and C too, where beta != 0), for which every partial sum is an
exact integer, so device results can be compared bit for bit.

Seeds: workload number i uses seed 1000+i for A, 2000+i for B and 3000+i for
C (the twin adds 500).  Values are drawn as float32 by a CPU
``torch.Generator`` and converted with ``Tensor.to`` (round-to-nearest-even).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32, "e4m3": torch.float8_e4m3fn,
          "e5m2": torch.float8_e5m2, "tf32": torch.float32}
ELEMENT_BYTES = {"f16": 2, "bf16": 2, "f32": 4, "e4m3": 1, "e5m2": 1, "tf32": 4}


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    M: int
    N: int
    K: int
    in_dtype: str          # "f16" | "bf16" | "e4m3" | "e5m2" | "tf32"
    layoutA: str           # "row" | "col"
    layoutB: str
    accum_dtype: str       # "f32" | "f16"
    out_dtype: str         # "f32" | "f16" | "bf16"
    alpha: float
    beta: float
    dist: str              # "u1" = U[-1,1], "u05" = U[-0.5,0.5], "n01" = N(0,1)

    @property
    def lda(self) -> int:
        return self.K if self.layoutA == "row" else self.M

    @property
    def ldb(self) -> int:
        return self.N if self.layoutB == "row" else self.K

    @property
    def ldc(self) -> int:
        return self.N

    @property
    def flops(self) -> int:
        """2*M*N*K: one multiply and one add per multiply-accumulate."""
        return 2 * self.M * self.N * self.K

    def algorithmic_bytes(self) -> int:
        """|A| + |B| + |C if beta != 0| + |D|, each read or written once."""
        e_in = ELEMENT_BYTES[self.in_dtype]
        e_out = ELEMENT_BYTES[self.out_dtype]
        b = (self.M * self.K + self.K * self.N) * e_in + self.M * self.N * e_out
        if self.beta != 0.0:
            b += self.M * self.N * e_out
        return b

    def with_shape(self, M: int, N: int, K: int, name: str | None = None) -> "Workload":
        return replace(self, M=M, N=N, K=K, name=name or f"{self.name}@{M}x{N}x{K}")


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("pr1", 1, 256, 256, 256, "f16", "row", "row", "f32", "f32", 1.0, 0.0, "u1"),
        Workload("sq4096", 2, 4096, 4096, 4096, "f16", "row", "row", "f32", "f32", 1.0, 0.0, "u1"),
        Workload("sq4096h", 3, 4096, 4096, 4096, "f16", "row", "col", "f16", "f16", 1.0, 0.0, "u05"),
        Workload("ragged", 4, 4097, 2055, 1000, "f16", "row", "col", "f32", "f32", 0.5, 1.0, "n01"),
        Workload("bf16_1024", 5, 1024, 1024, 1024, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"),
        Workload("bf16_2048", 5, 2048, 2048, 2048, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"),
        Workload("bf16_8192", 5, 8192, 8192, 8192, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"),
        Workload("bf16_16384", 5, 16384, 16384, 16384, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"),
        Workload("skinny", 5, 16, 8192, 8192, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"),
        # the second square size the throughput target names (fp16 -> fp32 at 8192^3)
        Workload("sq8192", 6, 8192, 8192, 8192, "f16", "row", "row", "f32", "f32", 1.0, 0.0, "u1"),
        # the other tensor-core input kinds (K-major operands)
        Workload("e4m3_8192", 7, 8192, 8192, 8192, "e4m3", "row", "col", "f32", "bf16", 1.0, 0.0, "u1"),
        Workload("e5m2_8192", 8, 8192, 8192, 8192, "e5m2", "row", "col", "f32", "bf16", 1.0, 0.0, "u1"),
        Workload("tf32_4096", 9, 4096, 4096, 4096, "tf32", "row", "col", "f32", "f32", 1.0, 0.0, "u1"),
    ]
}


def _storage_shape(rows: int, cols: int, layout: str, ld: int) -> tuple[int, int]:
    """2-D shape of the buffer that holds a rows x cols matrix with leading
    dimension ld: row-major keeps rows of ld elements, column-major keeps
    columns of ld elements."""
    return (rows, ld) if layout == "row" else (cols, ld)


def draw(shape, dist: str, dtype: str, seed: int, integer: bool = False) -> torch.Tensor:
    """iid entries of the given distribution, rounded to ``dtype`` (CPU)."""
    g = torch.Generator().manual_seed(seed)
    if integer:
        x = torch.randint(-2, 3, shape, generator=g, dtype=torch.int32).to(torch.float32)
    elif dist == "u1":
        x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
    elif dist == "u05":
        x = torch.rand(shape, generator=g, dtype=torch.float32) - 0.5
    elif dist == "n01":
        x = torch.randn(shape, generator=g, dtype=torch.float32)
    else:
        raise ValueError(dist)
    if dtype == "tf32":
        # fp32 storage with the 13 low fraction bits cleared: TF32-exact values
        return (x.view(torch.int32) & -8192).view(torch.float32)
    return x.to(DTYPES[dtype])


def draw_matrix(rows: int, cols: int, layout: str, ld: int, dist: str, dtype: str,
                seed: int, integer: bool = False) -> torch.Tensor:
    """A rows x cols matrix in the given storage order, as its 2-D storage
    buffer (entries beyond the logical extent, when ld is larger, are drawn
    too; they are never part of the product)."""
    return draw(_storage_shape(rows, cols, layout, ld), dist, dtype, seed, integer)


@dataclass
class Inputs:
    A: torch.Tensor          # storage buffer (row-major: M x lda, col-major: K x lda)
    B: torch.Tensor          # storage buffer (row-major: K x ldb, col-major: N x ldb)
    C: torch.Tensor | None   # M x ldc in out_dtype, or None when beta == 0
    lda: int
    ldb: int
    ldc: int


def make_inputs(w: Workload, integer: bool = False, lda: int | None = None,
                ldb: int | None = None, ldc: int | None = None, with_c: bool | None = None,
                seed_offset: int = 0) -> Inputs:
    """Host (CPU) inputs of workload ``w``; padded leading dimensions may be
    asked for.  ``with_c`` forces a C buffer even when beta == 0 (to check
    that C is then not read)."""
    lda = lda or w.lda
    ldb = ldb or w.ldb
    ldc = ldc or w.ldc
    twin = 500 if integer else 0
    s = seed_offset + twin
    A = draw_matrix(w.M, w.K, w.layoutA, lda, w.dist, w.in_dtype, 1000 + w.index + s, integer)
    B = draw_matrix(w.K, w.N, w.layoutB, ldb, w.dist, w.in_dtype, 2000 + w.index + s, integer)
    need_c = (w.beta != 0.0) if with_c is None else with_c
    C = None
    if need_c:
        C = draw((w.M, ldc), "n01", w.out_dtype, 3000 + w.index + s, integer)
    return Inputs(A, B, C, lda, ldb, ldc)


def logical(mat: torch.Tensor, rows: int, cols: int, layout: str) -> torch.Tensor:
    """The rows x cols logical view of a storage buffer (no copy)."""
    if layout == "row":
        return mat[:rows, :cols]
    return mat[:cols, :rows].t()


def bits(t: torch.Tensor):
    """numpy view of a CPU tensor as the oracle wants it: uint16 bit patterns
    for fp16/bf16, uint8 for the 8-bit floats, float32 for fp32 (and TF32
    operands)."""
    t = t.contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError(t.dtype)
