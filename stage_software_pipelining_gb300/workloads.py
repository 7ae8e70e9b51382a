"""Seeded synthetic inputs for the pipelined GEMM workloads.

This module only draws random matrices; it holds none of the GEMM's
arithmetic.  Both the CUDA path and the CPU oracle take their inputs from it,
and nothing else is shared between the two.

The five workloads are the ones the GEMM is measured on:

=====================  =====================================  ==============================
name                   shape / types                          values
=====================  =====================================  ==============================
``fp32_256``           256^3, fp32 -> fp32, SIMT, stages 1,2   A, B ~ U[-1, 1]
``fp32_2048``          2048^3, fp32 -> fp32, SIMT 128x64       A, B ~ U[-1, 1]
``fp16_2048``          2048^3, fp16 -> fp32, tensor cores      A, B ~ N(0, 1) rounded to fp16
``bf16_8192_beta1``    8192^3, bf16 -> fp32, beta = 1          A, B ~ U[-1, 1] rounded to bf16;
                                                               C0 ~ U[-1, 1] fp32
``bf16_ragged_colB``   8191 x 28672 x 4096, bf16 -> bf16,      A, B ~ N(0, 0.02) rounded to bf16
                       A row-major, B column-major
=====================  =====================================  ==============================

The pages measure on no public data set, so these synthetic matrices are the
whole workload.  Values are drawn in fp32 on the host by a seeded
``torch.Generator`` (seed 20261202 + workload index) and rounded to the input
type with round-to-nearest-even; every consumer reads those rounded host copies.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

SEED_BASE = 20261202

# Input/output type pairs of the C entry point (mirrors gemm_dtype_t in include/gemm.h).
GEMM_F32 = 0          # fp32 inputs, fp32 output: CUDA-core SIMT path
GEMM_F16_F32 = 1      # fp16 inputs, fp32 accumulate and output: tensor cores
GEMM_BF16_F32 = 2     # bf16 inputs, fp32 accumulate and output: tensor cores
GEMM_BF16_BF16 = 3    # bf16 inputs, fp32 accumulate, bf16 output: tensor cores

IN_DTYPE = {GEMM_F32: torch.float32, GEMM_F16_F32: torch.float16,
            GEMM_BF16_F32: torch.bfloat16, GEMM_BF16_BF16: torch.bfloat16}
OUT_DTYPE = {GEMM_F32: torch.float32, GEMM_F16_F32: torch.float32,
             GEMM_BF16_F32: torch.float32, GEMM_BF16_BF16: torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    index: int            # position in the workload list; selects the seed
    M: int
    N: int
    K: int
    dtype: int            # GEMM_* type pair
    dist: str             # "uniform" (U[-1,1]) or "normal"
    std: float = 1.0      # standard deviation for "normal"
    alpha: float = 1.0
    beta: float = 0.0
    b_col_major: bool = False
    stages: tuple = field(default=(1, 2))

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def resized(self, M: int, N: int, K: int) -> "Workload":
        """Same distributions, types and scalars at another shape."""
        return replace(self, M=M, N=N, K=K)


WORKLOADS = [
    Workload("fp32_256", 0, 256, 256, 256, GEMM_F32, "uniform", stages=(1, 2)),
    Workload("fp32_2048", 1, 2048, 2048, 2048, GEMM_F32, "uniform", stages=(1, 2)),
    Workload("fp16_2048", 2, 2048, 2048, 2048, GEMM_F16_F32, "normal", 1.0,
             stages=(1, 2, 3, 4)),
    Workload("bf16_8192_beta1", 3, 8192, 8192, 8192, GEMM_BF16_F32, "uniform", beta=1.0,
             stages=(1, 2, 3, 4, 5, 6)),
    Workload("bf16_ragged_colB", 4, 8191, 28672, 4096, GEMM_BF16_BF16, "normal", 0.02,
             b_col_major=True, stages=(4,)),
]
BY_NAME = {w.name: w for w in WORKLOADS}


def _draw(gen: torch.Generator, shape, w: Workload) -> torch.Tensor:
    if w.dist == "uniform":
        x = torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    elif w.dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32) * w.std
    else:
        raise ValueError(w.dist)
    return x


@dataclass
class Inputs:
    """Host (CPU) tensors of one workload instance.

    A is M x K row-major.  B is the logical K x N matrix: row-major storage, or,
    when the workload says column-major, a transposed view of an N x K
    row-major tensor.  C0 is the M x N initial C (None when beta == 0).
    """
    workload: Workload
    A: torch.Tensor
    B: torch.Tensor
    C0: torch.Tensor | None


def make_inputs(w: Workload, seed_offset: int = 0) -> Inputs:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(SEED_BASE + w.index + 1000 * seed_offset)
    in_dt = IN_DTYPE[w.dtype]
    A = _draw(gen, (w.M, w.K), w).to(in_dt)
    if w.b_col_major:
        B = _draw(gen, (w.N, w.K), w).to(in_dt).t()      # K x N view, column-major storage
    else:
        B = _draw(gen, (w.K, w.N), w).to(in_dt)
    C0 = None
    if w.beta != 0.0:
        C0 = (torch.rand((w.M, w.N), generator=gen, dtype=torch.float32) * 2.0 - 1.0)
        C0 = C0.to(OUT_DTYPE[w.dtype])
    return Inputs(w, A, B, C0)
