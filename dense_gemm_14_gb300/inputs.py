"""Seeded synthetic inputs for the GEMM workloads.

This module draws random matrices and nothing else: it holds none of the
product's arithmetic, so both the CUDA path's tests/bench and the CPU oracle
may take their inputs from it.

Recipe (the pages fix only the shapes and the fp32 element type of their
worked example; the distributions and seeds below are this library's choice):
A is drawn first, then B, from one ``torch.Generator`` seeded per workload, in
float32 on the CPU; uniform[-1, 1) is ``rand * 2 - 1`` and normal(0, s) is
``randn * s``. For the 16-bit workloads the float32 draws are rounded to
bfloat16 / float16 with torch's round-to-nearest-even ``.to()``; the library
and the oracle both see exactly those rounded values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

_TORCH_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dtype: str          # input element type: "f32", "bf16" or "f16"
    dist: str           # "uniform" (on [-1, 1)) or "normal"
    sigma: float        # standard deviation for "normal"
    seed: int
    note: str = ""


# The workloads: the pages' worked example (square n = 3072, fp32) and its
# small PR-sized companion, a ragged fp32 shape, and the 16-bit tensor-core
# shapes (square 8192, a transformer-MLP-like rectangle and a skinny N = 64).
WORKLOADS = {
    w.name: w for w in [
        Workload("f32_256", 256, 256, 256, "f32", "uniform", 1.0, 14001,
                 "fp32 256^3, uniform[-1,1)"),
        Workload("f32_3072", 3072, 3072, 3072, "f32", "uniform", 1.0, 14002,
                 "fp32 3072^3, uniform[-1,1) (worked-example size)"),
        Workload("f32_ragged", 4097, 3001, 513, "f32", "normal", 1.0, 14003,
                 "fp32 4097x3001x513, normal(0,1): non-tile-multiple edges"),
        Workload("bf16_8192", 8192, 8192, 8192, "bf16", "normal", 1.0 / math.sqrt(8192), 14004,
                 "bf16 in, fp32 acc/out, 8192^3, normal(0,1/sqrt(K))"),
        Workload("f16_8192", 8192, 8192, 8192, "f16", "normal", 1.0 / math.sqrt(8192), 14004,
                 "fp16 in, fp32 acc/out, 8192^3, same draws as bf16_8192"),
        Workload("bf16_mlp", 16384, 11008, 4096, "bf16", "normal", 0.02, 14005,
                 "bf16 16384x11008x4096, normal(0,0.02)"),
        Workload("bf16_skinny", 16384, 64, 4096, "bf16", "normal", 0.02, 14006,
                 "bf16 16384x64x4096, normal(0,0.02): memory-bound side"),
    ]
}


def torch_dtype(dtype: str) -> torch.dtype:
    return _TORCH_DTYPES[dtype]


def draw(shape, dist: str, sigma: float, gen: torch.Generator) -> torch.Tensor:
    """One float32 draw on the CPU from ``gen``."""
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * sigma
    raise ValueError(f"unknown distribution {dist!r}")


def make(M: int, N: int, K: int, dtype: str = "f32", dist: str = "uniform",
         sigma: float = 1.0, seed: int = 0):
    """Returns (A, B): CPU tensors of shape (M, K) and (K, N) in ``dtype``."""
    g = torch.Generator().manual_seed(seed)
    A = draw((M, K), dist, sigma, g)
    B = draw((K, N), dist, sigma, g)
    td = _TORCH_DTYPES[dtype]
    if td != torch.float32:
        A, B = A.to(td), B.to(td)
    return A.contiguous(), B.contiguous()


def make_workload(name: str, M: int | None = None, N: int | None = None, K: int | None = None):
    """Inputs of a named workload; M/N/K override its shape (same recipe)."""
    w = WORKLOADS[name]
    return make(M or w.M, N or w.N, K or w.K, w.dtype, w.dist, w.sigma, w.seed)


def make_integer(M: int, N: int, K: int, r: int, dtype: str = "f32", seed: int = 0):
    """Integer-valued matrices with entries uniform in [-r, r] (exactly representable)."""
    g = torch.Generator().manual_seed(seed)
    A = torch.randint(-r, r + 1, (M, K), generator=g).to(torch.float32)
    B = torch.randint(-r, r + 1, (K, N), generator=g).to(torch.float32)
    td = _TORCH_DTYPES[dtype]
    return A.to(td).contiguous(), B.to(td).contiguous()


def host_view(x: torch.Tensor) -> np.ndarray:
    """The numpy view the oracle takes: float32 values or raw 16-bit patterns."""
    x = x.detach().cpu()
    if x.dtype == torch.float32:
        return x.numpy()
    if x.dtype in (torch.bfloat16, torch.float16):
        return x.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(f"unsupported dtype {x.dtype}")
