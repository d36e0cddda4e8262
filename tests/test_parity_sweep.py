"""GPU parity over a seeded sample of small ragged sizes, M, N, K each from
{1, 2, 3, 15, 16, 17, 31, 33, 127, 129, 255, 257}: one below, at and above
the warp, k-group and tile boundaries of every kernel. Each product runs
through the plain entry point (data-parallel) and through the workspace entry
point with the workspace gemm14_workspace_bytes_ex asks for (stream-K and
operand copies where the policy takes them), against the oracle element by
element. All calls go through the C ABI."""
import itertools

import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import oracle_check, run_abi

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 3, 15, 16, 17, 31, 33, 127, 129, 255, 257]
CODES = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16,
         "f16": g14.GEMM14_DTYPE_F16}


def sample(n, seed):
    g = np.random.default_rng(seed)
    every = list(itertools.product(SIZES, SIZES, SIZES))
    picks = g.choice(len(every), size=n, replace=False)
    return [every[i] for i in sorted(picks)]


def rup(x, m):
    return (x + m - 1) // m * m


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_ragged_size_sweep(oracle_mod, dt):
    q = 4 if dt == "f32" else 8
    for M, N, K in sample(40, seed={"f32": 1, "bf16": 2, "f16": 3}[dt]):
        A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=M * 65536 + N * 256 + K)
        lda, ldb, ldc = rup(K, q), rup(N, q), N
        C = run_abi(A, B, lda=lda, ldb=ldb, ldc=ldc)
        oracle_check(oracle_mod, A, B, C)
        need = g14.workspace_bytes_ex(CODES[dt], 0, 0, M, N, K, 1 << 16, lda, 1 << 16, ldb,
                                      1 << 16, ldc, 0)
        if need:
            ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
            Cw = run_abi(A, B, lda=lda, ldb=ldb, ldc=ldc, workspace=ws)
            oracle_check(oracle_mod, A, B, Cw)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_ragged_size_sweep_unaligned(oracle_mod, dt):
    """The same sizes with pitches and offsets TMA cannot take: the software
    loaders, and with a workspace the re-pitched copies on the TMA loaders."""
    for M, N, K in sample(16, seed={"f32": 4, "bf16": 5}[dt]):
        A, B = inputs.make(M, N, K, dt, "uniform", 1.0, seed=M + 7 * N + 13 * K)
        lda, ldb, ldc = K + 1, N + 3, N + 1
        C = run_abi(A, B, lda=lda, ldb=ldb, ldc=ldc, a_off=1, b_off=1, c_off=1)
        oracle_check(oracle_mod, A, B, C)
        eb = 4 if dt == "f32" else 2
        need = g14.workspace_bytes_ex(CODES[dt], 0, 0, M, N, K, (1 << 16) + eb, lda,
                                      (1 << 16) + eb, ldb, (1 << 16) + 4, ldc, 0)
        if need:
            ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
            Cw = run_abi(A, B, lda=lda, ldb=ldb, ldc=ldc, a_off=1, b_off=1, c_off=1,
                         workspace=ws)
            oracle_check(oracle_mod, A, B, Cw)
