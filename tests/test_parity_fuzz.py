"""Seeded random calls of gemm14_gemm_ex against the oracle: dtype, stored
transposes, shapes near tile edges, pitches and offsets that TMA can or
cannot read (one operand or both), alpha / beta with a C to accumulate into,
and a workspace that is absent, exactly what the call asks for (re-pitching,
transposed copies, stream-K) or only the stream-K part (the split runs on the
operands as stored). Each case is checked element by element on a sample of
rows (the oracle's product of those rows of op(A) with op(B)). The cases are
drawn from fixed seeds, so every run checks the same calls."""
import random

import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import DTYPE_CODE, oracle_check_ex, run_ex

pytestmark = pytest.mark.gpu

TILE_EDGES = [1, 7, 63, 64, 65, 127, 128, 129, 255, 256, 257, 383, 513]


def draw(seed):
    rng = random.Random(seed)
    dt = rng.choice(["f32", "bf16", "f16", "bf16"])

    def dim():
        r = rng.random()
        if r < 0.4:
            return rng.choice(TILE_EDGES)
        if r < 0.8:
            return rng.randint(1, 1200)
        if r < 0.95:
            return rng.randint(1200, 3000)
        return rng.randint(3000, 6000)

    M, N, K = dim(), dim(), dim()
    ta, tb = rng.randint(0, 1), rng.randint(0, 1)
    q = 4 if dt == "f32" else 8  # elements per 16 bytes

    def pitch(cols):
        # a pitch TMA can take, or any other
        return -(-cols // q) * q if rng.random() < 0.5 else cols + rng.randint(1, 9)

    a_cols, b_cols = (M if ta else K), (K if tb else N)
    lda, ldb = pitch(a_cols), pitch(b_cols)
    a_off = 0 if rng.random() < 0.6 else rng.randint(1, q - 1)
    b_off = 0 if rng.random() < 0.6 else rng.randint(1, q - 1)
    ldc = N + rng.choice([0, 0, 1, 3, 4])
    alpha, beta = rng.choice([(1.0, 0.0), (1.0, 0.0), (0.5, 0.0), (1.0, 1.0), (-2.0, 0.25)])
    ws_mode = rng.choice(["none", "exact", "split"])
    return dict(dt=dt, M=M, N=N, K=K, ta=ta, tb=tb, lda=lda, ldb=ldb, a_off=a_off,
                b_off=b_off, ldc=ldc, alpha=alpha, beta=beta, ws_mode=ws_mode)


def workspace_for(c):
    code = DTYPE_CODE[c["dt"]]
    eb = 4 if c["dt"] == "f32" else 2
    if c["ws_mode"] == "none":
        return None
    if c["ws_mode"] == "split":
        n = g14.workspace_bytes(code, c["M"], c["N"], c["K"], 0)
    else:
        # the alignment of run_ex's buffers: 256-byte bases plus the offsets
        base = 1 << 20
        n = g14.workspace_bytes_ex(code, c["ta"], c["tb"], c["M"], c["N"], c["K"],
                                   base + eb * c["a_off"], c["lda"], (base << 1) + eb * c["b_off"],
                                   c["ldb"], base << 2, c["ldc"])
    return torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("seed", range(160))
def test_fuzz_against_oracle(oracle_mod, seed):
    c = draw(20260 + seed)
    M, N, K = c["M"], c["N"], c["K"]
    A, B = inputs.make(M, N, K, c["dt"], "uniform", 1.0, seed=30000 + seed)
    C0 = (torch.rand(M, N, generator=torch.Generator().manual_seed(seed)) * 2 - 1
          if c["beta"] != 0.0 else None)
    ws = workspace_for(c)
    C = run_ex(A, B, c["ta"], c["tb"], c["alpha"], c["beta"], C0, lda=c["lda"], ldb=c["ldb"],
               ldc=c["ldc"], a_off=c["a_off"], b_off=c["b_off"], c_off=1, workspace=ws)
    rows = torch.tensor(sorted(random.Random(seed).sample(range(M), min(M, 24))))
    oracle_check_ex(oracle_mod, A[rows].contiguous(), B, C[rows].contiguous(), c["ta"], c["tb"],
                    c["alpha"], c["beta"], C0[rows].contiguous() if C0 is not None else None)


def draw_large(seed):
    """Output shapes of one to a few waves of the large tiles (the fp32 128 x 256
    kernel, the 16-bit one-SM and pair kernels), moderate k: stream-K splits,
    re-pitch copies and stored transposes on the large kernels."""
    rng = random.Random(seed)
    c = draw(seed)
    c["dt"] = rng.choice(["f32", "bf16", "f32", "f16"])
    c["M"], c["N"] = rng.randint(1500, 5000), rng.randint(1500, 5000)
    c["K"] = rng.choice([rng.randint(1, 96), rng.randint(96, 1500)])
    q = 4 if c["dt"] == "f32" else 8
    a_cols, b_cols = (c["M"] if c["ta"] else c["K"]), (c["K"] if c["tb"] else c["N"])
    c["lda"] = -(-a_cols // q) * q if rng.random() < 0.5 else a_cols + rng.randint(1, 9)
    c["ldb"] = -(-b_cols // q) * q if rng.random() < 0.5 else b_cols + rng.randint(1, 9)
    c["a_off"] = 0 if rng.random() < 0.6 else rng.randint(1, q - 1)
    c["b_off"] = 0 if rng.random() < 0.6 else rng.randint(1, q - 1)
    c["ldc"] = c["N"] + rng.choice([0, 1, 4])
    c["ws_mode"] = rng.choice(["none", "exact", "split", "split"])
    return c


@pytest.mark.parametrize("seed", range(40))
def test_fuzz_large_tiles_against_oracle(oracle_mod, seed):
    c = draw_large(50000 + seed)
    M, N, K = c["M"], c["N"], c["K"]
    A, B = inputs.make(M, N, K, c["dt"], "uniform", 1.0, seed=60000 + seed)
    C0 = (torch.rand(M, N, generator=torch.Generator().manual_seed(seed)) * 2 - 1
          if c["beta"] != 0.0 else None)
    ws = workspace_for(c)
    C = run_ex(A, B, c["ta"], c["tb"], c["alpha"], c["beta"], C0, lda=c["lda"], ldb=c["ldb"],
               ldc=c["ldc"], a_off=c["a_off"], b_off=c["b_off"], c_off=1, workspace=ws)
    rows = torch.tensor(sorted(random.Random(seed).sample(range(M), 24)))
    oracle_check_ex(oracle_mod, A[rows].contiguous(), B, C[rows].contiguous(), c["ta"], c["tb"],
                    c["alpha"], c["beta"], C0[rows].contiguous() if C0 is not None else None)
