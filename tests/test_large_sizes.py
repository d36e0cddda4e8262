"""GPU tests at sizes where C holds more than 2^31 elements (8.6 GB of fp32):
element offsets of C, row indices and TMA coordinates beyond int32 ranges
that the parity workloads never reach. Short k keeps them quick. Checked on
sampled rows (every column), sampled columns (every row) and random entries
against the oracle, and for NaN anywhere (C is NaN-filled first)."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import TOL

pytestmark = pytest.mark.gpu

ENTRY = {"f32": g14.gemm_f32, "bf16": g14.gemm_bf16_f32acc}


def check_sampled(oracle_mod, dt, A, B, c, seed):
    M, N = c.shape
    assert not torch.isnan(c).any().item()
    Ah, Bh = inputs.host_view(A), inputs.host_view(B)
    g = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, M - 1, M // 2], g.integers(0, M, 5)]))
    got = c[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref, refabs = oracle_mod.gemm(np.ascontiguousarray(Ah[rows]), Bh, dt)
    ok, worst = oracle_mod.within_bound(got, ref, refabs, TOL[dt])
    assert ok, ("rows", worst)
    cols = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 3)]))
    got = c[:, torch.from_numpy(cols).cuda()].cpu().numpy()
    ref, refabs = oracle_mod.gemm(Ah, np.ascontiguousarray(Bh[:, cols]), dt)
    ok, worst = oracle_mod.within_bound(got, ref, refabs, TOL[dt])
    assert ok, ("cols", worst)
    ri, ci = g.integers(0, M, 2048), g.integers(0, N, 2048)
    got = c[torch.from_numpy(ri).cuda(), torch.from_numpy(ci).cuda()].cpu().numpy()
    ref, refabs = oracle_mod.gemm_entries(Ah, Bh, ri, ci, dt)
    ok, worst = oracle_mod.within_bound(got, ref, refabs, TOL[dt])
    assert ok, ("entries", worst)


@pytest.mark.parametrize("dt,M,N,K,kernel", [
    ("bf16", 65536, 32770, 32, 3),      # CTA pairs, ragged last column tile
    ("bf16", (1 << 24) + 3, 128, 16, 2),  # one SM per tile, 2^24 + 3 rows
    ("f32", 65600, 32768, 16, 1),       # fp32 FFMA
])
def test_c_beyond_2_31_elements(oracle_mod, dt, M, N, K, kernel):
    assert M * N > 2 ** 31
    A, B = inputs.make(M, N, K, dt, "normal", 0.5, seed=M % 1000 + N + K)
    P = 1 << 20
    q = 4 if dt == "f32" else 8
    st, plan = g14.plan({"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16}[dt],
                        M, N, K, P, K, P, (N + q - 1) // q * q, P, N, 152)
    assert st == 0 and plan.kernel == kernel
    ldb = (N + q - 1) // q * q  # TMA-addressable B, so that the planned kernel runs
    a = A.cuda()
    b = torch.zeros(K, ldb, dtype=B.dtype, device="cuda")
    b[:, :N] = B.cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    ENTRY[dt](M, N, K, a.data_ptr(), K, b.data_ptr(), ldb, c.data_ptr(), N, s)
    assert g14.check_device_error(s) == 0
    check_sampled(oracle_mod, dt, A, B, c, seed=M + N)
    del c
    torch.cuda.empty_cache()
