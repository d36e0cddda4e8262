"""GPU parity of the stream-K schedule (the *_ws entry points): tiles split
over several SMs, partial sums combined in a fixed order through the
workspace. Checked against the oracle, for run-to-run bit equality, and
against the data-parallel schedule within the bound."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import _lib, inputs

from gpu_util import make_workspace, oracle_check, run_abi

pytestmark = pytest.mark.gpu


def rup(x, m):
    return (x + m - 1) // m * m


# (M, N, K): just over one wave (the last tiles shared by every SM), about
# two waves (each tile split in two), a ragged tail; and products of few
# tiles, which take the small-tile kernel and no workspace.
F32_CASES = [(2560, 2048, 256), (3072, 3072, 3072), (4097, 3001, 513), (129, 257, 4000),
             (256, 256, 256), (1, 1, 1), (7, 300, 35)]


@pytest.mark.parametrize("M,N,K", F32_CASES)
@pytest.mark.parametrize("soft", [False, True])
def test_f32_streamk(oracle_mod, M, N, K, soft):
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M + 3 * N + 7 * K)
    lda = K + 1 if soft else rup(K, 4)
    ldb = N + 1 if soft else rup(N, 4)
    ws = make_workspace("f32", M, N, K)
    C1 = run_abi(A, B, lda=lda, ldb=ldb, ldc=N, workspace=ws)
    big = M * N * K > 2e9
    oracle_check(oracle_mod, A, B, C1, rows=np.arange(0, M, 97) if big else None)
    C2 = run_abi(A, B, lda=lda, ldb=ldb, ldc=N, workspace=ws)  # same workspace, next epoch
    assert torch.equal(C1, C2)


# (2000, 128, 4000): 16 tiles of 63 k-blocks over 63 workers of 16 -- ranges
# that start mid-tile, tiles with up to four contributors.
TC_CASES = [(16384, 64, 4096), (300, 100, 5000), (2000, 128, 777), (129, 65, 3000),
            (1, 8, 8), (500, 64, 64), (2000, 128, 4000)]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", TC_CASES)
def test_tensor_core_streamk(oracle_mod, dt, M, N, K):
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=M + N + K)
    ws = make_workspace(dt, M, N, K)
    C1 = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N, workspace=ws)
    oracle_check(oracle_mod, A, B, C1,
                 rows=np.arange(0, M, 61) if M * N * K > 2e9 else None)
    C2 = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N, workspace=ws)
    assert torch.equal(C1, C2)
    # software loader + stream-K
    C3 = run_abi(A, B, lda=K + 1, ldb=N + 1, ldc=N, a_off=1, workspace=ws)
    assert torch.equal(C1, C3)


# fp32 products split over a workspace need a wave of 128 x 256 tiles or
# more (fewer take the small-tile kernel): 160 tiles here
F32_SPLIT = (2560, 2048, 256)


def test_streamk_vs_data_parallel_within_bound(oracle_mod):
    M, N, K = F32_SPLIT
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=5)
    ws = make_workspace("f32", M, N, K)
    assert ws.numel() > 256
    C_sk = run_abi(A, B, workspace=ws)
    C_dp = run_abi(A, B)
    oracle_check(oracle_mod, A, B, C_sk)
    oracle_check(oracle_mod, A, B, C_dp)
    # exact on integer inputs, whatever the split
    Ai, Bi = inputs.make_integer(M, N, K, 3, "f32", seed=6)
    want = (Ai.double() @ Bi.double()).float()
    assert torch.equal(run_abi(Ai, Bi, workspace=ws), want)


def test_small_workspace_falls_back_to_data_parallel():
    A, B = inputs.make(*F32_SPLIT, "f32", "normal", 1.0, seed=7)
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    assert torch.equal(run_abi(A, B, workspace=small), run_abi(A, B))


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_streamk_expired_wait_reports_timeout(oracle_mod, dt):
    M, N, K = F32_SPLIT if dt == "f32" else (300, 100, 5000)
    A, B = inputs.make(M, N, K, dt, "uniform", 1.0, seed=8)
    ws = make_workspace(dt, M, N, K)
    s = torch.cuda.current_stream()
    assert g14.check_device_error(s.cuda_stream) == 0
    g14.debug_inject(1, 20_000_000)
    run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), workspace=ws, check_err=False)
    assert g14.check_device_error(s.cuda_stream) == _lib.GEMM14_ERR_TIMEOUT
    C = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), workspace=ws)
    oracle_check(oracle_mod, A, B, C)


def test_workspace_reused_across_shapes(oracle_mod):
    """One workspace, products of different shapes and dtypes in turn: the
    flag words sit at a fixed place, so stale partial sums never pose as flags."""
    need = max(g14.workspace_bytes(g14.GEMM14_DTYPE_F32, 2560, 2048, 256, 0),
               g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, 300, 100, 5000, 0))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    cases = [("f32", 2560, 2048, 256), ("bf16", 300, 100, 5000), ("f32", 256, 256, 256),
             ("bf16", 500, 64, 64), ("f32", 2560, 2048, 256)]
    for i, (dt, M, N, K) in enumerate(cases):
        A, B = inputs.make(M, N, K, dt, "uniform", 1.0, seed=40 + i)
        C = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), workspace=ws)
        oracle_check(oracle_mod, A, B, C)


# ------------------------------------------------------------------ CTA pairs (cluster workers)

PAIR_CASES = [(512, 512, 16384),    # 4 pair tiles: 4 workers per tile
              (2304, 2560, 8192),   # 90 tiles, 1.2 waves: every tile split
              (2304, 2560, 4100),   # the same with a ragged last k-block
              (4096, 4096, 1024),   # 256 tiles, 3.4 waves: the last 1.4 split
              (3000, 4100, 777)]    # 204 ragged tiles, 2.7 waves, ragged k


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", PAIR_CASES)
def test_pair_streamk(oracle_mod, dt, M, N, K):
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=M + 2 * N + K)
    st, plan = g14.plan(g14.GEMM14_DTYPE_BF16, M, N, K, 1 << 16, rup(K, 8), 1 << 16, rup(N, 8),
                        1 << 16, N, 152)
    assert plan.kernel == 3
    ws = make_workspace(dt, M, N, K)
    assert ws.numel() > 256, "this shape must take the stream-K schedule"
    C1 = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N, workspace=ws)
    oracle_check(oracle_mod, A, B, C1, rows=np.arange(0, M, 7) if M * N * K > 3e9 else None)
    C2 = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N, workspace=ws)  # next epoch
    assert torch.equal(C1, C2)


def test_pair_streamk_integer_exact_and_ex_modes(oracle_mod):
    """Integer inputs stay exact whatever the split; transposes and alpha /
    beta apply once, where a tile is finished."""
    from gpu_util import oracle_check_ex, run_ex
    M, N, K = 512, 520, 16384
    Ai, Bi = inputs.make_integer(M, N, K, 3, "bf16", seed=61)
    want = (Ai.double() @ Bi.double()).float()
    ws = make_workspace("bf16", M, N, K)
    assert torch.equal(run_abi(Ai, Bi, lda=rup(K, 8), ldb=rup(N, 8), workspace=ws), want)
    A, B = inputs.make(M, N, K, "bf16", "uniform", 0.05, seed=62)
    C0 = torch.from_numpy(np.random.default_rng(63).standard_normal((M, N)).astype(np.float32))
    for ta, tb in ((0, 0), (1, 0), (0, 1), (1, 1)):
        C = run_ex(A, B, ta, tb, -0.5, 2.0, C0, lda=rup(K if not ta else M, 8),
                   ldb=rup(N if not tb else K, 8), workspace=ws)
        oracle_check_ex(oracle_mod, A, B, C, ta, tb, -0.5, 2.0, C0)


def test_pair_streamk_expired_wait_reports_timeout(oracle_mod):
    M, N, K = 512, 512, 8192
    A, B = inputs.make(M, N, K, "bf16", "uniform", 1.0, seed=65)
    ws = make_workspace("bf16", M, N, K)
    s = torch.cuda.current_stream()
    assert g14.check_device_error(s.cuda_stream) == 0
    g14.debug_inject(1, 20_000_000)
    run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), workspace=ws, check_err=False)
    assert g14.check_device_error(s.cuda_stream) == _lib.GEMM14_ERR_TIMEOUT
    C = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), workspace=ws)
    oracle_check(oracle_mod, A, B, C)


def test_pair_hybrid_split_integer_exact():
    """More than two waves that are not whole: whole waves data-parallel, the
    last one and a half split; integer inputs stay exact, and the result is
    the bits of the next call (a new epoch on the same workspace)."""
    M, N, K = 4096, 4096, 1024
    Ai, Bi = inputs.make_integer(M, N, K, 4, "bf16", seed=66)
    want = (Ai.double() @ Bi.double()).float()
    ws = make_workspace("bf16", M, N, K)
    assert ws.numel() > 256
    C1 = run_abi(Ai, Bi, workspace=ws)
    assert torch.equal(C1, want)
    assert torch.equal(run_abi(Ai, Bi, workspace=ws), C1)
