"""GPU parity of the small-tile paths against the oracle, element by element:

- fp32 products with few 128 x 256 tiles run on the 64 x 64-tile kernel whose
  k range is split over a cluster of 2-8 CTAs and added up through
  distributed shared memory (plan kernel 6);
- 16-bit products whose 64-row tiles fit in one wave run on the one-SM
  tensor-core kernel with 64-row tiles (M = 64 MMAs, plan kernel 2 with
  bm = 64), data-parallel or split over a caller workspace (stream-K).

Each shape is chosen so that the plan is the one named (asserted first), and
checked against the fp64 oracle on the same (rounded) inputs within the
bounds 1e-5 (|A||B|) for fp32 and 4e-3 (|A||B|) for 16-bit inputs.
"""
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import make_workspace, oracle_check, oracle_check_ex, run_abi, run_ex

pytestmark = pytest.mark.gpu

F32, BF16 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16
P = 1 << 16  # an aligned stand-in address for the host-only planner


def rup(x, m):
    return (x + m - 1) // m * m


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def f32_plan(M, N, K, lda=None, ldb=None):
    st, p = g14.plan(F32, M, N, K, P, lda or K, P, ldb or N, P, N, sms())
    assert st == 0
    return p


# ------------------------------------------------------------------ fp32, 64 x 64 tiles

# (M, N, K): split 8 (the 256^3 workload), 4, 2 and 1; a ragged edge in
# every dimension; K below one k-block; K not a multiple of the split's share
F32_SMALL = [(256, 256, 256), (512, 512, 512), (256, 256, 64), (1024, 1024, 1024),
             (300, 190, 333), (65, 129, 17), (1, 1, 1), (7, 300, 4099), (129, 64, 96)]


@pytest.mark.parametrize("M,N,K", F32_SMALL)
def test_f32_small_kernel(oracle_mod, M, N, K):
    p = f32_plan(M, N, K)
    assert p.kernel == 6
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=3 * M + 5 * N + K)
    C = run_abi(A, B)
    oracle_check(oracle_mod, A, B, C)
    # run-to-run deterministic: the cluster adds its partial tiles in rank order
    assert torch.equal(C, run_abi(A, B))


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (300, 190, 333), (65, 129, 17)])
def test_f32_small_kernel_any_pitch_and_offset(oracle_mod, M, N, K):
    """Pitches that are not multiples of 4 floats and 4-byte offsets take the
    4-byte loader, which fills the same shared-memory tiles: the same bits."""
    assert f32_plan(M, N, K, lda=K + 1, ldb=N + 3).loader == 2
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=M + N + K)
    C = run_abi(A, B, lda=K + 1, ldb=N + 3, ldc=N + 1, a_off=1, b_off=3, c_off=1)
    oracle_check(oracle_mod, A, B, C)
    assert torch.equal(C, run_abi(A, B, lda=rup(K, 4), ldb=rup(N, 4), ldc=rup(N, 4)))


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-1.5, 0.5)])
def test_f32_small_kernel_transposes_and_epilogue(oracle_mod, ta, tb, alpha, beta):
    M, N, K = 200, 300, 250
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=ta + 2 * tb + 7)
    C0 = torch.arange(M * N, dtype=torch.float32).reshape(M, N) / (M * N) - 0.5
    C = run_ex(A, B, ta, tb, alpha, beta, C0 if beta else None)
    oracle_check_ex(oracle_mod, A, B, C, ta, tb, alpha, beta, C0 if beta else None)
    if alpha == 1.0 and beta == 0.0:
        # every storage lands in the same tiles and sums in the same order
        assert torch.equal(C, run_abi(A, B))


def test_f32_small_kernel_integer_exact():
    """Integer entries in [-3, 3]: every partial sum (each CTA's, and the sum
    of the cluster's partial tiles) is an integer below 2^24, so the result is
    exact bit for bit."""
    M, N, K = 256, 256, 4096
    assert f32_plan(M, N, K).kernel == 6
    g = torch.Generator().manual_seed(5)
    A = torch.randint(-3, 4, (M, K), generator=g).float()
    B = torch.randint(-3, 4, (K, N), generator=g).float()
    C = run_abi(A, B)
    assert torch.equal(C, (A.double() @ B.double()).float())


def test_f32_few_tiles_with_a_workspace_above_2_30_flop(oracle_mod):
    """1024^3 (32 tiles of 128 x 256): the plain call takes the small-tile
    kernel, a call with the workspace it asks for the large kernel split over
    every SM; both within the bound."""
    M, N, K = 1024, 1024, 1024
    assert f32_plan(M, N, K).kernel == 6
    ws = make_workspace("f32", M, N, K)
    assert ws.numel() == 768 + sms() * 128 * 256 * 4
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=15)
    C_ws = run_abi(A, B, workspace=ws)
    oracle_check(oracle_mod, A, B, C_ws)
    oracle_check(oracle_mod, A, B, run_abi(A, B))
    # a workspace too small for the split: the small-tile kernel, as without one
    short = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    assert torch.equal(run_abi(A, B, workspace=short), run_abi(A, B))


def test_f32_small_kernel_workspace_entry_is_the_same():
    """The workspace entry point plans the same kernel (it needs none) and
    gives the plain entry point's bits."""
    M, N, K = 256, 256, 256
    A, B = inputs.make_workload("f32_256")
    ws = make_workspace("f32", M, N, K)
    assert torch.equal(run_abi(A, B, workspace=ws), run_abi(A, B))


# ------------------------------------------------------------------ 16-bit, 64-row tiles

def tc_plan(M, N, K, lda=None, ldb=None):
    st, p = g14.plan(BF16, M, N, K, P, lda or rup(K, 8), P, ldb or rup(N, 8), P, N, sms())
    assert st == 0
    return p


# (M, N, K): the skinny workload's tile shape at a size the oracle checks in
# full, ragged M and N, every tile width (N <= 64, <= 128, <= 256 with M <=
# 128), k not a multiple of the 64-deep k-block
BM64 = [(4096, 64, 4096), (1000, 64, 1000), (2050, 100, 300), (64, 64, 64), (1, 1, 1),
        (100, 200, 77), (127, 256, 520), (3000, 7, 129)]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", BM64)
def test_tensor_core_64_row_tiles(oracle_mod, dt, M, N, K):
    p = tc_plan(M, N, K)
    assert p.kernel == 2 and p.bm == 64
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=M + 3 * N + K)
    C = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N)
    oracle_check(oracle_mod, A, B, C)


@pytest.mark.parametrize("M,N,K", [(1000, 64, 1000), (100, 200, 77), (3000, 7, 129)])
def test_tensor_core_64_row_tiles_pitch_and_software_loader(oracle_mod, M, N, K):
    """Odd pitches and 2-byte offsets (the software loader), C with a pitch
    that is not a multiple of 4 (direct stores): the TMA path's bits."""
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.25, seed=M + N)
    C = run_abi(A, B, lda=K + 1, ldb=N + 3, ldc=N + 1, a_off=1, b_off=5, c_off=2)
    oracle_check(oracle_mod, A, B, C)
    assert torch.equal(C, run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N))


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1), (1, 1)])
def test_tensor_core_64_row_tiles_transposes(oracle_mod, ta, tb):
    M, N, K = 1000, 100, 600
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.05, seed=ta + 2 * tb)
    C0 = torch.ones(M, N)
    C = run_ex(A, B, ta, tb, -2.0, 0.5, C0)
    oracle_check_ex(oracle_mod, A, B, C, ta, tb, -2.0, 0.5, C0)
    C1 = run_ex(A, B, ta, tb)
    assert torch.equal(C1, run_ex(A, B))


@pytest.mark.parametrize("M,N,K", [(1024, 64, 4096), (128, 64, 4096), (600, 128, 8192),
                                   (2000, 64, 2048)])
def test_tensor_core_64_row_tiles_stream_k(oracle_mod, M, N, K):
    """Few 64-row tiles split over a caller workspace: workers' partial sums
    in 64 x BN slots, added by each tile's owner in worker order."""
    p = tc_plan(M, N, K)
    assert p.kernel == 2 and p.bm == 64
    assert g14.workspace_bytes(BF16, M, N, K, sms()) > 0
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=M + N + K)
    ws = make_workspace("bf16", M, N, K)
    C1 = run_abi(A, B, workspace=ws)
    oracle_check(oracle_mod, A, B, C1)
    assert torch.equal(C1, run_abi(A, B, workspace=ws))


def test_largest_one_wave_skinny_product_on_64_row_tiles(oracle_mod):
    """9728 x 64 x 4096: 76 tiles of 128 rows, so 152 tiles of 64 rows -- one
    full wave, the largest skinny product that takes them; every 16th row in
    full against the oracle."""
    M, N, K = 9728, 64, 4096
    p = tc_plan(M, N, K)
    assert p.kernel == 2 and p.bm == 64 and p.tiles == 152
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.02, seed=14)
    C = run_abi(A, B)
    oracle_check(oracle_mod, A, B, C, rows=list(range(0, M, 16)) + [M - 1])
    # one row tile more: 128-row tiles
    assert tc_plan(M + 128, N, K).bm == 128
