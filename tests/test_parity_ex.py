"""GPU parity of gemm14_gemm_ex, C = alpha * op(A) op(B) + beta * C, with A
and B stored transposed or not, on every kernel, loader and schedule, against
the oracle's extended product (which reads the same stored matrices).

The accumulate form with transposable operands is the pages' wgmma account
(gpu-hpc-book ch.06, "Tensor Cores" / "wgmma": D = A*B + D, A and B
optionally transposed, D scaled by 0 or 1), taken for general alpha, beta.
"""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import (DTYPE_CODE, TOL, make_workspace, oracle_check_ex, run_abi, run_ex,
                      stored)

pytestmark = pytest.mark.gpu

TRANS = [(0, 0), (1, 0), (0, 1), (1, 1)]


def rup(x, m):
    return (x + m - 1) // m * m


def pitches(M, N, K, ta, tb, mult):
    """Row pitches of the stored A and B rounded up to `mult` elements."""
    return rup(M if ta else K, mult), rup(K if tb else N, mult)


def odd_pitch(cols):
    return cols + 1 if (cols + 1) % 4 else cols + 2


# ------------------------------------------------------------------ fp32

# small products (64 x 64 tiles) and one with 17 x 7 tiles of 128 x 256 (the
# large kernel's stored-transpose layouts)
F32_SHAPES = [(3, 5, 7), (129, 257, 33), (300, 520, 200), (1000, 70, 513), (2049, 1537, 97)]


@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", F32_SHAPES)
def test_f32_transposes(oracle_mod, M, N, K, ta, tb):
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M + 5 * N + 11 * K + ta + 2 * tb)
    lda, ldb = pitches(M, N, K, ta, tb, 4)
    C = run_ex(A, B, ta, tb, lda=lda, ldb=ldb, ldc=rup(N, 4))
    oracle_check_ex(oracle_mod, A, B, C, ta, tb)
    # the cp.async loader fills the same shared-memory tiles whatever the
    # storage, so every storage gives the plain product's very bits
    C_nn = run_abi(A, B, lda=rup(K, 4), ldb=rup(N, 4), ldc=rup(N, 4))
    assert torch.equal(C, C_nn)
    # odd pitches and 4-byte offsets
    C2 = run_ex(A, B, ta, tb, lda=odd_pitch(M if ta else K), ldb=odd_pitch(K if tb else N),
                ldc=N + 1, a_off=1, b_off=3, c_off=1)
    assert torch.equal(C2, C_nn)


@pytest.mark.parametrize("ta", [0, 1])
def test_f32_b_stored_nk_transposed_in_shared_memory(oracle_mod, ta):
    """B stored N x K reaches the 128 x 256 kernel through TMA as K-major tiles,
    which the CTA transposes in shared memory stage by stage into two
    alternating buffers. Several tiles per CTA, a ragged k tail (K = 333) and
    ragged edges; the FMAs then run in the order of B stored K x N, so the
    product has that call's very bits. Rows sampled against the oracle."""
    M, N, K = 4100, 2600, 333
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=91 + ta)
    lda, ldb = pitches(M, N, K, ta, 1, 4)
    C = run_ex(A, B, ta, 1, lda=lda, ldb=ldb, ldc=rup(N, 4))
    C_nn = run_ex(A, B, 0, 0, lda=rup(K, 4), ldb=rup(N, 4), ldc=rup(N, 4))
    assert torch.equal(C, C_nn)
    rows = torch.arange(0, M, 41)
    oracle_check_ex(oracle_mod, A[rows].contiguous(), B, C[rows].contiguous())


# ------------------------------------------------------------------ bf16 / fp16

TC_SHAPES = [(5, 7, 3), (128, 64, 64), (129, 65, 130), (200, 300, 100), (257, 129, 1000),
             (384, 1000, 200)]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", TC_SHAPES)
def test_tensor_core_transposes_tma(oracle_mod, dt, M, N, K, ta, tb):
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=3 * M + N + K + 7 * ta + tb)
    lda, ldb = pitches(M, N, K, ta, tb, 8)
    C = run_ex(A, B, ta, tb, lda=lda, ldb=ldb, ldc=N)
    oracle_check_ex(oracle_mod, A, B, C, ta, tb)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", [(5, 7, 3), (200, 300, 100), (129, 65, 130)])
def test_tensor_core_transposes_soft_loader(oracle_mod, dt, M, N, K, ta, tb):
    A, B = inputs.make(M, N, K, dt, "uniform", 1.0, seed=M + N + K + 5 * ta + tb)
    # odd pitches and 2-byte offsets break TMA's rules -> software loader
    C = run_ex(A, B, ta, tb, lda=(M if ta else K) + 1, ldb=(K if tb else N) + 1, ldc=N + 3,
               a_off=1, b_off=3, c_off=1)
    oracle_check_ex(oracle_mod, A, B, C, ta, tb)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("ta,tb", TRANS[1:])
def test_tensor_core_transposes_one_sm_wide(oracle_mod, dt, ta, tb):
    """The one-SM kernel's 256-column tiles with transposed operands (pairs
    forbidden), against the oracle and against the pair kernel."""
    M, N, K = 384, 1000, 200
    A, B = inputs.make(M, N, K, dt, "normal", 0.1, seed=77 + ta + 2 * tb)
    lda, ldb = pitches(M, N, K, ta, tb, 8)
    prev = g14.set_pair_kernel(False)
    try:
        C1 = run_ex(A, B, ta, tb, lda=lda, ldb=ldb)
    finally:
        g14.set_pair_kernel(prev)
    oracle_check_ex(oracle_mod, A, B, C1, ta, tb)
    C2 = run_ex(A, B, ta, tb, lda=lda, ldb=ldb)
    oracle_check_ex(oracle_mod, A, B, C2, ta, tb)


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(200, 300, 100), (129, 65, 130), (37, 29, 53)])
def test_integer_exact_every_storage(dt, M, N, K):
    """Integer matrices, integer C0 and alpha = 2, beta = -1: every sum,
    product and update is exact in fp32, so every storage, kernel and loader
    must give the int64 result bit for bit."""
    A, B = inputs.make_integer(M, N, K, 4, dtype=dt, seed=M + N + K)
    C0 = torch.from_numpy(np.random.default_rng(M * N).integers(-64, 65, (M, N)).astype(np.float32))
    want = 2 * (A.to(torch.int64) @ B.to(torch.int64)) - C0.to(torch.int64)
    mult = 4 if dt == "f32" else 8
    for ta, tb in TRANS:
        lda, ldb = pitches(M, N, K, ta, tb, mult)
        C = run_ex(A, B, ta, tb, 2.0, -1.0, C0, lda=lda, ldb=ldb, ldc=N)
        assert torch.equal(C.to(torch.int64), want), (ta, tb)
        C = run_ex(A, B, ta, tb, 2.0, -1.0, C0, lda=(M if ta else K) + 1,
                   ldb=(K if tb else N) + 1, ldc=N + 1, a_off=1)
        assert torch.equal(C.to(torch.int64), want), (ta, tb, "unaligned")


# ------------------------------------------------------------------ alpha, beta

AB = [(2.5, 0.0), (-1.0, 1.0), (0.5, -2.0), (1.0, 1.0), (-0.75, 0.25)]


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("alpha,beta", AB)
@pytest.mark.parametrize("vec", [True, False])
def test_alpha_beta(oracle_mod, dt, alpha, beta, vec):
    M, N, K = 300, 260, 190
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=int(100 * alpha + 10 * beta) + 1000)
    C0 = torch.from_numpy(np.random.default_rng(5).standard_normal((M, N)).astype(np.float32))
    mult = 4 if dt == "f32" else 8
    ldc = rup(N, 4) if vec else N + 1
    C = run_ex(A, B, 0, 0, alpha, beta, C0, lda=rup(K, mult), ldb=rup(N, mult), ldc=ldc)
    oracle_check_ex(oracle_mod, A, B, C, 0, 0, alpha, beta, C0)
    if beta == 0.0:
        # C = alpha * (the plain product): one fp32 multiply per element
        P = run_abi(A, B, lda=rup(K, mult), ldb=rup(N, mult), ldc=ldc)
        assert torch.equal(C, alpha * P)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("ta,tb", TRANS)
def test_alpha_beta_stream_k(oracle_mod, dt, ta, tb):
    """alpha, beta applied once, after the stream-K fixup (tiles split over
    many SMs), with transposed storage; repeatable bit for bit."""
    M, N, K = (2560, 2048, 256) if dt == "f32" else (300, 100, 5000)
    A, B = inputs.make(M, N, K, dt, "uniform", 1.0 / K ** 0.5, seed=9 + ta + 2 * tb)
    C0 = torch.from_numpy(np.random.default_rng(6).uniform(-1, 1, (M, N)).astype(np.float32))
    ws = make_workspace(dt, M, N, K)
    assert ws.numel() > 256, "this shape must take the stream-K schedule"
    mult = 4 if dt == "f32" else 8
    lda, ldb = pitches(M, N, K, ta, tb, mult)
    C1 = run_ex(A, B, ta, tb, -1.5, 0.5, C0, lda=lda, ldb=ldb, workspace=ws)
    oracle_check_ex(oracle_mod, A, B, C1, ta, tb, -1.5, 0.5, C0)
    C2 = run_ex(A, B, ta, tb, -1.5, 0.5, C0, lda=lda, ldb=ldb, workspace=ws)
    assert torch.equal(C1, C2)


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("beta", [0.0, 1.0, -3.0, 0.1])
def test_alpha_zero_reads_neither_operand(dt, beta):
    """alpha == 0: C = beta * C; A and B are not read (they hold NaN)."""
    M, N, K = 70, 90, 50
    td = inputs.torch_dtype(dt)
    A = torch.full((M, K), float("nan"), dtype=td)
    B = torch.full((K, N), float("nan"), dtype=td)
    C0 = torch.from_numpy(np.random.default_rng(7).standard_normal((M, N)).astype(np.float32))
    for ldc in (N, N + 1):
        C = run_ex(A, B, 0, 1, 0.0, beta, C0, ldc=ldc)
        assert torch.equal(C, beta * C0 if beta != 0.0 else torch.zeros_like(C0)), ldc


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_empty_inner_dimension_scales_c(dt):
    M, N = 33, 45
    td = inputs.torch_dtype(dt)
    C0 = torch.from_numpy(np.random.default_rng(8).standard_normal((M, N)).astype(np.float32))
    A, B = torch.zeros((M, 0), dtype=td), torch.zeros((0, N), dtype=td)
    assert torch.equal(run_ex(A, B, 0, 0, 3.0, 2.0, C0), 2.0 * C0)
    assert torch.equal(run_ex(A, B, 1, 1, 3.0, 0.0, C0), torch.zeros_like(C0))


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_identity_call_matches_plain_entry(dt):
    """alpha = 1, beta = 0, no transposes: the plain entry point's bits."""
    M, N, K = 517, 389, 300
    A, B = inputs.make(M, N, K, dt, "normal", 0.05, seed=12)
    mult = 4 if dt == "f32" else 8
    C1 = run_ex(A, B, lda=rup(K, mult), ldb=rup(N, mult))
    C2 = run_abi(A, B, lda=rup(K, mult), ldb=rup(N, mult))
    assert torch.equal(C1, C2)


def test_invalid_transpose_flags():
    p = torch.zeros(64, device="cuda")
    for ta, tb in ((2, 0), (0, -1)):
        st = g14.gemm_ex(DTYPE_CODE["f32"], ta, tb, 4, 4, 4, 1.0, p.data_ptr(), 4, p.data_ptr(),
                         4, 0.0, p.data_ptr(), 4, check=False)
        assert st == 1


def test_tensor_level_views(oracle_mod):
    """gemm_into recognises transposed views and passes alpha, beta."""
    M, N, K = 260, 300, 130
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.1, seed=31)
    a_t = A.t().contiguous().cuda()   # stored K x M
    b_t = B.t().contiguous().cuda()   # stored N x K
    C0 = torch.from_numpy(np.random.default_rng(9).standard_normal((M, N)).astype(np.float32))
    out = C0.cuda()
    g14.gemm_into(a_t.t(), b_t.t(), out, alpha=0.5, beta=-1.0)
    torch.cuda.synchronize()
    oracle_check_ex(oracle_mod, A, B, out.cpu(), 1, 1, 0.5, -1.0, C0)


# ------------------------------------------------------------------ full size

@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1)])
def test_bf16_8192_transposed_sampled(oracle_mod, ta, tb):
    """The 8192^3 bf16 product with a transposed operand, on the pair kernel:
    sampled rows and random entries against the oracle's dot products."""
    A, B = inputs.make_workload("bf16_8192")
    M, K = A.shape
    N = B.shape[1]
    C = run_ex(A, B, ta, tb, 1.0, 0.0)
    Cg = C.numpy()
    assert not np.isnan(Cg).any()
    Ah, Bh = inputs.host_view(A), inputs.host_view(B)
    g = np.random.default_rng(ta + 2 * tb)
    rows = np.unique(np.concatenate([[0, M - 1], g.integers(0, M, 6)]))
    ref, refabs = oracle_mod.gemm(np.ascontiguousarray(Ah[rows]), Bh, "bf16")
    ok, worst = oracle_mod.within_bound(Cg[rows], ref, refabs, TOL["bf16"])
    assert ok, worst
    ri, ci = g.integers(0, M, 2048), g.integers(0, N, 2048)
    ref, refabs = oracle_mod.gemm_entries(Ah, Bh, ri, ci, "bf16")
    ok, worst = oracle_mod.within_bound(Cg[ri, ci], ref, refabs, TOL["bf16"])
    assert ok, worst
    # the stored transpose the kernel read is the one the test made
    assert stored(A, ta).shape == ((K, M) if ta else (M, K))
