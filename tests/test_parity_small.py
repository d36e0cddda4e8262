"""GPU parity at sizes the oracle checks element by element: several tiles,
ragged tails, both fp32 loaders, every tensor-core tile width, exact
integer sums, structured matrices that expose layout bugs, and the
degenerate sizes. All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import oracle_check, run_abi, to_device_padded

pytestmark = pytest.mark.gpu


def rup(x, m):
    return (x + m - 1) // m * m


F32_SHAPES = [(1, 1, 1), (3, 5, 7), (17, 33, 5), (128, 256, 32), (129, 257, 33),
              (300, 520, 200), (64, 1000, 96), (1000, 70, 513), (513, 769, 1025)]


@pytest.mark.parametrize("M,N,K", F32_SHAPES)
def test_f32_tma_loader(oracle_mod, M, N, K):
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M * 7 + N * 3 + K)
    # pitches rounded to 4 elements -> TMA loader and vector stores
    C = run_abi(A, B, lda=rup(K, 4), ldb=rup(N, 4), ldc=rup(N, 4))
    oracle_check(oracle_mod, A, B, C)


@pytest.mark.parametrize("M,N,K", F32_SHAPES)
def test_f32_cpasync_loader(oracle_mod, M, N, K):
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=M + N + K)
    # odd pitches and 4-byte offsets break TMA's rules -> cp.async loader, scalar stores
    C = run_abi(A, B, lda=K + 1 if (K + 1) % 4 else K + 2, ldb=N + 1 if (N + 1) % 4 else N + 2,
                ldc=N + 1, a_off=1, b_off=3, c_off=1)
    oracle_check(oracle_mod, A, B, C)


TC_SHAPES = [(1, 1, 1), (5, 7, 3), (128, 64, 64), (128, 128, 64), (128, 256, 64),
             (200, 300, 100), (257, 129, 1000), (129, 65, 130), (512, 512, 512), (384, 1000, 200)]


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", TC_SHAPES)
def test_tensor_core(oracle_mod, dt, M, N, K):
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / max(K, 1) ** 0.5, seed=M * 5 + N + K)
    C = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N)
    oracle_check(oracle_mod, A, B, C)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_tensor_core_padded_pitches(oracle_mod, dt):
    A, B = inputs.make(300, 200, 150, dt, "uniform", 1.0, seed=3)
    C = run_abi(A, B, lda=160, ldb=264, ldc=203, a_off=8, b_off=16, c_off=3)
    oracle_check(oracle_mod, A, B, C)


@pytest.mark.parametrize("pair,M,N,K", [(False, 300, 200, 150), (False, 129, 36, 64),
                                        (False, 1000, 777, 130), (False, 300, 201, 64),
                                        (True, 300, 200, 150), (True, 1000, 777, 130),
                                        (True, 1000, 779, 130)])
def test_tensor_core_tma_store_keeps_padding(oracle_mod, pair, M, N, K):
    """The TMA-store epilogue writes 32 x 32 blocks that the TMA unit clips at
    M rows, but only at 16-byte granularity at N columns: with a padded pitch
    the columns past N (N not a multiple of 4 included), and the memory past
    the last row, keep the NaN they were filled with; C is within the bound."""
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=M + 3 * N + K)
    lda, ldb, ldc = rup(K, 8), rup(N, 8), rup(N, 4) + 8
    prev = g14.set_pair_kernel(pair)
    try:
        st, plan = g14.plan(g14.GEMM14_DTYPE_BF16, M, N, K, 1 << 16, lda, 1 << 16, ldb,
                            1 << 16, ldc, 152)
        assert st == 0 and plan.kernel == (3 if pair else 2) and plan.vec_store == 1
        _abuf, a = to_device_padded(A, lda)
        _bbuf, b = to_device_padded(B, ldb)
        cbuf = torch.full((M * ldc + 4096,), float("nan"), device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        g14.gemm_bf16_f32acc(M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb, cbuf.data_ptr(),
                             ldc, s)
        assert g14.check_device_error(s) == 0
        torch.cuda.synchronize()
    finally:
        g14.set_pair_kernel(prev)
    full = cbuf.cpu()
    rows = full[:M * ldc].view(M, ldc)
    assert torch.isnan(rows[:, N:]).all()
    assert torch.isnan(full[M * ldc:]).all()
    assert not torch.isnan(rows[:, :N]).any()
    oracle_check(oracle_mod, A, B, rows[:, :N].contiguous())


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (190, 300, 257), (128, 64, 130), (300, 129, 77)])
def test_tensor_core_software_loader(oracle_mod, dt, M, N, K):
    """Pitches that are not multiples of 8 elements and 2-byte offsets: the
    software loader must give the same results as the TMA path."""
    A, B = inputs.make(M, N, K, dt, "normal", 0.25, seed=M + 2 * N + 3 * K)
    C = run_abi(A, B, lda=K + 1, ldb=N + 3, ldc=N + 1, a_off=1, b_off=5, c_off=2)
    oracle_check(oracle_mod, A, B, C)
    C_tma = run_abi(A, B, lda=rup(K, 8), ldb=rup(N, 8), ldc=N)
    assert torch.equal(C, C_tma)


# ------------------------------------------------------------------ exact results

def test_f32_integer_exact():
    """Entries in [-3, 3], K = 3072: every partial sum is an integer below 2^24,
    so any summation order gives the exact result bit for bit."""
    A, B = inputs.make_integer(300, 520, 3072, 3, "f32", seed=21)
    C = run_abi(A, B)
    assert torch.equal(C, (A.double() @ B.double()).float())
    C = run_abi(A, B, lda=3073, ldb=521, ldc=521)  # cp.async loader
    assert torch.equal(C, (A.double() @ B.double()).float())


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_tensor_core_integer_exact(dt):
    """Entries in [-4, 4], K = 8192: partial sums stay below 2^24 -> exact."""
    A, B = inputs.make_integer(256, 320, 8192, 4, dt, seed=22)
    C = run_abi(A, B)
    assert torch.equal(C, (A.double() @ B.double()).float())


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_permutation_and_identity(dt):
    """P @ B must return the rows of B permuted and A @ I must return A, bit
    for bit: a wrong tile index, swizzle or descriptor shows here."""
    td = inputs.torch_dtype(dt)
    g = torch.Generator().manual_seed(23)
    K = 320
    perm = torch.randperm(K, generator=g)
    P = torch.zeros(K, K)
    P[torch.arange(K), perm] = 1
    B = (torch.rand(K, 264, generator=g) * 2 - 1).to(td)
    C = run_abi(P.to(td), B)
    assert torch.equal(C, B.float()[perm])
    A = (torch.rand(200, K, generator=g) * 2 - 1).to(td)
    C = run_abi(A, torch.eye(K).to(td))
    assert torch.equal(C, A.float())


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_rank_one_closed_form(dt):
    td = inputs.torch_dtype(dt)
    M, N, K = 260, 300, 96
    a = (torch.arange(M) % 7 + 1).float()
    b = (torch.arange(N) % 5 + 1).float()
    A = a[:, None].expand(M, K).contiguous().to(td)
    B = b[None, :].expand(K, N).contiguous().to(td)
    C = run_abi(A, B)
    assert torch.equal(C, K * torch.outer(a, b))


def test_f16_subnormal_inputs(oracle_mod):
    """fp16 subnormals are values, not zeros, on the tensor-core path."""
    g = torch.Generator().manual_seed(24)
    A = (torch.randint(1, 1024, (128, 64), generator=g) * 2.0 ** -24).half()  # all subnormal
    B = torch.randint(-8, 9, (64, 128), generator=g).float().half()
    C = run_abi(A, B)
    assert torch.equal(C, (A.double() @ B.double()).float())
    oracle_check(oracle_mod, A, B, C)


# ------------------------------------------------------------------ degenerate sizes

@pytest.mark.parametrize("dt", ["f32", "bf16", "f16"])
def test_k_zero_zeroes_c(dt):
    td = inputs.torch_dtype(dt)
    A = torch.zeros(7, 0, dtype=td)
    B = torch.zeros(0, 9, dtype=td)
    C = run_abi(A, B, lda=8, ldb=16, ldc=11)
    assert C.shape == (7, 9) and torch.all(C == 0)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_empty_m_or_n(dt):
    td = inputs.torch_dtype(dt)
    assert run_abi(torch.zeros(0, 8, dtype=td), torch.zeros(8, 8, dtype=td)).shape == (0, 8)
    C = run_abi(torch.ones(8, 8, dtype=td), torch.zeros(8, 0, dtype=td), ldb=8, ldc=8)
    assert C.shape == (8, 0)


def test_nan_propagates_along_its_row():
    A, B = inputs.make(130, 260, 64, "f32", "uniform", 1.0, seed=25)
    A[5, 10] = float("nan")
    C = run_abi(A, B)
    assert torch.isnan(C[5]).all()
    assert not torch.isnan(C[torch.arange(130) != 5]).any()


# ------------------------------------------------------------------ streams, API, determinism

def test_non_default_stream_and_repeatability():
    A, B = inputs.make(700, 900, 333, "f32", "normal", 1.0, seed=26)
    s = torch.cuda.Stream()
    C1 = run_abi(A, B, stream=s)
    C2 = run_abi(A, B)
    assert torch.equal(C1, C2)  # run-to-run deterministic (no atomics)


def test_tensor_api_cuda_and_host(oracle_mod):
    """The tensor API runs the workspace entry (this shape takes the stream-K
    split, so its last bits may differ from the unsplit ABI call): within the
    bound, and the host path gives the device path's bits (same plan)."""
    A, B = inputs.make(257, 300, 190, "bf16", "normal", 0.1, seed=27)
    got_dev = g14.gemm(A.cuda(), B.cuda())
    torch.cuda.synchronize()
    oracle_check(oracle_mod, A, B, got_dev.cpu())
    got_host = g14.gemm(A, B)  # host tensors: copied in, computed, copied back
    assert got_host.device.type == "cpu" and torch.equal(got_host, got_dev.cpu())


def test_device_error_word_is_clear_after_good_calls():
    A, B = inputs.make(256, 256, 256, "f32", "uniform", 1.0, seed=28)
    run_abi(A, B, check_err=False)
    assert g14.check_device_error(None) == 0


# ------------------------------------------------------------------ CTA-pair vs one-SM kernel

@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N,K", [(129, 129, 64), (256, 256, 64), (300, 520, 200),
                                   (1000, 777, 1000), (2048, 1536, 640)])
def test_pair_kernel_matches_single_sm_kernel(oracle_mod, dt, M, N, K):
    """The 256 x 256 CTA-pair kernel and the 128-row one-SM kernel accumulate in
    the same order: bit-identical results, both within the oracle's bound."""
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=M + N + K)
    ldb = rup(N, 8)
    st, plan = g14.plan(g14.GEMM14_DTYPE_BF16, M, N, K, 1 << 16, rup(K, 8), 1 << 16, ldb,
                        1 << 16, N, 152)
    assert plan.kernel == 3
    C_pair = run_abi(A, B, lda=rup(K, 8), ldb=ldb, ldc=N)
    prev = g14.set_pair_kernel(False)
    try:
        C_one = run_abi(A, B, lda=rup(K, 8), ldb=ldb, ldc=N)
    finally:
        g14.set_pair_kernel(prev)
    oracle_check(oracle_mod, A, B, C_pair)
    assert torch.equal(C_pair, C_one)


@pytest.mark.parametrize("pair,M,N,K", [(True, 2304, 2557, 8192), (False, 512, 125, 8192)])
def test_split_products_keep_padding(oracle_mod, pair, M, N, K):
    """Stream-K variants of both 16-bit kernels (the tile owners store through
    the TMA-store epilogue) with N not a multiple of 4 and a padded pitch:
    the columns past N and the memory past the last row keep their NaN; C is
    within the bound on sampled rows."""
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=M + N + K)
    lda, ldb, ldc = rup(K, 8), rup(N, 8), rup(N, 4) + 8
    prev = g14.set_pair_kernel(pair)
    try:
        st, plan = g14.plan(g14.GEMM14_DTYPE_BF16, M, N, K, 1 << 16, lda, 1 << 16, ldb,
                            1 << 16, ldc, 152)
        assert st == 0 and plan.kernel == (3 if pair else 2) and plan.vec_store == 1
        need = g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, M, N, K, 0)
        assert need > 0  # split
        _abuf, a = to_device_padded(A, lda)
        _bbuf, b = to_device_padded(B, ldb)
        cbuf = torch.full((M * ldc + 4096,), float("nan"), device="cuda")
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        s = torch.cuda.current_stream().cuda_stream
        g14.gemm_bf16_f32acc_ws(M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb, cbuf.data_ptr(),
                                ldc, ws.data_ptr(), need, s)
        assert g14.check_device_error(s) == 0
        torch.cuda.synchronize()
    finally:
        g14.set_pair_kernel(prev)
    full = cbuf.cpu()
    rows = full[:M * ldc].view(M, ldc)
    assert torch.isnan(rows[:, N:]).all()
    assert torch.isnan(full[M * ldc:]).all()
    assert not torch.isnan(rows[:, :N]).any()
    sample = np.unique(np.concatenate([[0, M - 1], np.arange(1, M, 97)]))
    oracle_check(oracle_mod, A, B, rows[:, :N].contiguous(), rows=sample)
