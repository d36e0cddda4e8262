"""GPU parity of the fp32-input tensor-core modes (tcgen05 kind::tf32 on CTA
pairs) against the oracle:

- gemm_f32_3xtf32 (split hi/lo tf32 arithmetic): within the fp32 bound
  1e-5 (|A||B|) of the exact product of the fp32 inputs;
- gemm_tf32_f32acc (inputs read as tf32 by the tensor cores, i.e. with their
  13 low fraction bits dropped): within the fp32 bound of the exact product of
  the oracle-truncated inputs, and within 4e-3 (|A||B|) of the exact product
  of the fp32 ones (two truncations of under 2^-10 per product, doubled).

TF32 is the pages' tensor-core format for fp32 data (gpu-hpc-book ch.06,
"Tensor Cores")."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import TOL, oracle_check_ex, run_abi, run_ex, stored, to_device_padded

pytestmark = pytest.mark.gpu

X3, TF32 = g14.GEMM14_DTYPE_F32_3XTF32, g14.GEMM14_DTYPE_TF32
TOL_TF32 = 4e-3
TRANS = [(0, 0), (1, 0), (0, 1), (1, 1)]


def rup(x, m):
    return (x + m - 1) // m * m


def run_mode(code, A, B, transa=0, transb=0, alpha=1.0, beta=0.0, C0=None, lda=None,
             ldb=None, ldc=None, a_off=0, b_off=0, c_off=0):
    """C = alpha op(A) op(B) + beta C0 through gemm14_gemm_ex with a tf32 mode;
    pitches rounded to 4 floats by default (the tensor-core kernel)."""
    M, K = A.shape
    N = B.shape[1]
    As, Bs = stored(A, transa), stored(B, transb)
    lda = lda or rup(max(As.shape[1], 1), 4)
    ldb = ldb or rup(max(Bs.shape[1], 1), 4)
    ldc = ldc or max(N, 1)
    _ab, a = to_device_padded(As, lda, a_off)
    _bb, b = to_device_padded(Bs, ldb, b_off)
    cbuf = torch.full((c_off + max(M, 1) * ldc + 16,), float("nan"), device="cuda")
    if C0 is not None:
        cbuf[c_off:c_off + M * ldc].view(M, ldc)[:, :N].copy_(C0.cuda())
    s = torch.cuda.current_stream()
    g14.gemm_ex(code, transa, transb, M, N, K, alpha, a.data_ptr() if As.numel() else 0, lda,
                b.data_ptr() if Bs.numel() else 0, ldb, beta, cbuf.data_ptr() + 4 * c_off, ldc,
                None, 0, s.cuda_stream)
    assert g14.check_device_error(s.cuda_stream) == 0
    torch.cuda.synchronize()
    return cbuf[c_off:c_off + M * ldc].view(M, ldc)[:, :N].cpu()


def check(oracle_mod, A, B, C, tol, transa=0, transb=0, alpha=1.0, beta=0.0, C0=None,
          rounded=False):
    """C against the oracle's extended product of the stored fp32 matrices,
    or (rounded) of their tf32 values, the oracle's truncation."""
    As = stored(A, transa).numpy()
    Bs = stored(B, transb).numpy()
    if rounded:
        As, Bs = oracle_mod.truncate_tf32(As), oracle_mod.truncate_tf32(Bs)
    c0 = C0.numpy() if C0 is not None else None
    ref, refabs = oracle_mod.gemm_ex(As, Bs, "f32", bool(transa), bool(transb), alpha, beta, c0)
    Cg = C.numpy()
    ok, worst = oracle_mod.within_bound(Cg, ref, refabs, tol)
    if not ok:
        diff = np.abs(Cg.astype(np.float64) - ref) - tol * refabs
        bad = np.argwhere(~(diff <= 0))
        i, j = bad[0]
        raise AssertionError(f"{len(bad)} out of bound; first ({i},{j}) gpu={Cg[i, j]!r} "
                             f"ref={ref[i, j]!r} abs={refabs[i, j]!r}; worst={worst:.3g}")
    return worst


SHAPES = [(1, 1, 1), (5, 7, 3), (128, 128, 32), (255, 257, 33), (300, 520, 200),
          (513, 769, 1025), (64, 1000, 96)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_3xtf32_meets_the_fp32_bound(oracle_mod, M, N, K):
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M * 3 + N + 7 * K)
    C = run_mode(X3, A, B)
    worst = check(oracle_mod, A, B, C, TOL["f32"])
    print(f"3xtf32 {M}x{N}x{K}: worst {worst:.3g}")


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_tf32_is_the_product_of_truncated_inputs(oracle_mod, M, N, K):
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=M + 5 * N + K)
    C = run_mode(TF32, A, B)
    check(oracle_mod, A, B, C, TOL["f32"], rounded=True)
    check(oracle_mod, A, B, C, TOL_TF32)


@pytest.mark.parametrize("code", [X3, TF32])
@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (129, 65, 130), (7, 300, 35)])
def test_transposes(oracle_mod, code, ta, tb, M, N, K):
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=11 * ta + 3 * tb + M + K)
    C = run_mode(code, A, B, ta, tb)
    if code == X3:
        check(oracle_mod, A, B, C, TOL["f32"], ta, tb)
    else:
        check(oracle_mod, A, B, C, TOL["f32"], ta, tb, rounded=True)
    # every storage feeds the same values to the same MMAs in the same order
    assert torch.equal(C, run_mode(code, A, B))


@pytest.mark.parametrize("code", [X3, TF32])
@pytest.mark.parametrize("alpha,beta", [(2.5, 0.0), (-1.0, 1.0), (0.5, -2.0)])
def test_alpha_beta(oracle_mod, code, alpha, beta):
    M, N, K = 300, 260, 190
    A, B = inputs.make(M, N, K, "f32", "normal", 0.1, seed=int(10 * alpha - 7 * beta) + 77)
    C0 = torch.from_numpy(np.random.default_rng(4).standard_normal((M, N)).astype(np.float32))
    for ldc in (N, N + 1):
        C = run_mode(code, A, B, 0, 0, alpha, beta, C0, ldc=ldc)
        check(oracle_mod, A, B, C, TOL["f32"], 0, 0, alpha, beta, C0, rounded=code == TF32)


@pytest.mark.parametrize("code", [X3, TF32])
def test_integer_inputs_exact(code):
    """Integers of at most 11 significant bits are tf32 values (lo = 0), and
    their sums stay below 2^24: both modes give the int64 product bit for bit,
    in every storage."""
    M, N, K = 300, 260, 190
    A, B = inputs.make_integer(M, N, K, 8, dtype="f32", seed=5)
    want = (A.to(torch.int64) @ B.to(torch.int64)).to(torch.float32)
    for ta, tb in TRANS:
        assert torch.equal(run_mode(code, A, B, ta, tb), want), (ta, tb)


def test_3xtf32_recovers_what_tf32_loses(oracle_mod):
    """Inputs with bits below tf32's 10 fraction bits: the tf32 mode misses the
    fp32 bound against the unrounded inputs, the split mode meets it."""
    M, N, K = 256, 256, 512
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=99)
    C1 = run_mode(TF32, A, B)
    C3 = run_mode(X3, A, B)
    ref, refabs = oracle_mod.gemm(A.numpy(), B.numpy())
    ok1, worst1 = oracle_mod.within_bound(C1.numpy(), ref, refabs, TOL["f32"])
    ok3, worst3 = oracle_mod.within_bound(C3.numpy(), ref, refabs, TOL["f32"])
    assert not ok1 and ok3, (worst1, worst3)
    assert worst3 < worst1 / 50


@pytest.mark.parametrize("code", [X3, TF32])
def test_unaligned_operands_run_the_fp32_kernel(code):
    """Pitches TMA cannot take: the call runs gemm_f32's kernel, exact fp32
    products, the very bits of gemm_f32 with the same operands."""
    M, N, K = 300, 200, 150
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=8)
    C = run_mode(code, A, B, lda=K + 1, ldb=N + 3, ldc=N, a_off=1)
    P = run_abi(A, B, lda=K + 1, ldb=N + 3, ldc=N, a_off=1)
    assert torch.equal(C, P)


@pytest.mark.parametrize("code", [X3, TF32])
def test_nan_propagates_to_its_row(code):
    M, N, K = 260, 300, 64
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=12)
    A[17, 5] = float("nan")
    C = run_mode(code, A, B)
    assert torch.isnan(C[17]).all()
    assert not torch.isnan(C[torch.arange(M) != 17]).any()


def test_entry_points_match_gemm_ex():
    M, N, K = 260, 300, 72
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=13)
    a, b = A.cuda(), B.cuda()
    for fn, code in ((g14.gemm_f32_3xtf32, X3), (g14.gemm_tf32_f32acc, TF32)):
        c = torch.full((M, N), float("nan"), device="cuda")
        fn(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N,
           torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert torch.equal(c.cpu(), run_mode(code, A, B, lda=K, ldb=N))


def test_tensor_level_fp32_mode(oracle_mod):
    M, N, K = 300, 310, 120
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=14)
    out = torch.empty(M, N, device="cuda")
    g14.gemm_into(A.cuda(), B.cuda().t().contiguous().t(), out, fp32_mode="3xtf32")
    torch.cuda.synchronize()
    check(oracle_mod, A, B, out.cpu(), TOL["f32"])


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
def test_3xtf32_full_size_3072_sampled(oracle_mod, ta, tb):
    """The fp32 3072^3 workload in 3xTF32: sampled rows, sampled columns and
    random entries against the oracle's dot products, fp32 bound."""
    A, B = inputs.make_workload("f32_3072")
    C = run_mode(X3, A, B, ta, tb)
    Cg = C.numpy()
    assert not np.isnan(Cg).any()
    Ah, Bh = A.numpy(), B.numpy()
    g = np.random.default_rng(3 + ta)
    rows = np.unique(np.concatenate([[0, 3071], g.integers(0, 3072, 14)]))
    ref, refabs = oracle_mod.gemm(np.ascontiguousarray(Ah[rows]), Bh)
    ok, w1 = oracle_mod.within_bound(Cg[rows], ref, refabs, TOL["f32"])
    assert ok, w1
    cols = np.unique(np.concatenate([[0, 3071], g.integers(0, 3072, 6)]))
    ref, refabs = oracle_mod.gemm(Ah, np.ascontiguousarray(Bh[:, cols]))
    ok, w2 = oracle_mod.within_bound(Cg[:, cols], ref, refabs, TOL["f32"])
    assert ok, w2
    ri, ci = g.integers(0, 3072, 4096), g.integers(0, 3072, 4096)
    ref, refabs = oracle_mod.gemm_entries(Ah, Bh, ri, ci)
    ok, w3 = oracle_mod.within_bound(Cg[ri, ci], ref, refabs, TOL["f32"])
    assert ok, w3
    print(f"3xtf32 3072^3 ta={ta} tb={tb}: worst {max(w1, w2, w3):.3g}")


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (2.5, 0.0), (-1.0, 1.0)])
def test_tf32_nt_on_the_pair_kernel_matches_the_converter_kernel(oracle_mod, alpha, beta):
    """TF32 with A stored M x K and B stored N x K runs the 16-bit pair
    kernel's mainloop with kind::tf32 MMAs (plan kernel 5): the same tf32
    values in the same MMAs as the converter kernel on NN storage, so the same
    bits, alpha and beta included."""
    M, N, K = 300, 520, 200
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=31)
    C0 = torch.from_numpy(np.random.default_rng(6).standard_normal((M, N)).astype(np.float32))
    P = 1 << 16
    st, plan = g14.plan_ex(TF32, 0, 1, M, N, K, P, K, P, K, P, N, 152)
    assert st == 0 and plan.kernel == 5
    c_nt = run_mode(TF32, A, B, 0, 1, alpha, beta, C0)
    c_nn = run_mode(TF32, A, B, 0, 0, alpha, beta, C0)
    assert torch.equal(c_nt, c_nn)
    check(oracle_mod, A, B, c_nt, TOL["f32"], 0, 1, alpha, beta, C0, rounded=True)


def test_tf32_nt_split_over_clusters(oracle_mod):
    """Few tiles with long k on plan kernel 5 with a workspace: the stream-K
    split over clusters (4 tiles, 256 k-blocks: 16 workers), within the fp32
    bound of the product of the truncated inputs."""
    M, N, K = 512, 512, 8192
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=32)
    Bs = B.t().contiguous()
    a, b = A.cuda(), Bs.cuda()
    need = g14.workspace_bytes_ex(TF32, 0, 1, M, N, K, a.data_ptr(), K, b.data_ptr(), K,
                                  a.data_ptr(), N)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    c = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    g14.gemm_ex(TF32, 0, 1, M, N, K, 1.0, a.data_ptr(), K, b.data_ptr(), K, 0.0, c.data_ptr(), N,
                ws.data_ptr(), need, s)
    assert g14.check_device_error(s) == 0
    check(oracle_mod, A, B, c.cpu(), TOL["f32"], rounded=True)
