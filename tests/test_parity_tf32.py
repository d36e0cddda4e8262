"""GPU parity of the fp32-input tensor-core modes (tcgen05 kind::tf32 on CTA
pairs) against the oracle:

- gemm_f32_3xtf32 (split hi/lo tf32 arithmetic): within the fp32 bound
  1e-5 (|A||B|) of the exact product of the fp32 inputs;
- gemm_tf32_f32acc (inputs read as tf32 by the tensor cores, i.e. with their
  13 low fraction bits dropped), two checks of different standing:
  * within 4e-3 (|A||B|) of the exact product of the fp32 inputs. This is the
    pin the page fixes: its format (fp32's exponent, 10 fraction bits) bounds
    each operand's change by 2^-10 relative, so each product by about
    2 * 2^-10, whatever the conversion's rounding;
  * within the fp32 bound of the exact product of the oracle-truncated
    inputs. The truncation is the hardware's reading of an fp32 operand, taken
    from a check on the GPU rather than from the page, so this tighter check
    is self-consistency: it shows the kernel applies the same reading
    everywhere (no term dropped, no operand swapped), not that the reading is
    the page's.

TF32 is the pages' tensor-core format for fp32 data (gpu-hpc-book ch.06,
"Tensor Cores" -> "TF32 (TensorFloat-32) 精度")."""
import random

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
             ldb=None, ldc=None, a_off=0, b_off=0, c_off=0, workspace=False):
    """C = alpha op(A) op(B) + beta C0 through gemm14_gemm_ex with a tf32 mode;
    pitches rounded to 4 floats by default (the tensor-core kernel). With
    workspace, the call gets the workspace gemm14_workspace_bytes_ex asks for
    (its K-major copies, lo parts and stream-K region), NaN-filled."""
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
    ws, ws_bytes = None, 0
    if workspace:
        ws_bytes = g14.workspace_bytes_ex(code, transa, transb, M, N, K,
                                          a.data_ptr() if As.numel() else 0, lda,
                                          b.data_ptr() if Bs.numel() else 0, ldb,
                                          cbuf.data_ptr() + 4 * c_off, ldc)
        ws = torch.full((max(ws_bytes, 16) // 4 + 1,), float("nan"), device="cuda")
    g14.gemm_ex(code, transa, transb, M, N, K, alpha, a.data_ptr() if As.numel() else 0, lda,
                b.data_ptr() if Bs.numel() else 0, ldb, beta, cbuf.data_ptr() + 4 * c_off, ldc,
                ws.data_ptr() if ws is not None else None, ws_bytes, s.cuda_stream)
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


@pytest.mark.parametrize("code", [TF32, X3])
def test_more_pair_tiles_than_clusters_every_storage(oracle_mod, code):
    """90 pair tiles of 256 x 256 (ragged at both edges) on 76 clusters of a
    152-SM GB300: 14 clusters run a second tile through the rings (TF32: 3 raw
    and 4 copy stages; 3xTF32: its own layout), each over 11 k-blocks, the last
    a quarter full. Every storage gives NN's bits; NN's sampled rows are
    checked against the oracle."""
    M, N, K = 2500, 2250, 328
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=2718 + code)
    C = run_mode(code, A, B)
    g = np.random.default_rng(code)
    rows = torch.tensor(sorted(set([0, 255, 256, 2303, 2304, M - 1]) |
                               set(g.integers(0, M, 26).tolist())))
    check(oracle_mod, A[rows].contiguous(), B, C[rows].contiguous(), TOL["f32"],
          rounded=code == TF32)
    for ta, tb in TRANS[1:]:
        assert torch.equal(run_mode(code, A, B, ta, tb), C), (ta, tb)


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


# ------------------------------------------------------------------ 3xTF32 split ahead of the call

def split_bytes(code, M, N, K, ta=0, tb=0):
    P = 1 << 16
    As_cols = M if ta else K
    Bs_cols = K if tb else N
    return g14.workspace_bytes_ex(code, ta, tb, M, N, K, P, rup(As_cols, 4), P, rup(Bs_cols, 4),
                                  P, N, 152)


@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (5, 7, 3), (255, 257, 33), (300, 520, 200),
                                   (513, 769, 1025), (64, 1000, 96)])
def test_3xtf32_split_meets_the_fp32_bound(oracle_mod, ta, tb, M, N, K):
    """With a workspace, 3xTF32 writes lo(A) and lo(B) (and K-major copies of
    operands stored otherwise) ahead of the product, which runs on the pair
    kernel as three k sums: within the fp32 bound in every storage, with the
    same bits in every storage (the same values reach the same MMAs)."""
    assert split_bytes(X3, M, N, K, ta, tb) >= (M + N) * rup(K, 4) * 4
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M * 3 + N + 7 * K + 5 * ta + tb)
    C = run_mode(X3, A, B, ta, tb, workspace=True)
    worst = check(oracle_mod, A, B, C, TOL["f32"], ta, tb)
    print(f"3xtf32 split {M}x{N}x{K} ta={ta} tb={tb}: worst {worst:.3g}")
    if (ta, tb) != (0, 1):
        assert torch.equal(C, run_mode(X3, A, B, 0, 1, workspace=True))


def fractional(rows, cols, seed):
    """i + j / 4096 with i, j in [-4, 4]: hi(x) + lo(x) = x with lo(x) a
    multiple of 2^-12, nonzero for most entries (e.g. 4 + 3 / 4096 has hi 4,
    lo 3 / 4096; 1 - 4 / 4096 is a tf32 value, lo 0)."""
    g = torch.Generator().manual_seed(seed)
    i = torch.randint(-4, 5, (rows, cols), generator=g)
    j = torch.randint(-4, 5, (rows, cols), generator=g)
    return (i.double() + j.double() / 4096).float()


@pytest.mark.parametrize("which", ["lo(A) hi(B)", "hi(A) lo(B)"])
def test_3xtf32_split_lo_terms_exact(which):
    """One operand with 2^-12 steps below its tf32 part, the other integer
    (lo = 0, so the dropped lo(A) lo(B) term is 0): every product and partial
    sum is a multiple of 2^-12 below 2^10, exact in fp32, so the split product
    must give A B bit for bit -- a missing or misplaced lo term (or one read
    at the wrong k) shows at once."""
    M, N, K = 300, 260, 64
    g = torch.Generator().manual_seed(41)
    if which == "lo(A) hi(B)":
        A = fractional(M, K, 42)
        B = torch.randint(-3, 4, (K, N), generator=g).float()
    else:
        A = torch.randint(-3, 4, (M, K), generator=g).float()
        B = fractional(K, N, 43)
    want = (A.double() @ B.double()).float()
    assert torch.equal(want.double(), A.double() @ B.double())
    for ta, tb in TRANS:
        C = run_mode(X3, A, B, ta, tb, workspace=True)
        assert torch.equal(C, want), (which, ta, tb)
    # the tf32 product misses the lo parts
    assert not torch.equal(run_mode(TF32, A, B, workspace=True), want)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (2.5, 0.0), (-1.0, 1.0), (0.5, -2.0)])
def test_3xtf32_split_alpha_beta(oracle_mod, alpha, beta):
    M, N, K = 300, 260, 190
    A, B = inputs.make(M, N, K, "f32", "normal", 0.1, seed=int(10 * alpha - 7 * beta) + 78)
    C0 = torch.from_numpy(np.random.default_rng(5).standard_normal((M, N)).astype(np.float32))
    for ldc in (N, N + 1):
        C = run_mode(X3, A, B, 0, 0, alpha, beta, C0, ldc=ldc, workspace=True)
        check(oracle_mod, A, B, C, TOL["f32"], 0, 0, alpha, beta, C0)


@pytest.mark.parametrize("M,N,K", [(512, 384, 1001), (512, 512, 8192), (2304, 2560, 1024)])
def test_3xtf32_split_over_clusters(oracle_mod, M, N, K):
    """Few tiles with 3 x L k-blocks: the stream-K split over clusters cuts
    across the three terms (a range may start in one term and end in
    another), within the fp32 bound; unaligned K pads each term's last k-block
    with TMA's zero fill."""
    P = 1 << 16
    L3 = 3 * ((K + 31) // 32)
    tiles = ((M + 255) // 256) * ((N + 255) // 256)
    lo = (M + N) * rup(K, 4) * 4
    # split: the stream-K slots (one 128 x 256 fp32 slot per SM) before the lo parts
    assert split_bytes(X3, M, N, K, 0, 1) >= lo + 152 * 128 * 256 * 4
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M + N + K)
    C = run_mode(X3, A, B, 0, 1, workspace=True)
    worst = check(oracle_mod, A, B, C, TOL["f32"], 0, 1)
    print(f"3xtf32 split {M}x{N}x{K} ({tiles} tiles, {L3} k-blocks): worst {worst:.3g}")


def test_3xtf32_split_full_size_3072_sampled(oracle_mod):
    """The fp32 3072^3 workload in 3xTF32 with its workspace (B transposed,
    lo parts): sampled rows and random entries against the oracle."""
    A, B = inputs.make_workload("f32_3072")
    C = run_mode(X3, A, B, workspace=True)
    Cg = C.numpy()
    assert not np.isnan(Cg).any()
    Ah, Bh = A.numpy(), B.numpy()
    g = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, 3071], g.integers(0, 3072, 14)]))
    ref, refabs = oracle_mod.gemm(np.ascontiguousarray(Ah[rows]), Bh)
    ok, w1 = oracle_mod.within_bound(Cg[rows], ref, refabs, TOL["f32"])
    assert ok, w1
    ri, ci = g.integers(0, 3072, 4096), g.integers(0, 3072, 4096)
    ref, refabs = oracle_mod.gemm_entries(Ah, Bh, ri, ci)
    ok, w2 = oracle_mod.within_bound(Cg[ri, ci], ref, refabs, TOL["f32"])
    assert ok, w2
    print(f"3xtf32 split 3072^3: worst {max(w1, w2):.3g}")


@pytest.mark.parametrize("code", [TF32, X3])
@pytest.mark.parametrize("M,N,K", [(1000, 777, 130), (300, 520, 64)])
def test_pair_kernel_tf32_keeps_padding(oracle_mod, code, M, N, K):
    """TF32 and split 3xTF32 on the pair kernel (A stored M x K, B N x K, a
    workspace) write C through its TMA-store epilogue: with a padded pitch the
    columns past N and the memory past the last row keep their NaN."""
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M + N + K + code)
    As, Bs = stored(A, 0), stored(B, 1)
    lda = ldb = rup(K, 4)
    ldc = rup(N, 4) + 8
    _ab, a = to_device_padded(As, lda)
    _bb, b = to_device_padded(Bs, ldb)
    cbuf = torch.full((M * ldc + 4096,), float("nan"), device="cuda")
    need = g14.workspace_bytes_ex(code, 0, 1, M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb,
                                  cbuf.data_ptr(), ldc)
    ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    g14.gemm_ex(code, 0, 1, M, N, K, 1.0, a.data_ptr(), lda, b.data_ptr(), ldb, 0.0,
                cbuf.data_ptr(), ldc, ws.data_ptr(), need, s)
    assert g14.check_device_error(s) == 0
    torch.cuda.synchronize()
    full = cbuf.cpu()
    rows = full[:M * ldc].view(M, ldc)
    assert torch.isnan(rows[:, N:]).all()
    assert torch.isnan(full[M * ldc:]).all()
    check(oracle_mod, A, B, rows[:, :N].contiguous(), TOL["f32"], 0, 0,
          rounded=code == TF32)


TF32_EDGES = [1, 7, 31, 32, 33, 127, 128, 129, 255, 256, 257, 511, 513]


def draw_tf32(seed):
    """One random call of a tf32 mode: sizes near tile and k-block edges or
    anywhere up to 3000, a stored transpose of either operand, alpha / beta,
    and a workspace or none (the split-ahead pair kernel or the converter
    kernel)."""
    rng = random.Random(seed)

    def dim():
        r = rng.random()
        if r < 0.35:
            return rng.choice(TF32_EDGES)
        return rng.randint(1, 1500) if r < 0.9 else rng.randint(1500, 3000)

    return dict(code=rng.choice([TF32, X3]), M=dim(), N=dim(), K=dim(), ta=rng.randint(0, 1),
                tb=rng.randint(0, 1),
                ab=rng.choice([(1.0, 0.0), (1.0, 0.0), (0.5, 0.0), (1.0, 1.0), (-2.0, 0.25)]),
                workspace=rng.random() < 0.5)


def run_tf32_case(oracle_mod, seed):
    c = draw_tf32(seed)
    M, N, K, code = c["M"], c["N"], c["K"], c["code"]
    alpha, beta = c["ab"]
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=seed)
    C0 = (torch.rand(M, N, generator=torch.Generator().manual_seed(seed)) * 2 - 1
          if beta != 0.0 else None)
    C = run_mode(code, A, B, c["ta"], c["tb"], alpha, beta, C0, workspace=c["workspace"])
    rows = torch.tensor(sorted(random.Random(seed).sample(range(M), min(M, 24))))
    check(oracle_mod, A[rows].contiguous(), B, C[rows].contiguous(), TOL["f32"], c["ta"],
          c["tb"], alpha, beta, C0[rows].contiguous() if C0 is not None else None,
          rounded=code == TF32)


@pytest.mark.parametrize("seed", range(48))
def test_tf32_modes_fuzz_against_oracle(oracle_mod, seed):
    """48 seeded random calls of the tf32 modes, each on sampled rows against
    the oracle: 3xTF32 within the fp32 bound of the exact product, TF32 within
    it of the product of the truncated inputs."""
    run_tf32_case(oracle_mod, 70000 + seed)
