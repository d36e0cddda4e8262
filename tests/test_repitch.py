"""GPU tests of re-pitching: an operand TMA cannot read (base or row pitch not
a multiple of 16 bytes), given a workspace of gemm14_workspace_bytes_ex bytes,
is copied into it with a 16-byte pitch and the product runs on the TMA
loaders. The result must have the bits of the same product on operands
stored with 16-byte pitches from the start (same kernels, same schedule), and
meet the oracle's bound."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import TOL, oracle_check, oracle_check_ex, stored, to_device_padded

pytestmark = pytest.mark.gpu

CODE = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16, "f16": g14.GEMM14_DTYPE_F16,
        "tf32": g14.GEMM14_DTYPE_TF32, "3xtf32": g14.GEMM14_DTYPE_F32_3XTF32}


def rup(x, m):
    return (x + m - 1) // m * m


def run(mode, A, B, ta=0, tb=0, lda=None, ldb=None, a_off=0, workspace=True, alpha=1.0,
        beta=0.0, C0=None, ws_bytes=None):
    """C = alpha op(A) op(B) + beta C0 through gemm14_gemm_ex on stored
    operands with the given pitches and element offsets, with a workspace of
    exactly workspace_bytes_ex bytes (or ws_bytes, or none). Returns (C, ws)."""
    M, K = A.shape
    N = B.shape[1]
    As, Bs = stored(A, ta), stored(B, tb)
    lda = lda or As.shape[1]
    ldb = ldb or Bs.shape[1]
    _ab, a = to_device_padded(As, lda, a_off)
    _bb, b = to_device_padded(Bs, ldb, 0)
    c = torch.full((M, N), float("nan"), device="cuda") if C0 is None else C0.clone().cuda()
    code = CODE[mode]
    s = torch.cuda.current_stream().cuda_stream
    need = g14.workspace_bytes_ex(code, ta, tb, M, N, K, a.data_ptr(), lda, b.data_ptr(), ldb,
                                  c.data_ptr(), N)
    nb = need if ws_bytes is None else ws_bytes
    ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device="cuda") if workspace else None
    g14.gemm_ex(code, ta, tb, M, N, K, alpha, a.data_ptr(), lda, b.data_ptr(), ldb, beta,
                c.data_ptr(), N, ws.data_ptr() if ws is not None else None,
                nb if ws is not None else 0, s)
    assert g14.check_device_error(s) == 0
    torch.cuda.synchronize()
    return c.cpu(), need


@pytest.mark.parametrize("mode,M,N,K", [("f32", 4097, 3001, 513), ("f32", 2049, 2047, 301),
                                        ("bf16", 1000, 777, 1000), ("f16", 300, 1001, 259),
                                        ("3xtf32", 1000, 777, 301), ("tf32", 513, 700, 129)])
def test_unaligned_pitches_give_the_aligned_bits(oracle_mod, mode, M, N, K):
    dt = "f32" if mode in ("f32", "tf32", "3xtf32") else mode
    A, B = inputs.make(M, N, K, dt, "normal", 0.5, seed=M + N + K)
    C1, need = run(mode, A, B)                       # pitches K and N: not 16-byte multiples
    q = 4 if dt == "f32" else 8
    assert need > 0
    C2, _ = run(mode, A, B, lda=rup(K, q), ldb=rup(N, q))  # 16-byte pitches from the start
    assert torch.equal(C1, C2)
    if mode == "tf32":
        As, Bs = oracle_mod.truncate_tf32(A.numpy()), oracle_mod.truncate_tf32(B.numpy())
        ref, refabs = oracle_mod.gemm(As, Bs)
        ok, worst = oracle_mod.within_bound(C1.numpy(), ref, refabs, TOL["f32"])
        assert ok, worst
    else:
        oracle_check(oracle_mod, A, B, C1, rows=np.arange(0, M, 7))


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1), (1, 1)])
def test_stored_transposes_and_misaligned_bases(oracle_mod, ta, tb):
    """Stored transposes with odd pitches and A's base 4 bytes off: the same
    bits as 16-byte-aligned storage, alpha and beta included."""
    M, N, K = 2049, 1537, 333  # 17 x 7 tiles of 128 x 256: the large kernel
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=11 * ta + tb)
    C0 = torch.from_numpy(np.random.default_rng(3).standard_normal((M, N)).astype(np.float32))
    C1, need = run("f32", A, B, ta, tb, a_off=1, alpha=-1.5, beta=0.5, C0=C0)
    assert need > 0
    As, Bs = stored(A, ta), stored(B, tb)
    C2, _ = run("f32", A, B, ta, tb, lda=rup(As.shape[1], 4), ldb=rup(Bs.shape[1], 4),
                alpha=-1.5, beta=0.5, C0=C0)
    assert torch.equal(C1, C2)
    oracle_check_ex(oracle_mod, A, B, C1, ta, tb, -1.5, 0.5, C0)


def test_too_small_a_workspace_reads_operands_as_they_are(oracle_mod):
    """One byte short of workspace_bytes_ex: no copy; the stream-K schedule on
    the element-wise loader, the bits of a workspace of the shape-only size."""
    M, N, K = 2560, 2048, 150  # 160 tiles: split over every SM
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=5)
    _, need = run("f32", A, B)
    sk = g14.workspace_bytes(CODE["f32"], M, N, K, 0)
    assert 0 < sk < need - 1
    C_short, _ = run("f32", A, B, ws_bytes=need - 1)
    C_sk, _ = run("f32", A, B, ws_bytes=sk)
    assert torch.equal(C_short, C_sk)
    oracle_check(oracle_mod, A, B, C_short)


def test_one_workspace_for_split_and_repitched_products(oracle_mod):
    """A workspace reused by stream-K products and re-pitched ones in turn:
    the copies never land on the flag words (integer data: exact)."""
    g14.load()
    cases = [(2560, 2048, 256, 256, 2048), (4097, 3001, 513, 513, 3001),
             (2560, 2048, 256, 256, 2048), (2049, 2047, 301, 301, 2047)]
    need = 0
    for M, N, K, lda, ldb in cases:
        need = max(need, g14.workspace_bytes_ex(CODE["f32"], 0, 0, M, N, K, 1 << 20, lda, 1 << 20,
                                                ldb, 1 << 20, N, 0))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for i, (M, N, K, lda, ldb) in enumerate(cases * 2):
        A, B = inputs.make_integer(M, N, K, 3, "f32", seed=20 + i)
        _ab, a = to_device_padded(A, lda)
        _bb, b = to_device_padded(B, ldb)
        c = torch.full((M, N), float("nan"), device="cuda")
        g14.gemm_ex(CODE["f32"], 0, 0, M, N, K, 1.0, a.data_ptr(), lda, b.data_ptr(), ldb, 0.0,
                    c.data_ptr(), N, ws.data_ptr(), need, s)
        assert g14.check_device_error(s) == 0
        assert torch.equal(c.cpu().double(), A.double() @ B.double()), (M, N, K)


def test_tensor_level_call_repitches():
    """gemm_into sizes its workspace for the operands it gets: an odd-pitched
    bf16 view takes the TMA path (the bits of a contiguous copy)."""
    M, N, K = 1000, 777, 1000
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.05, seed=9)
    big = torch.zeros(M, K + 3, dtype=torch.bfloat16, device="cuda")
    big[:, :K] = A.cuda()
    a_view = big[:, :K]                      # pitch K + 3 = 1003 elements
    out1 = torch.empty(M, N, device="cuda")
    g14.gemm_into(a_view, B.cuda(), out1)
    a_pad = torch.zeros(M, rup(K, 8), dtype=torch.bfloat16, device="cuda")
    a_pad[:, :K] = A.cuda()
    out2 = torch.empty(M, N, device="cuda")
    g14.gemm_into(a_pad[:, :K], B.cuda(), out2)
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(300, 520, 200), (513, 700, 129), (1000, 777, 301)])
def test_tf32_any_storage_runs_k_major_with_a_workspace(oracle_mod, ta, tb, M, N, K):
    """TF32 with a workspace of workspace_bytes_ex bytes: MN-major operands are
    transposed into K-major copies (odd pitches re-pitched on the way) and the
    product runs on the pair kernel as for A stored M x K and B stored N x K,
    with that storage's bits."""
    A, B = inputs.make(M, N, K, "f32", "normal", 1.0, seed=M + 3 * N + 7 * K + ta + 2 * tb)
    C, need = run("tf32", A, B, ta, tb)
    assert need > 0
    C_nt, _ = run("tf32", A, B, 0, 1)
    assert torch.equal(C, C_nt)
    As, Bs = oracle_mod.truncate_tf32(A.numpy()), oracle_mod.truncate_tf32(B.numpy())
    ref, refabs = oracle_mod.gemm(As, Bs)
    ok, worst = oracle_mod.within_bound(C.numpy(), ref, refabs, TOL["f32"])
    assert ok, worst


def test_tf32_transposed_copies_with_alpha_beta(oracle_mod):
    M, N, K = 700, 530, 333
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=41)
    C0 = torch.from_numpy(np.random.default_rng(42).standard_normal((M, N)).astype(np.float32))
    C, need = run("tf32", A, B, 1, 0, a_off=1, alpha=-1.5, beta=0.5, C0=C0)
    C_nt, _ = run("tf32", A, B, 0, 1, alpha=-1.5, beta=0.5, C0=C0)
    assert need > 0 and torch.equal(C, C_nt)


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("M,N,K", [(2048, 1536, 200), (2049, 2047, 301), (3072, 3072, 3072)])
def test_fp32_b_stored_n_by_k_runs_k_by_n(oracle_mod, ta, M, N, K):
    """fp32 with B stored N x K and a workspace: B is transposed into K x N and
    the product has the bits of B stored K x N from the start."""
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=M + N + K + ta)
    C, need = run("f32", A, B, ta, 1)
    assert need > 0
    C_kn, _ = run("f32", A, B, ta, 0)
    assert torch.equal(C, C_kn)
    oracle_check(oracle_mod, A, B, C, rows=np.arange(0, M, 17) if M * N * K > 1e9 else None)
