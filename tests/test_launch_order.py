"""Back-to-back products on one stream, with no host synchronisation between
them. The library launches its kernels with programmatic stream serialisation,
so a kernel may start while the one before it still runs, and must wait for
it before touching global memory. Chains in which a product reads the
previous one's output (read after write), or overwrites what the previous one
reads (write after read), must give the bits that the same calls give one at
a time with a synchronisation after each, and, with integer-valued data, the
exact products."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14

pytestmark = pytest.mark.gpu

F32, BF16, X3 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16, g14.GEMM14_DTYPE_F32_3XTF32


def signed_sparse(K, N, nnz, seed):
    """K x N with exactly nnz entries of +-1 per column (nnz = 1: a signed
    permutation when K == N), so that integer data grow at most nnz-fold."""
    g = np.random.default_rng(seed)
    W = np.zeros((K, N), dtype=np.float32)
    if nnz == 1 and K == N:
        W[g.permutation(N), np.arange(N)] = g.choice([-1.0, 1.0], size=N)
    else:
        for j in range(N):
            W[g.permutation(K)[:nnz], j] = g.choice([-1.0, 1.0], size=nnz)
    return torch.from_numpy(W)


def small_ints(shape, r, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(-r, r + 1, shape, generator=g).float()


def ex(dtype, M, N, K, A, B, C, alpha=1.0, beta=0.0):
    """One gemm14_gemm_ex call on the current stream: C = alpha A B + beta C,
    all row-major and dense (A, B, C device tensors or raw pointers)."""
    ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
    g14.gemm_ex(dtype, 0, 0, M, N, K, alpha, ptr(A), max(K, 1), ptr(B), N, beta, ptr(C), N, None, 0,
                torch.cuda.current_stream().cuda_stream)


def run_both(bufs, steps):
    """Runs steps (callables issuing one library call each) twice from the
    same starting buffers: chained, then one at a time with a synchronisation
    after each. Returns both final snapshots of every buffer."""
    start = {k: v.clone() for k, v in bufs.items()}
    out = []
    for sync_each in (False, True):
        for k in bufs:
            bufs[k].copy_(start[k])
        torch.cuda.synchronize()
        for step in steps:
            step()
            if sync_each:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert g14.check_device_error(torch.cuda.current_stream().cuda_stream) == 0
        out.append({k: v.clone().cpu() for k, v in bufs.items()})
    return out


def same_bits(a, b):
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


def check_all(chained, serial, want):
    for k in chained:
        assert same_bits(chained[k], serial[k]), k
    for k, v in want.items():
        assert torch.equal(chained[k].double(), v), k


@pytest.mark.parametrize("dtype,M", [(F32, 16384), (X3, 4096)])
def test_ping_pong(dtype, M):
    """Y = X W1, then X = Y W2, twenty times: every product reads what the one
    before wrote and overwrites what it read. W1, W2 are signed permutations,
    so the result is exact: X0 (W1 W2)^20."""
    K = 256
    X0 = small_ints((M, K), 3, 1)
    W1, W2 = signed_sparse(K, K, 1, 2), signed_sparse(K, K, 1, 3)
    d = {"X": X0.cuda(), "Y": torch.zeros(M, K, device="cuda"), "W1": W1.cuda(),
         "W2": W2.cuda()}
    steps = []
    for _ in range(20):
        steps.append(lambda: ex(dtype, M, K, K, d["X"], d["W1"], d["Y"]))
        steps.append(lambda: ex(dtype, M, K, K, d["Y"], d["W2"], d["X"]))
    chained, serial = run_both(d, steps)
    P = torch.linalg.matrix_power(W1.double() @ W2.double(), 20)
    check_all(chained, serial, {"X": X0.double() @ P})


def test_mixed_kernels_chain():
    """fp32 kernel -> CTA-pair bf16 kernel -> fp32 kernel -> 3xTF32 kernel with
    beta = 1 -> the beta-only scale kernel, each reading the one before's
    output; the last overwrites a matrix that the 3xTF32 product reads."""
    M, N, K, P = 1024, 1024, 512, 256
    g = torch.Generator().manual_seed(7)
    vals = torch.tensor([-2.0, -1.0, -0.5, 0.5, 1.0, 2.0])
    A16 = vals[torch.randint(0, 6, (M, K), generator=g)].to(torch.bfloat16)
    B16 = vals[torch.randint(0, 6, (K, N), generator=g)].to(torch.bfloat16)
    # A16's bytes as fp32: M x K/2 normal numbers (no high half is zero)
    S = A16.view(torch.float32)
    W = signed_sparse(N, P, 4, 8)
    W2 = signed_sparse(P, P, 1, 9)
    E0 = small_ints((M, P), 5, 10)
    d = {"S": S.cuda(), "I": torch.eye(K // 2).cuda(), "Acopy": torch.zeros(M, K // 2).cuda(),
         "B": B16.cuda(), "C": torch.zeros(M, N).cuda(), "W": W.cuda(),
         "D": torch.zeros(M, P).cuda(), "W2": W2.cuda(), "E": E0.cuda()}
    steps = [
        # Acopy = S I: the bits of A16, written by the fp32 kernel
        lambda: ex(F32, M, K // 2, K // 2, d["S"], d["I"], d["Acopy"]),
        # C = A16 B16 on the pair kernel, A read from Acopy's bytes
        lambda: ex(BF16, M, N, K, d["Acopy"].data_ptr(), d["B"], d["C"]),
        lambda: ex(F32, M, P, N, d["C"], d["W"], d["D"]),
        # E = 2 D W2 + E
        lambda: ex(X3, M, P, P, d["D"], d["W2"], d["E"], alpha=2.0, beta=1.0),
        # D = -D (no product term: the scale kernel), after D W2 has read it
        lambda: ex(F32, M, P, 0, 0, 0, d["D"], alpha=0.0, beta=-1.0),
    ]
    chained, serial = run_both(d, steps)
    C = A16.double() @ B16.double()
    D = C @ W.double()
    want = {"Acopy": S.double(), "C": C, "D": -D, "E": 2.0 * (D @ W2.double()) + E0.double()}
    assert same_bits(chained["Acopy"], S)
    check_all(chained, serial, want)


def test_split_products_share_a_workspace():
    """Stream-K products (one-SM tensor-core kernel, 4 workers per tile) back
    to back on one workspace, with an fp32 product between them that reads the
    first one's output before the last overwrites it."""
    M, N, K = 128, 64, 4096
    ws_bytes = g14.workspace_bytes(BF16, M, N, K, 0)
    assert ws_bytes > 0
    g = torch.Generator().manual_seed(11)
    A = torch.randint(-2, 3, (M, K), generator=g).to(torch.bfloat16)
    B1 = torch.randint(-2, 3, (K, N), generator=g).to(torch.bfloat16)
    B2 = torch.randint(-2, 3, (K, N), generator=g).to(torch.bfloat16)
    W = signed_sparse(N, N, 1, 12)
    d = {"A": A.cuda(), "B1": B1.cuda(), "B2": B2.cuda(), "W": W.cuda(),
         "C1": torch.zeros(M, N).cuda(), "C2": torch.zeros(M, N).cuda(),
         "D": torch.zeros(M, N).cuda(), "ws": torch.zeros(ws_bytes, dtype=torch.uint8).cuda()}
    s = lambda: torch.cuda.current_stream().cuda_stream

    def split(Bk, Ck):
        return lambda: g14.gemm_bf16_f32acc_ws(M, N, K, d["A"].data_ptr(), K, d[Bk].data_ptr(), N,
                                               d[Ck].data_ptr(), N, d["ws"].data_ptr(), ws_bytes,
                                               s())
    steps = [split("B1", "C1"), split("B2", "C2"),
             lambda: ex(F32, M, N, N, d["C1"], d["W"], d["D"]),
             split("B2", "C1")]
    chained, serial = run_both(d, steps)
    del chained["ws"], serial["ws"]  # flag words carry a per-call epoch
    A64 = A.double()
    want = {"C1": A64 @ B2.double(), "C2": A64 @ B2.double(),
            "D": (A64 @ B1.double()) @ W.double()}
    check_all(chained, serial, want)
