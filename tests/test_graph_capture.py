"""Products captured in a CUDA graph and replayed: the stream-K schedule's
publication flags must not let a replay's tile owner take a partial sum that
the replay has not yet written (the call's epoch is fixed at capture). Each
replay runs on new inputs and is checked against the oracle; the capture holds
split products of all three split kernels, a re-pitched one, and a 3xTF32 one
whose lo parts the replay writes afresh."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import oracle_check

pytestmark = pytest.mark.gpu

F32, BF16, X3 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16, g14.GEMM14_DTYPE_F32_3XTF32
CODE = {"f32": F32, "bf16": BF16, "x3": X3}

# (dtype, M, N, K, ldb): fp32 just over one wave of tiles (the last ones
# shared by every SM, A transposed first), the one-SM tensor kernel with 4
# workers a 64-row tile, the pair kernel between one and two waves, fp32 with
# an odd B pitch (re-pitched, then split), and 3xTF32 split ahead (B
# transposed, lo parts) on the pair kernel over 12 clusters
CASES = [("f32", 2560, 2048, 256, 2048), ("bf16", 300, 100, 5000, 104),
         ("bf16", 2304, 2560, 8192, 2560), ("f32", 2560, 2047, 129, 2049),
         ("x3", 512, 384, 1001, 384)]


def test_split_products_replayed_from_a_graph(oracle_mod):
    s = torch.cuda.Stream()
    bufs = []
    for i, (dt, M, N, K, ldb) in enumerate(CASES):
        code = CODE[dt]
        td = torch.bfloat16 if dt == "bf16" else torch.float32
        a = torch.zeros(M, K, dtype=td, device="cuda")
        b = torch.zeros(K, ldb, dtype=td, device="cuda")
        c = torch.zeros(M, N, device="cuda")
        need = g14.workspace_bytes_ex(code, 0, 0, M, N, K, a.data_ptr(), K, b.data_ptr(), ldb,
                                      c.data_ptr(), N)
        assert need > 0
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        bufs.append((code, dt, M, N, K, ldb, a, b, c, ws, need))

    def issue():
        for code, dt, M, N, K, ldb, a, b, c, ws, need in bufs:
            g14.gemm_ex(code, 0, 0, M, N, K, 1.0, a.data_ptr(), K, b.data_ptr(), ldb, 0.0,
                        c.data_ptr(), N, ws.data_ptr(), need, s.cuda_stream)

    # warm-up outside the capture (kernel attributes, first-use set-up)
    with torch.cuda.stream(s):
        issue()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        issue()
    for rep in range(4):
        host = []
        for i, (code, dt, M, N, K, ldb, a, b, c, ws, need) in enumerate(bufs):
            A, B = inputs.make(M, N, K, "bf16" if dt == "bf16" else "f32", "normal",
                               1.0 / K ** 0.5, seed=100 * rep + i)
            a.copy_(A.cuda())
            b[:, :N].copy_(B.cuda())
            c.fill_(float("nan"))
            host.append((A, B, c))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert g14.check_device_error(torch.cuda.current_stream().cuda_stream) == 0
        for (A, B, c), (code, dt, M, N, K, *_rest) in zip(host, bufs):
            oracle_check(oracle_mod, A, B, c.cpu(),
                         rows=np.arange(0, M, 13) if M * N * K > 1e9 else None)


def test_small_tile_products_replayed_from_a_graph(oracle_mod):
    """The fp32 small-tile kernel's cluster launches (the k split summed
    through distributed shared memory) captured in a graph with a 64-row
    tensor-core product between them, replayed on new inputs."""
    cases = [("f32", 256, 256, 256), ("bf16", 1000, 64, 1000), ("f32", 300, 260, 190)]
    s = torch.cuda.Stream()
    bufs = []
    for dt, M, N, K in cases:
        td = torch.bfloat16 if dt == "bf16" else torch.float32
        bufs.append((dt, M, N, K, torch.zeros(M, K, dtype=td, device="cuda"),
                     torch.zeros(K, N, dtype=td, device="cuda"), torch.zeros(M, N, device="cuda")))
    entry = {"f32": g14.gemm_f32, "bf16": g14.gemm_bf16_f32acc}

    def issue():
        for dt, M, N, K, a, b, c in bufs:
            entry[dt](M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, s.cuda_stream)

    with torch.cuda.stream(s):
        issue()  # warm-up outside the capture (kernel attributes)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        issue()
    for rep in range(3):
        host = []
        for i, (dt, M, N, K, a, b, c) in enumerate(bufs):
            A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=300 + 10 * rep + i)
            a.copy_(A.cuda())
            b.copy_(B.cuda())
            c.fill_(float("nan"))
            host.append((A, B, c))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert g14.check_device_error(torch.cuda.current_stream().cuda_stream) == 0
        for A, B, c in host:
            oracle_check(oracle_mod, A, B, c.cpu())


def test_plain_loader_variants_replayed_from_a_graph(oracle_mod):
    """Plain calls (no workspace) of the loader variants captured in one graph:
    fp32 with B stored N x K (tiles transposed in shared memory), fp32 with
    odd pitches (the cp.async loader), bf16 with only A by the software loader
    (B by TMA in the same stages), and bf16 with both by software; replayed on
    new inputs against the oracle."""
    from gpu_util import oracle_check_ex, stored
    # (dt, tb, M, N, K, extra pitch of A, extra pitch of B)
    cases = [("f32", 1, 2100, 2048, 300, 0, 0), ("f32", 0, 2100, 2047, 129, 1, 1),
             ("bf16", 0, 700, 520, 333, 1, 0), ("bf16", 0, 300, 130, 257, 1, 3)]
    s = torch.cuda.Stream()
    bufs = []
    for dt, tb, M, N, K, xa, xb in cases:
        td = torch.bfloat16 if dt == "bf16" else torch.float32
        q = 8 if dt == "bf16" else 4
        b_cols = K if tb else N
        lda = (-(-K // q) * q) if xa == 0 else K + xa
        ldb = (-(-b_cols // q) * q) if xb == 0 else b_cols + xb
        a = torch.zeros(M, lda, dtype=td, device="cuda")
        b = torch.zeros(N if tb else K, ldb, dtype=td, device="cuda")
        c = torch.zeros(M, N, device="cuda")
        bufs.append((dt, tb, M, N, K, lda, ldb, a, b, c))

    def issue():
        for dt, tb, M, N, K, lda, ldb, a, b, c in bufs:
            g14.gemm_ex(CODE[dt], 0, tb, M, N, K, 1.0, a.data_ptr(), lda, b.data_ptr(), ldb, 0.0,
                        c.data_ptr(), N, None, 0, s.cuda_stream)

    with torch.cuda.stream(s):
        issue()  # warm-up outside the capture (kernel attributes)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        issue()
    for rep in range(3):
        host = []
        for i, (dt, tb, M, N, K, lda, ldb, a, b, c) in enumerate(bufs):
            A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=500 + 10 * rep + i)
            Bs = stored(B, tb)
            a[:, :K].copy_(A.cuda())
            b[:, :Bs.shape[1]].copy_(Bs.cuda())
            c.fill_(float("nan"))
            host.append((A, B, c))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert g14.check_device_error(torch.cuda.current_stream().cuda_stream) == 0
        for (A, B, c), (dt, tb, M, *_rest) in zip(host, bufs):
            rows = torch.arange(0, M, 17)
            oracle_check_ex(oracle_mod, A[rows].contiguous(), B, c.cpu()[rows].contiguous(), 0, tb)
