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
