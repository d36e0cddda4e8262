"""Runs a fixed set of products through gemm14_gemm_ex on whichever library
GEMM14_LIB names, covering every kernel, loader and schedule: the fp32 FFMA
kernel (TMA and cp.async loaders, data-parallel and stream-K, the A transpose
copy), the fp32 small-product kernel (cluster split, both loaders), the
one-SM tensor-core kernel with 64- and 128-row tiles and the CTA-pair one
(data-parallel, stream-K, the hybrid split, the software loader, the
TMA-store epilogue with a ragged N), TF32 on both tf32 kernels and split
3xTF32, the alpha/beta epilogue and stored transposes.

    python device_checks_worker.py OUT.npz

writes every case's C and the status gemm14_check_device_error returned
after it (tests/test_device_checks.py runs it on the build with device-side
bounds checks and compares with the product build in its own process)."""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import dense_gemm_14_gb300 as g14  # noqa: E402
from dense_gemm_14_gb300 import inputs  # noqa: E402

F32, BF16, F16 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16, g14.GEMM14_DTYPE_F16
TF32, X3 = g14.GEMM14_DTYPE_TF32, g14.GEMM14_DTYPE_F32_3XTF32
DT = {F32: "f32", BF16: "bf16", F16: "f16", TF32: "f32", X3: "f32"}

# name, dtype, transa, transb, M, N, K, alpha, beta, workspace, pitch pad (elements), offset
CASES = [
    ("f32 dp", F32, 0, 0, 2048, 2048, 200, 1.0, 0.0, False, 0, 0),
    ("f32 stream-K", F32, 0, 0, 2560, 2048, 513, 1.0, 0.0, True, 0, 0),
    ("f32 A transposed copy", F32, 0, 0, 2048, 2048, 256, 1.0, 0.0, True, 0, 0),
    ("f32 cp.async", F32, 0, 0, 2049, 2047, 129, 1.0, 0.0, False, 1, 1),
    ("f32 transposes alpha beta", F32, 1, 1, 2048, 1536, 190, -1.5, 0.5, True, 0, 0),
    ("f32 small split 8", F32, 0, 0, 256, 256, 256, 1.0, 0.0, False, 0, 0),
    ("f32 small 4-byte loader", F32, 0, 0, 257, 300, 129, 1.0, 0.0, False, 1, 1),
    ("f32 small transposes alpha beta", F32, 1, 1, 300, 260, 190, -1.5, 0.5, True, 0, 0),
    ("bf16 one-SM 64-row dp", BF16, 0, 0, 4096, 64, 512, 1.0, 0.0, False, 0, 0),
    ("bf16 one-SM 128-row dp", BF16, 0, 0, 32768, 64, 512, 1.0, 0.0, False, 0, 0),
    ("bf16 one-SM 64-row stream-K", BF16, 0, 0, 512, 128, 8192, 1.0, 0.0, True, 0, 0),
    ("bf16 one-SM 128-row stream-K", BF16, 0, 0, 23040, 64, 1024, 1.0, 0.0, True, 0, 0),
    ("bf16 pair dp ragged N", BF16, 0, 0, 1000, 777, 130, 1.0, 0.0, False, 0, 0),
    ("bf16 pair stream-K", BF16, 0, 0, 2304, 2560, 1024, 1.0, 0.0, True, 0, 0),
    ("bf16 pair hybrid", BF16, 0, 0, 4096, 5120, 256, 1.0, 0.0, True, 0, 0),
    ("bf16 software loader", BF16, 0, 0, 300, 129, 77, 1.0, 0.0, False, 1, 1),
    ("bf16 transposes beta", BF16, 1, 0, 520, 300, 200, 2.0, 1.0, True, 0, 0),
    ("f16 pair", F16, 0, 1, 512, 512, 512, 1.0, 0.0, True, 0, 0),
    ("tf32 converter", TF32, 0, 0, 300, 520, 200, 1.0, 0.0, False, 0, 0),
    ("tf32 pair", TF32, 0, 1, 512, 512, 8192, 1.0, 0.0, True, 0, 0),
    ("3xtf32 converter", X3, 0, 0, 300, 520, 200, 1.0, 0.0, False, 0, 0),
    ("3xtf32 split", X3, 0, 0, 512, 384, 1001, 1.0, 0.0, True, 0, 0),
]


def stored(X, trans):
    return X.t().contiguous() if trans else X


def run_case(case, stream):
    """Returns (C as a float32 numpy array, the status after the call)."""
    name, code, ta, tb, M, N, K, alpha, beta, use_ws, pad, off = case
    dt = DT[code]
    A, B = inputs.make(M, N, K, dt, "normal", 1.0 / K ** 0.5, seed=M + 3 * N + 7 * K + code)
    As, Bs = stored(A, ta), stored(B, tb)
    q = 4 if dt == "f32" else 8
    lda = (As.shape[1] + q - 1) // q * q + pad
    ldb = (Bs.shape[1] + q - 1) // q * q + pad
    # aligned cases: a padded pitch that takes 16-byte stores (and the TMA-store
    # epilogue, whose last chunk past a ragged N stores directly); else odd
    ldc = N + pad if pad else (N + 3) // 4 * 4 + 4
    a = torch.zeros(off + As.shape[0] * lda, dtype=As.dtype, device="cuda")
    b = torch.zeros(off + Bs.shape[0] * ldb, dtype=Bs.dtype, device="cuda")
    a[off:].view(As.shape[0], lda)[:, :As.shape[1]] = As.cuda()
    b[off:].view(Bs.shape[0], ldb)[:, :Bs.shape[1]] = Bs.cuda()
    g = torch.Generator().manual_seed(M + N)
    C0 = torch.randn(M, N, generator=g)
    c = torch.full((off + M * ldc,), float("nan"), device="cuda")
    c[off:].view(M, ldc)[:, :N] = C0.cuda()
    eb = a.element_size()
    pa, pb, pc = a.data_ptr() + eb * off, b.data_ptr() + eb * off, c.data_ptr() + 4 * off
    need = 0
    ws = None
    if use_ws:
        need = g14.workspace_bytes_ex(code, ta, tb, M, N, K, pa, lda, pb, ldb, pc, ldc)
        ws = torch.zeros(max(need, 16), dtype=torch.uint8, device="cuda")
    g14.gemm_ex(code, ta, tb, M, N, K, alpha, pa, lda, pb, ldb, beta, pc, ldc,
                ws.data_ptr() if ws is not None else None, need, stream)
    status = g14.check_device_error(stream)
    torch.cuda.synchronize()
    out = c[off:].view(M, ldc).cpu().numpy()
    return out, status


def main():
    stream = torch.cuda.current_stream().cuda_stream
    results = {}
    for i, case in enumerate(CASES):
        out, status = run_case(case, stream)
        results[f"c{i}"] = out
        results[f"s{i}"] = np.array(status)
    results["lib"] = np.array(g14.lib_path())
    np.savez(sys.argv[1], **results)


if __name__ == "__main__":
    main()
