"""Helpers for the GPU tests: run the library through its C ABI on buffers
with chosen leading dimensions and offsets, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

# Element-wise bounds |C - C_ref| <= tol * (|A||B|)_ij (inputs as rounded).
TOL = {"f32": 1e-5, "bf16": 4e-3, "f16": 4e-3}
ENTRY = {"f32": g14.gemm_f32, "bf16": g14.gemm_bf16_f32acc, "f16": g14.gemm_f16_f32acc}


def dtype_name(t: torch.Tensor) -> str:
    return {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[t.dtype]


def to_device_padded(x: torch.Tensor, ld: int, offset_elems: int = 0) -> tuple[torch.Tensor, torch.Tensor]:
    """Copies a (rows, cols) CPU matrix into a device buffer with row pitch ld,
    starting offset_elems into the buffer. Returns (buffer, view)."""
    rows, cols = x.shape
    buf = torch.zeros(offset_elems + max(rows, 1) * ld + 16, dtype=x.dtype, device="cuda")
    view = buf[offset_elems:offset_elems + rows * ld].view(rows, ld)[:, :cols] if rows else \
        buf[offset_elems:offset_elems].view(0, ld)[:, :cols]
    view.copy_(x.to("cuda"))
    return buf, view


ENTRY_WS = {"f32": g14.gemm_f32_ws, "bf16": g14.gemm_bf16_f32acc_ws,
            "f16": g14.gemm_f16_f32acc_ws}


def run_abi(A: torch.Tensor, B: torch.Tensor, lda=None, ldb=None, ldc=None, a_off=0, b_off=0,
            c_off=0, stream=None, poison=True, check_err=True, workspace=None):
    """C = A @ B through the C ABI entry point for A's dtype (the *_ws entry
    point when a workspace tensor is given). Returns C (CPU fp32)."""
    M, K = A.shape
    _, N = B.shape
    lda = lda or max(K, 1)
    ldb = ldb or max(N, 1)
    ldc = ldc or max(N, 1)
    _abuf, a = to_device_padded(A, lda, a_off)
    _bbuf, b = to_device_padded(B, ldb, b_off)
    cbuf = torch.full((c_off + max(M, 1) * ldc + 16,), float("nan") if poison else 0.0,
                      dtype=torch.float32, device="cuda")
    c_ptr = cbuf.data_ptr() + 4 * c_off
    s = stream if stream is not None else torch.cuda.current_stream()
    if workspace is None:
        ENTRY[dtype_name(A)](M, N, K, a.data_ptr() if M and K else 0, lda,
                             b.data_ptr() if K and N else 0, ldb, c_ptr, ldc, s.cuda_stream)
    else:
        ENTRY_WS[dtype_name(A)](M, N, K, a.data_ptr() if M and K else 0, lda,
                                b.data_ptr() if K and N else 0, ldb, c_ptr, ldc,
                                workspace.data_ptr(), workspace.numel(), s.cuda_stream)
    if check_err:
        st = g14.check_device_error(s.cuda_stream)
        assert st == 0, g14.status_string(st)
    torch.cuda.synchronize()
    if M == 0:
        return torch.empty((0, N))
    C = cbuf[c_off:c_off + M * ldc].view(M, ldc)[:, :N].cpu()
    return C


def oracle_check(oracle_mod, A: torch.Tensor, B: torch.Tensor, C: torch.Tensor, rows=None):
    """Element-wise comparison with the oracle on all rows (or the given rows)."""
    dt = dtype_name(A)
    Ah = inputs.host_view(A)
    Bh = inputs.host_view(B)
    if rows is not None:
        Ah = np.ascontiguousarray(Ah[rows])
        Cg = C.numpy()[rows]
    else:
        Cg = C.numpy()
    ref, refabs = oracle_mod.gemm(Ah, Bh, dt)
    ok, worst = oracle_mod.within_bound(Cg, ref, refabs, TOL[dt])
    if not ok:
        diff = np.abs(Cg.astype(np.float64) - ref) - TOL[dt] * refabs
        bad = np.argwhere(~(diff <= 0))
        i, j = bad[0]
        raise AssertionError(
            f"{dt} {tuple(A.shape)}x{tuple(B.shape)}: {len(bad)} elements out of bound; "
            f"first at ({i},{j}) gpu={Cg[i, j]!r} ref={ref[i, j]!r} abs={refabs[i, j]!r}; worst={worst:.3g}")
    return worst


def make_workspace(dtype: str, M: int, N: int, K: int) -> torch.Tensor:
    """A zero-filled device workspace large enough for the stream-K schedule."""
    code = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16,
            "f16": g14.GEMM14_DTYPE_F16}[dtype]
    n = g14.workspace_bytes(code, M, N, K, 0)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")


DTYPE_CODE = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16,
              "f16": g14.GEMM14_DTYPE_F16}


def stored(X: torch.Tensor, trans: int) -> torch.Tensor:
    """The matrix as the library reads it: X itself, or X^T stored row-major."""
    return X.t().contiguous() if trans else X


def run_ex(A: torch.Tensor, B: torch.Tensor, transa=0, transb=0, alpha=1.0, beta=0.0,
           C0: torch.Tensor | None = None, lda=None, ldb=None, ldc=None, a_off=0, b_off=0,
           c_off=0, workspace=None, stream=None, check_err=True):
    """C = alpha * A @ B + beta * C0 through gemm14_gemm_ex, with A (M x K) and
    B (K x N) stored transposed when transa / transb. C0 None: C starts as NaN
    (which beta == 0 must ignore). Returns C (CPU fp32)."""
    M, K = A.shape
    _, N = B.shape
    As, Bs = stored(A, transa), stored(B, transb)
    lda = lda or max(As.shape[1], 1)
    ldb = ldb or max(Bs.shape[1], 1)
    ldc = ldc or max(N, 1)
    _abuf, a = to_device_padded(As, lda, a_off)
    _bbuf, b = to_device_padded(Bs, ldb, b_off)
    cbuf = torch.full((c_off + max(M, 1) * ldc + 16,), float("nan"), dtype=torch.float32,
                      device="cuda")
    if C0 is not None and M:
        cbuf[c_off:c_off + M * ldc].view(M, ldc)[:, :N].copy_(C0.to("cuda"))
    c_ptr = cbuf.data_ptr() + 4 * c_off
    s = stream if stream is not None else torch.cuda.current_stream()
    g14.gemm_ex(DTYPE_CODE[dtype_name(A)], transa, transb, M, N, K, alpha,
                a.data_ptr() if As.numel() else 0, lda, b.data_ptr() if Bs.numel() else 0, ldb,
                beta, c_ptr, ldc, workspace.data_ptr() if workspace is not None else None,
                workspace.numel() if workspace is not None else 0, s.cuda_stream)
    if check_err:
        st = g14.check_device_error(s.cuda_stream)
        assert st == 0, g14.status_string(st)
    torch.cuda.synchronize()
    if M == 0:
        return torch.empty((0, N))
    return cbuf[c_off:c_off + M * ldc].view(M, ldc)[:, :N].cpu()


def oracle_check_ex(oracle_mod, A, B, C, transa=0, transb=0, alpha=1.0, beta=0.0, C0=None):
    """Element-wise comparison with the oracle's extended product, which reads
    the same stored (possibly transposed) matrices."""
    dt = dtype_name(A)
    As = inputs.host_view(stored(A, transa))
    Bs = inputs.host_view(stored(B, transb))
    c0 = C0.numpy().astype(np.float32) if C0 is not None else None
    ref, refabs = oracle_mod.gemm_ex(As, Bs, dt, bool(transa), bool(transb), float(alpha),
                                     float(beta), c0)
    Cg = C.numpy()
    ok, worst = oracle_mod.within_bound(Cg, ref, refabs, TOL[dt])
    if not ok:
        diff = np.abs(Cg.astype(np.float64) - ref) - TOL[dt] * refabs
        bad = np.argwhere(~(diff <= 0))
        i, j = bad[0]
        raise AssertionError(
            f"{dt} op(A) {tuple(A.shape)} op(B) {tuple(B.shape)} ta={transa} tb={transb} "
            f"alpha={alpha} beta={beta}: {len(bad)} elements out of bound; first at ({i},{j}) "
            f"gpu={Cg[i, j]!r} ref={ref[i, j]!r} abs={refabs[i, j]!r}; worst={worst:.3g}")
    return worst
