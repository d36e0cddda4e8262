"""Tensor-level calls on top of the C ABI (argument marshalling only)."""
from __future__ import annotations

import torch

from . import _lib

_CODE = {torch.float32: _lib.GEMM14_DTYPE_F32, torch.bfloat16: _lib.GEMM14_DTYPE_BF16,
         torch.float16: _lib.GEMM14_DTYPE_F16}

# Stream-K workspaces, one per (device, stream): calls on one stream run in
# order, so they may share it; calls on different streams must not.
_workspaces: dict = {}


def _workspace(device: torch.device, stream_handle: int, nbytes: int) -> torch.Tensor:
    key = (device.index, stream_handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        # zero-filled once: the library leaves only epochs of finished calls in it
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _check_matrix(x: torch.Tensor, name: str) -> None:
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(x.shape)}")
    if x.size(1) > 1 and x.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its rows (row-major)")


def _operand(x: torch.Tensor, name: str) -> tuple[int, int]:
    """(trans, ld) of an operand view: trans 0 for a row-major view (unit
    stride along rows, pitch stride(0)); trans 1 for the transpose of a
    row-major matrix (unit stride down columns, pitch stride(1))."""
    if x.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(x.shape)}")
    rows, cols = x.shape
    if cols <= 1 or x.stride(1) == 1:
        if rows > 1 and x.stride(0) < max(cols, 1):
            raise ValueError(f"{name}: rows overlap (stride {x.stride()})")
        return 0, max(x.stride(0), cols, 1)
    if rows <= 1 or x.stride(0) == 1:
        if x.stride(1) < max(rows, 1):
            raise ValueError(f"{name}: columns overlap (stride {x.stride()})")
        return 1, max(x.stride(1), rows, 1)
    raise ValueError(f"{name} needs unit stride along its rows or its columns, got {x.stride()}")


_FP32_MODES = {None: _lib.GEMM14_DTYPE_F32, "fp32": _lib.GEMM14_DTYPE_F32,
               "tf32": _lib.GEMM14_DTYPE_TF32, "3xtf32": _lib.GEMM14_DTYPE_F32_3XTF32}


def gemm_into(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor, alpha: float = 1.0,
              beta: float = 0.0, stream=None, fp32_mode: str | None = None) -> torch.Tensor:
    """out = alpha * a @ b + beta * out on the GPU through the C ABI
    (gemm14_gemm_ex); a, b, out are CUDA tensors.

    a: (M, K), b: (K, N) in float32, bfloat16 or float16 (same dtype), each
    either a row-major view or the transpose of one (e.g. ``x.t()``), which
    becomes the call's transa / transb; out: (M, N) float32, row-major. With
    beta == 0, out is not read. Uses a stream-K workspace cached per (device,
    stream) when the product benefits from it. Runs on `stream` (default:
    torch's current stream) without synchronising. fp32_mode (float32 inputs
    only): "fp32" (default, FFMA), "tf32" or "3xtf32" (tensor cores).
    """
    if a.dtype != b.dtype or a.dtype not in _CODE:
        raise TypeError(f"unsupported dtypes {a.dtype}, {b.dtype}")
    if out.dtype != torch.float32:
        raise TypeError("out must be float32")
    for x, n in ((a, "a"), (b, "b"), (out, "out")):
        if not x.is_cuda:
            raise ValueError(f"{n} must be a CUDA tensor")
    _check_matrix(out, "out")
    ta, lda = _operand(a, "a")
    tb, ldb = _operand(b, "b")
    M, K = a.shape
    K2, N = b.shape
    if K != K2 or tuple(out.shape) != (M, N):
        raise ValueError(f"shape mismatch: {tuple(a.shape)} @ {tuple(b.shape)} -> {tuple(out.shape)}")
    if stream is None:
        stream = torch.cuda.current_stream(a.device).cuda_stream
    elif isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    if fp32_mode not in _FP32_MODES or (fp32_mode not in (None, "fp32") and a.dtype != torch.float32):
        raise ValueError(f"fp32_mode {fp32_mode!r} needs float32 inputs and one of {list(_FP32_MODES)}")
    code = _FP32_MODES[fp32_mode] if a.dtype == torch.float32 else _CODE[a.dtype]
    with torch.cuda.device(a.device):
        nbytes = _lib.workspace_bytes(code, M, N, K, 0) if M and N and K else 0
        ws = _workspace(a.device, int(stream or 0), nbytes) if nbytes else None
        _lib.gemm_ex(code, ta, tb, M, N, K, float(alpha), a.data_ptr(), lda,
                     b.data_ptr(), ldb, float(beta), out.data_ptr(), max(out.stride(0), N, 1),
                     ws.data_ptr() if ws is not None else None, nbytes, stream)
    return out


def gemm(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """C = a @ b with fp32 accumulation and output.

    CUDA inputs: computed on the current stream, returned on the GPU.
    CPU inputs: staged through pinned host memory to the current CUDA device,
    computed there, and the result is copied back to (pinned) host memory; the
    call returns once the result is on the host.
    """
    if a.is_cuda:
        if out is None:
            out = torch.empty((a.shape[0], b.shape[1]), dtype=torch.float32, device=a.device)
        return gemm_into(a, b, out)
    dev = torch.device("cuda", torch.cuda.current_device())
    a_d = a.pin_memory().to(dev, non_blocking=True) if not a.is_pinned() else a.to(dev, non_blocking=True)
    b_d = b.pin_memory().to(dev, non_blocking=True) if not b.is_pinned() else b.to(dev, non_blocking=True)
    c_d = torch.empty((a.shape[0], b.shape[1]), dtype=torch.float32, device=dev)
    gemm_into(a_d.contiguous(), b_d.contiguous(), c_d)
    if out is None:
        out = torch.empty((a.shape[0], b.shape[1]), dtype=torch.float32, pin_memory=True)
    out.copy_(c_d, non_blocking=True)
    torch.cuda.current_stream(dev).synchronize()
    return out
