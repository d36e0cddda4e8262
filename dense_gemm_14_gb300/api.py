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
        nbytes = _lib.workspace_bytes_ex(code, ta, tb, M, N, K, a.data_ptr(), lda, b.data_ptr(),
                                         ldb, out.data_ptr(), max(out.stride(0), N, 1)) \
            if M and N and K else 0
        ws = _workspace(a.device, int(stream or 0), nbytes) if nbytes else None
        _lib.gemm_ex(code, ta, tb, M, N, K, float(alpha), a.data_ptr(), lda,
                     b.data_ptr(), ldb, float(beta), out.data_ptr(), max(out.stride(0), N, 1),
                     ws.data_ptr() if ws is not None else None, nbytes, stream)
    return out


class HostGemm:
    """A product with host operands in flight (gemm_async): `out` is the host
    tensor that holds the result once wait() returns. Keeps the operands (and
    any pinned copies made of them) alive until then; a handle dropped unwaited
    waits in its finaliser."""

    def __init__(self, out: torch.Tensor, ticket: int, keep: tuple):
        self.out = out
        self._ticket = ticket
        self._keep = keep

    def wait(self) -> torch.Tensor:
        if self._ticket:
            t, self._ticket = self._ticket, 0
            _lib.host_wait(t)
            self._keep = ()
        return self.out

    def __del__(self):
        if getattr(self, "_ticket", 0):
            try:
                _lib.host_wait(self._ticket, check=False)
            except Exception:  # interpreter shutdown
                pass


def _product_code(a: torch.Tensor, b: torch.Tensor, fp32_mode: str | None) -> int:
    if a.dtype != b.dtype or a.dtype not in _CODE:
        raise TypeError(f"unsupported dtypes {a.dtype}, {b.dtype}")
    if fp32_mode not in _FP32_MODES or (fp32_mode not in (None, "fp32") and a.dtype != torch.float32):
        raise ValueError(f"fp32_mode {fp32_mode!r} needs float32 inputs and one of {list(_FP32_MODES)}")
    return _FP32_MODES[fp32_mode] if a.dtype == torch.float32 else _CODE[a.dtype]


def gemm_async(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
               alpha: float = 1.0, beta: float = 0.0, fp32_mode: str | None = None,
               panels: int | None = None) -> HostGemm:
    """C = alpha * a @ b + beta * out for host (CPU) tensors through the C ABI
    gemm14_gemm_host, on the current CUDA device, without waiting: returns a
    HostGemm whose wait() returns `out` (a float32 (M, N) row-major host
    tensor, pinned and allocated if not given) once the result is there.

    a, b: as for gemm_into (row-major views or transposes of them). Operands
    that are not pinned are pinned first (a copy kept until the wait). The
    library sends a in row panels (`panels`, or its own choice) after b, and
    overlaps copying panels in, computing and copying results out, within a
    product and from one product to the next; a product whose operand is the
    result of one still in flight waits for it. The caller must not change the
    operands, nor read `out`, before wait()."""
    if a.is_cuda or b.is_cuda:
        raise ValueError("gemm_async takes host tensors; use gemm_into for CUDA tensors")
    code = _product_code(a, b, fp32_mode)
    M, K = a.shape
    K2, N = b.shape
    if K != K2:
        raise ValueError(f"shape mismatch: {tuple(a.shape)} @ {tuple(b.shape)}")
    if not a.is_pinned():
        a = a.pin_memory()
    if not b.is_pinned():
        b = b.pin_memory()
    ta, lda = _operand(a, "a")
    tb, ldb = _operand(b, "b")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    elif out.is_cuda or out.dtype != torch.float32 or tuple(out.shape) != (M, N):
        raise ValueError("out must be a float32 (M, N) host tensor")
    _check_matrix(out, "out")
    ticket = _lib.gemm_host(code, ta, tb, M, N, K, float(alpha),
                            a.data_ptr() if a.numel() else None, lda,
                            b.data_ptr() if b.numel() else None, ldb, float(beta),
                            out.data_ptr() if out.numel() else None, max(out.stride(0), N, 1),
                            int(panels or 0))
    return HostGemm(out, ticket, (a, b))


def gemm(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
         alpha: float = 1.0, beta: float = 0.0, fp32_mode: str | None = None,
         panels: int | None = None) -> torch.Tensor:
    """C = alpha * a @ b + beta * out with fp32 accumulation and output.

    CUDA inputs: computed on the current stream, returned on the GPU (as
    gemm_into).

    CPU inputs: gemm_async(...).wait(): the result lands in host memory
    (`out`, a float32 (M, N) tensor, pinned and allocated if not given) and
    the call returns once it is there."""
    if a.is_cuda:
        if out is None:
            out = torch.empty((a.shape[0], b.shape[1]), dtype=torch.float32, device=a.device)
        return gemm_into(a, b, out, alpha, beta, fp32_mode=fp32_mode)
    return gemm_async(a, b, out, alpha, beta, fp32_mode, panels).wait()
