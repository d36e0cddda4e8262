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


# Host-path streams per device: copies in, copies out (compute runs on the
# caller's current stream).
_copy_streams: dict = {}


def _streams(dev: torch.device):
    s = _copy_streams.get(dev.index)
    if s is None:
        s = (torch.cuda.Stream(dev), torch.cuda.Stream(dev))
        _copy_streams[dev.index] = s
    return s


def host_panels(M: int, N: int, K: int) -> int:
    """Row panels the host path splits a product into: one for small products
    (transfers too short to pipeline), else one per 1024 rows, at most 8. On a
    GB300 host link (about 200 GB/s each way) this measured 1.43 ms for fp32
    3072^3 (3 panels; 1.66 ms unsplit) and 2.39 ms for bf16 8192^3 (8; 3.36
    ms unsplit), near the bound set by sending all of B before the first panel."""
    if M * N * K < (1 << 31) or M < 2048:
        return 1
    return min(8, M // 1024)


class HostGemm:
    """A product with host operands in flight (gemm_async): `out` is a pinned
    host tensor that holds the result once wait() returns."""

    def __init__(self, out: torch.Tensor, done: torch.cuda.Event | None):
        self.out = out
        self._done = done

    def ready(self) -> bool:
        return self._done is None or self._done.query()

    def wait(self) -> torch.Tensor:
        if self._done is not None:
            self._done.synchronize()
        return self.out


# Host outputs of products still in flight, per device: (first byte, end byte,
# event after the last copy out). A later product that reads host memory one
# of them still writes (a result fed back as an operand) waits for it first;
# every other order between products is kept by the copy streams themselves.
_pending: dict = {}


def _host_span(x: torch.Tensor) -> tuple[int, int]:
    if x.numel() == 0:
        return 0, 0
    last = sum((n - 1) * st for n, st in zip(x.shape, x.stride()))
    return x.data_ptr(), x.data_ptr() + (last + 1) * x.element_size()


def _wait_for_writers(dev_index: int, s_in: torch.cuda.Stream, inputs) -> None:
    live = [p for p in _pending.get(dev_index, []) if not p[2].query()]
    _pending[dev_index] = live
    for x in inputs:
        lo, hi = _host_span(x)
        for p_lo, p_hi, ev in live:
            if lo < p_hi and p_lo < hi:
                s_in.wait_event(ev)


def gemm_async(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
               alpha: float = 1.0, beta: float = 0.0, fp32_mode: str | None = None,
               panels: int | None = None) -> HostGemm:
    """C = alpha * a @ b + beta * out for host (CPU) operands, on the current
    CUDA device, without waiting for the result: returns a HostGemm whose
    wait() returns `out` (a pinned float32 (M, N) host tensor, allocated if not
    given) once the result is there.

    Inputs that are not pinned are pinned first. A row-major `a` is sent in row
    panels (host_panels, or `panels`) so that copying panel i+1 in, computing
    panel i and copying panel i-1 out overlap on three streams; b is sent once,
    first; with beta != 0 the panels of `out` are sent in too. Products issued
    one after another pipeline: the next one's operands go in while this one
    computes and its result comes out. A product whose host operand is the
    result of one still in flight waits for that result first. The caller
    must not change the operands, nor read `out`, before wait()."""
    if a.is_cuda:
        raise ValueError("gemm_async takes host tensors; use gemm_into for CUDA tensors")
    M, K = a.shape
    N = b.shape[1]
    dev = torch.device("cuda", torch.cuda.current_device())
    if not a.is_pinned():
        a = a.pin_memory()
    if not b.is_pinned():
        b = b.pin_memory()
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    elif out.is_cuda or out.dtype != torch.float32 or tuple(out.shape) != (M, N):
        raise ValueError("out must be a float32 (M, N) host tensor")
    if beta != 0.0 and not out.is_pinned():
        raise ValueError("beta != 0 needs a pinned out (its values are sent to the GPU)")
    row_major_a = a.dim() == 2 and (K <= 1 or a.stride(1) == 1) and a.stride(0) == K
    P = 1 if not row_major_a else (panels if panels else host_panels(M, N, K))
    P = max(1, min(P, M)) if M else 1
    compute = torch.cuda.current_stream(dev)
    s_in, s_out = _streams(dev)
    with torch.cuda.device(dev):
        _wait_for_writers(dev.index, s_in, [a, b] + ([out] if beta != 0.0 else []))
        # Device buffers in the input stream's order; record_stream keeps each
        # block from being handed out again before the other streams that use
        # it are done with it, so no stream waits for earlier products here.
        with torch.cuda.stream(s_in):
            b_d = torch.empty_strided(b.shape, b.stride(), dtype=b.dtype, device=dev)
            a_d = torch.empty_strided(a.shape, a.stride(), dtype=a.dtype, device=dev)
            c_d = torch.empty((M, N), dtype=torch.float32, device=dev)
        for t in (a_d, b_d, c_d):
            t.record_stream(compute)
        c_d.record_stream(s_out)
        bounds = [M * p // P for p in range(P + 1)]
        with torch.cuda.stream(s_in):
            b_d.copy_(b, non_blocking=True)
        done_in = []
        for p in range(P):
            r0, r1 = bounds[p], bounds[p + 1]
            with torch.cuda.stream(s_in):
                if P == 1:
                    a_d.copy_(a, non_blocking=True)
                else:
                    a_d[r0:r1].copy_(a[r0:r1], non_blocking=True)
                if beta != 0.0:
                    c_d[r0:r1].copy_(out[r0:r1], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
            done_in.append(e)
        for p in range(P):
            r0, r1 = bounds[p], bounds[p + 1]
            compute.wait_event(done_in[p])
            if r1 > r0:
                gemm_into(a_d[r0:r1], b_d, c_d[r0:r1], alpha, beta, fp32_mode=fp32_mode)
            e = torch.cuda.Event()
            e.record(compute)
            s_out.wait_event(e)
            with torch.cuda.stream(s_out):
                out[r0:r1].copy_(c_d[r0:r1], non_blocking=True)
        done = torch.cuda.Event()
        done.record(s_out)
    lo, hi = _host_span(out)
    _pending.setdefault(dev.index, []).append((lo, hi, done))
    return HostGemm(out, done)


def gemm(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
         alpha: float = 1.0, beta: float = 0.0, fp32_mode: str | None = None,
         panels: int | None = None) -> torch.Tensor:
    """C = alpha * a @ b + beta * out with fp32 accumulation and output.

    CUDA inputs: computed on the current stream, returned on the GPU (as
    gemm_into).

    CPU inputs: gemm_async(...).wait(): the result lands in host memory
    (`out`, a pinned float32 (M, N) tensor, allocated if not given) and the
    call returns once it is there."""
    if a.is_cuda:
        if out is None:
            out = torch.empty((a.shape[0], b.shape[1]), dtype=torch.float32, device=a.device)
        return gemm_into(a, b, out, alpha, beta, fp32_mode=fp32_mode)
    return gemm_async(a, b, out, alpha, beta, fp32_mode, panels).wait()
