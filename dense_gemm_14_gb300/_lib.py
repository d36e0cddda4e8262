"""ctypes binding of libgemm14.so: the C ABI of include/gemm14.h, argument
marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
_DEFAULT_LIB = os.path.join(_HERE, "_build", "libgemm14.so")

GEMM14_OK = 0
GEMM14_ERR_INVALID_ARG = 1
GEMM14_ERR_UNSUPPORTED_DEVICE = 2
GEMM14_ERR_CUDA = 3
GEMM14_ERR_TIMEOUT = 4
GEMM14_ERR_DEVICE_CHECK = 5

GEMM14_DTYPE_F32 = 0
GEMM14_DTYPE_BF16 = 1
GEMM14_DTYPE_F16 = 2
GEMM14_DTYPE_TF32 = 3
GEMM14_DTYPE_F32_3XTF32 = 4

# Every function the header declares, with (restype, argtypes).
_i64, _vp, _int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
_GEMM_ARGS = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp]


class _Plan(ctypes.Structure):
    _fields_ = [("kernel", _int), ("loader", _int), ("bm", _int), ("bn", _int), ("bk", _int),
                ("stages", _int), ("threads", _int), ("smem_bytes", _int),
                ("vec_store", _int), ("tiles", _i64), ("grid", _int)]


SIGNATURES = {
    "gemm_f32": (_int, _GEMM_ARGS),
    "gemm_bf16_f32acc": (_int, _GEMM_ARGS),
    "gemm_f16_f32acc": (_int, _GEMM_ARGS),
    "gemm_tf32_f32acc": (_int, _GEMM_ARGS),
    "gemm_f32_3xtf32": (_int, _GEMM_ARGS),
    "gemm14_status_string": (ctypes.c_char_p, [_int]),
    "gemm14_last_error_string": (ctypes.c_char_p, []),
    "gemm14_check_device_error": (_int, [_vp]),
    "gemm14_plan_gemm": (_int, [_int, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _int,
                                ctypes.POINTER(_Plan)]),
    "gemm14_version": (_int, []),
    "gemm14_debug_inject": (_int, [_int, ctypes.c_uint64]),
    "gemm14_set_pair_kernel": (_int, [_int]),
    "gemm_f32_ws": (_int, _GEMM_ARGS[:9] + [_vp, ctypes.c_size_t, _vp]),
    "gemm_bf16_f32acc_ws": (_int, _GEMM_ARGS[:9] + [_vp, ctypes.c_size_t, _vp]),
    "gemm_f16_f32acc_ws": (_int, _GEMM_ARGS[:9] + [_vp, ctypes.c_size_t, _vp]),
    "gemm14_workspace_bytes": (ctypes.c_size_t, [_int, _i64, _i64, _i64, _int]),
    "gemm_bf16_f32acc_noalloc": (_int, _GEMM_ARGS),
    "gemm14_gemm_ex": (_int, [_int, _int, _int, _i64, _i64, _i64, ctypes.c_float, _vp, _i64,
                              _vp, _i64, ctypes.c_float, _vp, _i64, _vp, ctypes.c_size_t, _vp]),
    "gemm14_plan_gemm_ex": (_int, [_int, _int, _int, _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                                   _vp, _i64, _int, ctypes.POINTER(_Plan)]),
    "gemm14_gemm_host": (_int, [_int, _int, _int, _i64, _i64, _i64, ctypes.c_float, _vp, _i64,
                                _vp, _i64, ctypes.c_float, _vp, _i64, _int,
                                ctypes.POINTER(ctypes.c_uint64)]),
    "gemm14_host_wait": (_int, [ctypes.c_uint64]),
    "gemm14_workspace_bytes_ex": (ctypes.c_size_t, [_int, _int, _int, _i64, _i64, _i64, _vp, _i64,
                                                    _vp, _i64, _vp, _i64, _int]),
    "gemm14_host_synchronize": (_int, []),
}

_lib = None
_lock = threading.Lock()


class Gemm14Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == GEMM14_ERR_CUDA and _lib is not None:
            detail = ": " + _lib.gemm14_last_error_string().decode(errors="replace")
        super().__init__(f"{where} failed: {status_string(status)} ({status}){detail}")


def lib_path() -> str:
    return os.environ.get("GEMM14_LIB", _DEFAULT_LIB)


def load():
    """Loads libgemm14.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"{path} is missing: build it with `python -m dense_gemm_14_gb300.build` "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().gemm14_status_string(int(status)).decode()


def version() -> int:
    return int(load().gemm14_version())


def _call(name: str, M, N, K, A, lda, B, ldb, C, ldc, stream) -> int:
    return int(getattr(load(), name)(M, N, K, A, lda, B, ldb, C, ldc, stream))


def gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream=None, check=True) -> int:
    """C ABI gemm_f32 on raw device pointers (ints); raises on a non-OK status if check."""
    st = _call("gemm_f32", M, N, K, A, lda, B, ldb, C, ldc, stream)
    if check and st:
        raise Gemm14Error(st, "gemm_f32")
    return st


def gemm_bf16_f32acc(M, N, K, A, lda, B, ldb, C, ldc, stream=None, check=True) -> int:
    """C ABI gemm_bf16_f32acc on raw device pointers (ints)."""
    st = _call("gemm_bf16_f32acc", M, N, K, A, lda, B, ldb, C, ldc, stream)
    if check and st:
        raise Gemm14Error(st, "gemm_bf16_f32acc")
    return st


def gemm_f16_f32acc(M, N, K, A, lda, B, ldb, C, ldc, stream=None, check=True) -> int:
    """C ABI gemm_f16_f32acc on raw device pointers (ints)."""
    st = _call("gemm_f16_f32acc", M, N, K, A, lda, B, ldb, C, ldc, stream)
    if check and st:
        raise Gemm14Error(st, "gemm_f16_f32acc")
    return st


def gemm_tf32_f32acc(M, N, K, A, lda, B, ldb, C, ldc, stream=None, check=True) -> int:
    """C ABI gemm_tf32_f32acc: fp32 inputs rounded to tf32 on the tensor cores."""
    st = _call("gemm_tf32_f32acc", M, N, K, A, lda, B, ldb, C, ldc, stream)
    if check and st:
        raise Gemm14Error(st, "gemm_tf32_f32acc")
    return st


def gemm_f32_3xtf32(M, N, K, A, lda, B, ldb, C, ldc, stream=None, check=True) -> int:
    """C ABI gemm_f32_3xtf32: fp32 inputs, split tf32 arithmetic on the tensor
    cores within the fp32 bound."""
    st = _call("gemm_f32_3xtf32", M, N, K, A, lda, B, ldb, C, ldc, stream)
    if check and st:
        raise Gemm14Error(st, "gemm_f32_3xtf32")
    return st


def _call_ws(name, M, N, K, A, lda, B, ldb, C, ldc, ws, ws_bytes, stream, check):
    st = int(getattr(load(), name)(M, N, K, A, lda, B, ldb, C, ldc, ws, ws_bytes, stream))
    if check and st:
        raise Gemm14Error(st, name)
    return st


def gemm_f32_ws(M, N, K, A, lda, B, ldb, C, ldc, workspace, workspace_bytes, stream=None,
                check=True) -> int:
    """C ABI gemm_f32_ws: gemm_f32 with a device workspace (stream-K schedule)."""
    return _call_ws("gemm_f32_ws", M, N, K, A, lda, B, ldb, C, ldc, workspace,
                    workspace_bytes, stream, check)


def gemm_bf16_f32acc_ws(M, N, K, A, lda, B, ldb, C, ldc, workspace, workspace_bytes,
                        stream=None, check=True) -> int:
    """C ABI gemm_bf16_f32acc_ws."""
    return _call_ws("gemm_bf16_f32acc_ws", M, N, K, A, lda, B, ldb, C, ldc, workspace,
                    workspace_bytes, stream, check)


def gemm_f16_f32acc_ws(M, N, K, A, lda, B, ldb, C, ldc, workspace, workspace_bytes,
                       stream=None, check=True) -> int:
    """C ABI gemm_f16_f32acc_ws."""
    return _call_ws("gemm_f16_f32acc_ws", M, N, K, A, lda, B, ldb, C, ldc, workspace,
                    workspace_bytes, stream, check)


def gemm_bf16_f32acc_noalloc(M, N, K, A, lda, B, ldb, C, ldc, stream=None, check=True) -> int:
    """C ABI gemm_bf16_f32acc_noalloc: gemm_bf16_f32acc for callers that may
    not allocate device memory; its stream-K scratch is a fixed array inside
    the library (see include/gemm14.h for the limit)."""
    st = _call("gemm_bf16_f32acc_noalloc", M, N, K, A, lda, B, ldb, C, ldc, stream)
    if check and st:
        raise Gemm14Error(st, "gemm_bf16_f32acc_noalloc")
    return st


def gemm_ex(dtype: int, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
            workspace=None, workspace_bytes=0, stream=None, check=True) -> int:
    """C ABI gemm14_gemm_ex: C = alpha * op(A) op(B) + beta * C on raw device
    pointers, op(A) = A stored M x K (transa 0) or its transpose stored K x M
    (transa 1), likewise B."""
    st = int(load().gemm14_gemm_ex(dtype, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta,
                                   C, ldc, workspace, workspace_bytes, stream))
    if check and st:
        raise Gemm14Error(st, "gemm14_gemm_ex")
    return st


def workspace_bytes_ex(dtype: int, transa, transb, M, N, K, A, lda, B, ldb, C, ldc,
                       sm_count: int = 0) -> int:
    """C ABI gemm14_workspace_bytes_ex: workspace for these exact operands,
    re-pitching of operands TMA cannot read included."""
    return int(load().gemm14_workspace_bytes_ex(dtype, transa, transb, M, N, K, A, lda, B, ldb,
                                                C, ldc, sm_count))


def gemm_host(dtype: int, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
              panels: int = 0, check=True) -> int:
    """C ABI gemm14_gemm_host on HOST pointers: enqueues the product and returns
    its ticket (for host_wait). Raises Gemm14Error on a failed call when check."""
    t = ctypes.c_uint64(0)
    st = int(load().gemm14_gemm_host(dtype, transa, transb, M, N, K, alpha, A, lda, B, ldb, beta,
                                     C, ldc, panels, ctypes.byref(t)))
    if st:
        if check:
            raise Gemm14Error(st, "gemm14_gemm_host")
        return -st
    return t.value


def host_wait(ticket: int, check=True) -> int:
    """C ABI gemm14_host_wait: blocks until that product's C is in host memory."""
    st = int(load().gemm14_host_wait(ticket))
    if check and st:
        raise Gemm14Error(st, "gemm14_host_wait")
    return st


def host_synchronize(check=True) -> int:
    """C ABI gemm14_host_synchronize: waits for every host-buffer product in flight."""
    st = int(load().gemm14_host_synchronize())
    if check and st:
        raise Gemm14Error(st, "gemm14_host_synchronize")
    return st


def last_error_string() -> str:
    """Text of the last failure seen by this thread (the C ABI's message)."""
    return load().gemm14_last_error_string().decode(errors="replace")


def workspace_bytes(dtype: int, M, N, K, sm_count: int = 0) -> int:
    """Workspace the *_ws call needs for the stream-K schedule (0: none)."""
    return int(load().gemm14_workspace_bytes(dtype, M, N, K, sm_count))


def debug_inject(fault: int, wait_limit_ns: int = 0) -> int:
    """Failure-detection hook: the next call on this thread runs with `fault`
    (1 = the producer never loads its first stage) and the given wait limit."""
    return int(load().gemm14_debug_inject(fault, wait_limit_ns))


def set_pair_kernel(enable: bool) -> bool:
    """Allows (default) or forbids the CTA-pair tensor-core kernel; returns the
    previous setting. Results are identical either way."""
    return bool(load().gemm14_set_pair_kernel(1 if enable else 0))


def check_device_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return int(load().gemm14_check_device_error(stream))


@dataclass
class Plan:
    kernel: int
    loader: int
    bm: int
    bn: int
    bk: int
    stages: int
    threads: int
    smem_bytes: int
    vec_store: int
    tiles: int
    grid: int


def plan(dtype: int, M, N, K, A, lda, B, ldb, C, ldc, sm_count: int):
    """Host-only launch plan (no CUDA call). Returns (status, Plan)."""
    p = _Plan()
    st = int(load().gemm14_plan_gemm(dtype, M, N, K, A, lda, B, ldb, C, ldc, sm_count,
                                     ctypes.byref(p)))
    return st, Plan(**{f: getattr(p, f) for f, _ in _Plan._fields_})


def plan_ex(dtype: int, transa, transb, M, N, K, A, lda, B, ldb, C, ldc, sm_count: int):
    """Host-only launch plan of a gemm_ex call. Returns (status, Plan)."""
    p = _Plan()
    st = int(load().gemm14_plan_gemm_ex(dtype, transa, transb, M, N, K, A, lda, B, ldb, C, ldc,
                                        sm_count, ctypes.byref(p)))
    return st, Plan(**{f: getattr(p, f) for f, _ in _Plan._fields_})
