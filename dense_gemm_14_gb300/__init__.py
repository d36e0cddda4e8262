"""GB300 (sm_103a) dense GEMM: C = A @ B on row-major matrices.

A thin binding over the C ABI of ``libgemm14.so`` (``include/gemm14.h``). The
three entry points keep their C names and arguments -- sizes, raw device
pointers, leading dimensions and a stream handle -- and only marshal them;
every step of the product runs in the library's CUDA kernels. There is no CPU
fallback: if the library is missing or the GPU is unsupported, calls raise.

``gemm(a, b)`` is the convenience call on torch tensors: CUDA tensors run on
the current stream; CPU tensors are copied through pinned host memory to the
GPU and the result is copied back (the end-to-end path).
"""
from __future__ import annotations

from ._lib import (GEMM14_DTYPE_BF16, GEMM14_DTYPE_F16, GEMM14_DTYPE_F32,
                   GEMM14_DTYPE_F32_3XTF32, GEMM14_DTYPE_TF32, GEMM14_ERR_CUDA,
                   GEMM14_ERR_DEVICE_CHECK, GEMM14_ERR_INVALID_ARG, GEMM14_ERR_TIMEOUT,
                   GEMM14_ERR_UNSUPPORTED_DEVICE, GEMM14_OK, Gemm14Error, Plan,
                   check_device_error, debug_inject, gemm_bf16_f32acc, gemm_bf16_f32acc_ws,
                   gemm_bf16_f32acc_noalloc, gemm_ex, gemm_host, host_synchronize, host_wait, workspace_bytes_ex, gemm_f16_f32acc, gemm_f16_f32acc_ws, gemm_f32,
                   gemm_f32_3xtf32, gemm_f32_ws, gemm_tf32_f32acc, last_error_string, lib_path, load, plan, plan_ex, set_pair_kernel, status_string, version, workspace_bytes)
from .api import HostGemm, gemm, gemm_async, gemm_into

__all__ = [
    "gemm", "gemm_async", "HostGemm", "gemm_into", "gemm_f32", "gemm_bf16_f32acc", "gemm_f16_f32acc", "gemm_f32_ws",
    "gemm_tf32_f32acc", "gemm_f32_3xtf32",
    "gemm_bf16_f32acc_ws", "gemm_f16_f32acc_ws", "gemm_bf16_f32acc_noalloc", "gemm_ex",
    "gemm_host", "host_wait", "host_synchronize", "workspace_bytes_ex", "workspace_bytes",
    "last_error_string", "plan", "plan_ex", "Plan",
    "check_device_error", "debug_inject", "set_pair_kernel", "status_string", "version", "load", "lib_path", "Gemm14Error",
    "GEMM14_DTYPE_F32", "GEMM14_DTYPE_BF16", "GEMM14_DTYPE_F16", "GEMM14_DTYPE_TF32",
    "GEMM14_DTYPE_F32_3XTF32",
    "GEMM14_OK", "GEMM14_ERR_INVALID_ARG", "GEMM14_ERR_UNSUPPORTED_DEVICE", "GEMM14_ERR_CUDA",
    "GEMM14_ERR_TIMEOUT", "GEMM14_ERR_DEVICE_CHECK",
]
