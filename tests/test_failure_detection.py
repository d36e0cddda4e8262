"""Failure detection without a GPU fault.

Every mbarrier wait in the kernels has a time limit. gemm14_debug_inject makes
the next call's producer skip its first shared-memory stage -- a barrier that
nothing will ever complete -- and shortens the wait limit. The kernel must
then report GEMM14_ERR_TIMEOUT through the device error word, end on its own
well within a few seconds, and leave the CUDA context usable.
"""
import time

import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import _lib, inputs

from gpu_util import oracle_check, oracle_check_ex, run_abi, run_ex


def test_inject_rejects_unknown_modes():
    g14.load()
    assert g14.debug_inject(7) == _lib.GEMM14_ERR_INVALID_ARG
    assert g14.debug_inject(0) == _lib.GEMM14_OK


def test_injection_is_consumed_by_the_next_call_even_if_invalid():
    g14.load()
    assert g14.debug_inject(1, 1000) == 0
    # an invalid call consumes the request without touching CUDA
    assert g14.gemm_f32(-1, 1, 1, 0, 1, 0, 1, 0, 1, None, check=False) == 1
    # M == 0: a valid no-op that would have carried a leftover request
    assert g14.gemm_f32(0, 4, 4, 0, 4, 0, 4, 0, 4, None, check=False) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("dt,soft", [("f32", False), ("f32", True), ("bf16", False),
                                     ("bf16", True), ("f16", False)])
def test_expired_wait_reports_timeout_and_context_survives(oracle_mod, dt, soft):
    # fp32: enough 128 x 256 tiles for the large kernel (the small-product
    # kernel has no mbarrier wait to expire, below)
    M, N, K = (2048, 2048, 200) if dt == "f32" else (300, 520, 200)
    A, B = inputs.make(M, N, K, dt, "uniform", 1.0, seed=31)
    lda = K + 1 if soft else (K + 7) // 8 * 8
    ldb = N + 1 if soft else (N + 7) // 8 * 8
    s = torch.cuda.current_stream()
    assert g14.check_device_error(s.cuda_stream) == 0
    assert g14.debug_inject(1, 20_000_000) == 0  # 20 ms per wait
    t0 = time.perf_counter()
    run_abi(A, B, lda=lda, ldb=ldb, check_err=False)
    st = g14.check_device_error(s.cuda_stream)
    elapsed = time.perf_counter() - t0
    assert st == _lib.GEMM14_ERR_TIMEOUT, g14.status_string(st)
    assert elapsed < 10.0
    # the error word was read and cleared; the context still computes correctly
    assert g14.check_device_error(s.cuda_stream) == 0
    C = run_abi(A, B, lda=lda, ldb=ldb)
    oracle_check(oracle_mod, A, B, C)


@pytest.mark.gpu
@pytest.mark.parametrize("dt,ta,tb,soft_a,soft_b", [
    ("f32", 0, 1, False, False),   # B stored N x K: tiles transposed in shared memory
    ("f32", 1, 1, False, False),
    ("bf16", 0, 0, True, False),   # A by the software loader, B by TMA in the same stages
    ("bf16", 0, 1, False, True),   # the reverse, B stored N x K
])
def test_expired_wait_with_transposes_and_mixed_loaders(oracle_mod, dt, ta, tb, soft_a, soft_b):
    """The same expired wait in the variants with their own stage bookkeeping:
    the fp32 kernel's three-stage ring with transposed B buffers (a bounded
    hand-over barrier per buffer), and the one-SM tensor-core kernel with one
    operand by TMA and the other by the software loader (two producers per
    stage, warp 0's TMA loads drained on abort)."""
    M, N, K = (2048, 2048, 200) if dt == "f32" else (300, 520, 200)
    A, B = inputs.make(M, N, K, dt, "uniform", 1.0, seed=33 + 2 * ta + tb)
    q = 4 if dt == "f32" else 8
    a_cols, b_cols = (M if ta else K), (K if tb else N)
    lda = a_cols + 1 if soft_a else -(-a_cols // q) * q
    ldb = b_cols + 1 if soft_b else -(-b_cols // q) * q
    s = torch.cuda.current_stream()
    assert g14.check_device_error(s.cuda_stream) == 0
    assert g14.debug_inject(1, 20_000_000) == 0
    t0 = time.perf_counter()
    run_ex(A, B, ta, tb, lda=lda, ldb=ldb, check_err=False)
    st = g14.check_device_error(s.cuda_stream)
    assert st == _lib.GEMM14_ERR_TIMEOUT, g14.status_string(st)
    assert time.perf_counter() - t0 < 10.0
    assert g14.check_device_error(s.cuda_stream) == 0
    C = run_ex(A, B, ta, tb, lda=lda, ldb=ldb)
    oracle_check_ex(oracle_mod, A, B, C, ta, tb)


@pytest.mark.gpu
def test_small_product_kernel_consumes_the_request(oracle_mod):
    """The fp32 small-product kernel synchronises through hardware barriers
    (block and cluster), with no mbarrier wait that a skipped stage could
    leave open: an injected fault is consumed by its call, which computes
    the product as usual, and the next call is unaffected."""
    M, N, K = 300, 520, 200
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=32)
    st, plan = g14.plan(g14.GEMM14_DTYPE_F32, M, N, K, 1 << 16, K, 1 << 16, N, 1 << 16, N,
                        torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan.kernel == 6
    s = torch.cuda.current_stream()
    assert g14.debug_inject(1, 20_000_000) == 0
    C = run_abi(A, B)
    assert g14.check_device_error(s.cuda_stream) == 0
    oracle_check(oracle_mod, A, B, C)
