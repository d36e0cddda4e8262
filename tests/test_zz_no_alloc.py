"""gemm_bf16_f32acc_noalloc: the product for callers that may not allocate
device memory (a framework pool that owns the GPU's memory, plug-ins barred
from the allocator, latency-critical code that cannot take cudaMalloc's
device synchronisation). Its stream-K scratch is a fixed array inside the
library instead of a caller workspace.

Each product is called through the C ABI twice in a row (the calls share the
built-in scratch) and checked element by element against the oracle, within
the bf16 bound the other tests use, and against the allocating entry point
gemm_bf16_f32acc within the same bound. This file is collected last on
purpose, and passes alone in a fresh process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

TOL = 4e-3  # |C - C_ref| <= TOL * (|A||B|)_ij for 16-bit inputs
SCRATCH_BYTES = 20 << 20  # the array built into the library


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _run(fn, A, B, lda=None):
    """C = A B through entry point fn, A copied with row pitch lda."""
    M, K = A.shape
    _, N = B.shape
    lda = lda or K
    abuf = torch.zeros(M * lda + 8, dtype=A.dtype, device="cuda")
    abuf[:M * lda].view(M, lda)[:, :K].copy_(A.cuda())
    b = B.cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    st = fn(M, N, K, abuf.data_ptr(), lda, b.data_ptr(), N, c.data_ptr(), N, s.cuda_stream,
            check=False)
    assert g14.check_device_error(s.cuda_stream) == 0
    torch.cuda.synchronize()
    return st, c.cpu()


def _within(got, ref, Cabs, what):
    got = got.numpy().astype(np.float64)
    assert not np.isnan(got).any(), what
    diff = np.abs(got - ref)
    assert np.all(diff <= TOL * Cabs), (what, float(np.max(diff / np.maximum(Cabs, 1e-30))))


def _check_twice(oracle_mod, A, B, lda=None):
    """Two no-alloc calls in a row, each against the oracle and against the
    allocating entry point; the two results are bit-identical."""
    C_ref, Cabs = oracle_mod.gemm(inputs.host_view(A), inputs.host_view(B), "bf16")
    st, plain = _run(g14.gemm_bf16_f32acc, A, B, lda)
    assert st == 0
    _within(plain, C_ref, Cabs, "gemm_bf16_f32acc against the oracle")
    results = []
    for call in range(2):
        st, got = _run(g14.gemm_bf16_f32acc_noalloc, A, B, lda)
        assert st == 0, g14.last_error_string()
        _within(got, C_ref, Cabs, f"no-alloc call {call} against the oracle")
        diff = np.abs(got.numpy().astype(np.float64) - plain.numpy().astype(np.float64))
        assert np.all(diff <= TOL * Cabs), f"no-alloc call {call} against gemm_bf16_f32acc"
        results.append(got)
    assert torch.equal(results[0], results[1])


# (M, N, K): products the one-SM kernel splits over all SMs (2 tiles of
# 128 x 64, and 8 tiles of 128 x 128), so the built-in scratch is used.
@pytest.mark.parametrize("M,N,K", [(256, 64, 8192), (1000, 100, 3000)])
def test_no_alloc_matches_oracle_and_allocating_entry_point(oracle_mod, M, N, K):
    assert g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, M, N, K, _sms()) > 0  # needs scratch
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=M + N + K)
    _check_twice(oracle_mod, A, B)


def test_no_alloc_pair_kernel_split(oracle_mod):
    # 4 tiles of 256 x 256 with long k: the CTA-pair kernel splits them over
    # 16 clusters, its slots in the built-in scratch
    M, N, K = 512, 512, 8192
    st, plan = g14.plan(g14.GEMM14_DTYPE_BF16, M, N, K, 1 << 16, K, 1 << 16, N, 1 << 16, N,
                        _sms())
    assert st == 0 and plan.kernel == 3
    assert 0 < g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, M, N, K, _sms()) <= SCRATCH_BYTES
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=9)
    _check_twice(oracle_mod, A, B)


def test_no_alloc_with_the_pair_kernel_off(oracle_mod):
    # with the pair kernel switched off, a wide product runs in 256-column
    # tiles on one SM each; 160 tiles are just over one wave on 152 SMs and
    # are split over all SMs (the largest split, 19.9 MB on 152 SMs)
    M, N, K = 2560, 2048, 512
    prev = g14.set_pair_kernel(False)
    try:
        need = g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, M, N, K, _sms())
        if need > SCRATCH_BYTES:
            pytest.skip(f"{_sms()} SMs: this split needs {need} bytes, beyond the scratch")
        A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=10)
        _check_twice(oracle_mod, A, B)
    finally:
        g14.set_pair_kernel(prev)


def test_no_alloc_odd_pitch(oracle_mod):
    # lda = K + 1 (not a multiple of 8 elements): A cannot be read by TMA as
    # stored, and is re-pitched into the scratch beside the split's region
    M, N, K = 1000, 100, 3000
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=11)
    _check_twice(oracle_mod, A, B, lda=K + 1)


def test_no_alloc_without_scratch_is_the_plain_product():
    # a wide product with few k-blocks: the CTA-pair kernel runs it unsplit,
    # exactly as gemm_bf16_f32acc does
    A, B = inputs.make(512, 512, 512, "bf16", "normal", 0.05, seed=7)
    st, plan = g14.plan(g14.GEMM14_DTYPE_BF16, 512, 512, 512, 1 << 16, 512, 1 << 16, 512,
                        1 << 16, 512, _sms())
    assert st == 0 and plan.kernel == 3
    assert g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, 512, 512, 512, _sms()) == 0
    _, want = _run(g14.gemm_bf16_f32acc, A, B)
    st, got = _run(g14.gemm_bf16_f32acc_noalloc, A, B)
    assert st == 0 and torch.equal(got, want)


def test_no_alloc_rejects_splits_beyond_its_scratch():
    # The largest split is one 128 x 256 fp32 slot (and a flag) per SM, which
    # exceeds the 20 MiB only beyond 159 SMs; on such a GPU the call is
    # rejected with a message naming the bytes needed.
    M, N, K = 64, 2048, 4096
    prev = g14.set_pair_kernel(False)
    try:
        need = g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, M, N, K, _sms())
        if need <= SCRATCH_BYTES:
            pytest.skip(f"{_sms()} SMs: every split fits the built-in scratch ({need} bytes)")
        A, B = inputs.make(M, N, K, "bf16", "normal", 0.02, seed=8)
        st, _ = _run(g14.gemm_bf16_f32acc_noalloc, A, B)
        assert st == _lib.GEMM14_ERR_INVALID_ARG
        msg = g14.last_error_string()
        assert "scratch" in msg and str(need) in msg
    finally:
        g14.set_pair_kernel(prev)
