"""gemm_bf16_f32acc_noalloc: the product for callers that may not allocate
device memory (a framework pool that owns the GPU's memory, plug-ins barred
from the allocator, latency-critical code that cannot take cudaMalloc's
device synchronisation). Its stream-K scratch is a fixed array inside the
library instead of a caller workspace.

Called through the C ABI and checked against the allocating entry point,
gemm_bf16_f32acc, within the bf16 bound the other tests use, on two calls in
a row. This file is collected last on purpose, and passes alone in a fresh
process as well as after the other tests.
"""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import _lib, inputs

pytestmark = pytest.mark.gpu

TOL = 4e-3  # |C - C_ref| <= TOL * (|A||B|)_ij for 16-bit inputs


def _run(fn, A, B):
    M, K = A.shape
    _, N = B.shape
    a, b = A.cuda(), B.cuda()
    c = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.current_stream()
    st = fn(M, N, K, a.data_ptr(), K, b.data_ptr(), N, c.data_ptr(), N, s.cuda_stream,
            check=False)
    assert g14.check_device_error(s.cuda_stream) == 0
    torch.cuda.synchronize()
    return st, c.cpu()


# (M, N, K): products the one-SM kernel splits over all SMs (2 tiles of
# 128 x 64, and 8 tiles of 128 x 128), so the built-in scratch is used.
@pytest.mark.parametrize("M,N,K", [(256, 64, 8192), (1000, 100, 3000)])
def test_no_alloc_matches_allocating_entry_point(oracle_mod, M, N, K):
    assert g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, M, N, K, 0) > 0  # needs scratch
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5, seed=M + N + K)
    _, Cabs = oracle_mod.gemm(inputs.host_view(A), inputs.host_view(B), "bf16")
    st, want = _run(g14.gemm_bf16_f32acc, A, B)
    assert st == 0
    results = []
    for _ in range(2):  # two calls in a row share the built-in scratch
        st, got = _run(g14.gemm_bf16_f32acc_noalloc, A, B)
        assert st == 0, g14.last_error_string()
        diff = np.abs(got.numpy().astype(np.float64) - want.numpy().astype(np.float64))
        assert not np.isnan(got.numpy()).any()
        assert np.all(diff <= TOL * Cabs), float(np.max(diff / np.maximum(Cabs, 1e-30)))
        results.append(got)
    assert torch.equal(results[0], results[1])


def test_no_alloc_without_scratch_is_the_plain_product():
    # a wide product runs on the CTA-pair kernel; the no-alloc entry runs it
    # unsplit (its split would need more than the built-in scratch), exactly
    # as gemm_bf16_f32acc does
    A, B = inputs.make(512, 512, 512, "bf16", "normal", 0.05, seed=7)
    st, plan = g14.plan(g14.GEMM14_DTYPE_BF16, 512, 512, 512, 1 << 16, 512, 1 << 16, 512,
                        1 << 16, 512, 0 or 152)
    assert st == 0 and plan.kernel == 3
    _, want = _run(g14.gemm_bf16_f32acc, A, B)
    st, got = _run(g14.gemm_bf16_f32acc_noalloc, A, B)
    assert st == 0 and torch.equal(got, want)


def test_no_alloc_rejects_products_beyond_its_scratch():
    # M <= 128 with wide N: 256-column tiles on one SM each, split over all
    # SMs -- about 20 MB of scratch on 152 SMs, more than the 16 MiB built in
    M, N, K = 64, 2048, 4096
    need = g14.workspace_bytes(g14.GEMM14_DTYPE_BF16, M, N, K, 0)
    assert need > 16 << 20
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.02, seed=8)
    st, _ = _run(g14.gemm_bf16_f32acc_noalloc, A, B)
    assert st == _lib.GEMM14_ERR_INVALID_ARG
    msg = g14.last_error_string()
    assert "scratch" in msg and str(need) in msg
