"""GPU tests of the public tensor API's host path: CPU tensors in, the result
in (pinned) host memory, with row panels pipelined over three streams."""
import numpy as np
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import TOL, oracle_check, oracle_check_ex

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("panels", [1, 2, 3, 4, 7])
def test_panels_bf16(oracle_mod, panels):
    """Any panel split is within the bound (a panel's tile count decides its
    stream-K split, so the last bits may vary between splits); one panel is
    the device call itself, bit for bit."""
    M, N, K = 1000, 700, 300
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.1, seed=41)
    got = g14.gemm(A, B, panels=panels)
    assert got.device.type == "cpu" and got.is_pinned()
    oracle_check(oracle_mod, A, B, got)
    if panels == 1:
        want = g14.gemm(A.cuda(), B.cuda())
        torch.cuda.synchronize()
        assert torch.equal(got, want.cpu())


@pytest.mark.parametrize("panels", [1, 4])
def test_panels_f32_within_bound(oracle_mod, panels):
    M, N, K = 1100, 600, 257
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=42)
    out = torch.full((M, N), float("nan"), pin_memory=True)
    got = g14.gemm(A, B, out=out, panels=panels)
    assert got.data_ptr() == out.data_ptr()
    oracle_check(oracle_mod, A, B, got)


def test_default_panels_on_a_large_product(oracle_mod):
    """2048 x 1024 x 1100 with the library's own panel split."""
    M, N, K = 2048, 1024, 1100
    A, B = inputs.make(M, N, K, "bf16", "normal", 0.03, seed=43)
    got = g14.gemm(A, B)
    rows = np.arange(0, M, 37)
    oracle_check(oracle_mod, A, B, got, rows=rows)


def test_host_alpha_beta_and_transposed_views(oracle_mod):
    M, N, K = 1500, 400, 200
    A, B = inputs.make(M, N, K, "f32", "normal", 0.3, seed=44)
    C0 = torch.from_numpy(np.random.default_rng(45).standard_normal((M, N)).astype(np.float32))
    out = C0.clone().pin_memory()
    g14.gemm(A, B, out=out, alpha=-2.0, beta=0.5, panels=3)
    oracle_check_ex(oracle_mod, A, B, out, 0, 0, -2.0, 0.5, C0)
    # a transposed host view of A: one panel, the same product
    At = A.t().contiguous()
    got = g14.gemm(At.t(), B)
    oracle_check(oracle_mod, A, B, got)


@pytest.mark.parametrize("mode", ["3xtf32", "tf32"])
@pytest.mark.parametrize("panels", [1, 2, 3])
def test_host_tf32_mode(oracle_mod, mode, panels):
    """The host-buffer path gives the TF32 modes the room for their K-major
    copies and lo parts, so each panel runs on the pair kernel: 3xTF32 within
    the fp32 bound, TF32 within 4e-3 of the fp32 inputs' product."""
    M, N, K = 1200, 512, 320
    A, B = inputs.make(M, N, K, "f32", "uniform", 1.0, seed=46)
    got = g14.gemm(A, B, fp32_mode=mode, panels=panels)
    if mode == "3xtf32":
        oracle_check(oracle_mod, A, B, got)
    else:
        ref, refabs = oracle_mod.gemm(A.numpy(), B.numpy())
        ok, worst = oracle_mod.within_bound(got.numpy(), ref, refabs, 4e-3)
        assert ok, worst
    # a stored transpose of B (N x K), read through a strided view
    Bt = B.t().contiguous().t()
    got_t = g14.gemm(A, Bt, fp32_mode=mode, panels=panels)
    if mode == "3xtf32":
        oracle_check(oracle_mod, A, B, got_t)
    else:
        ok, worst = oracle_mod.within_bound(got_t.numpy(), ref, refabs, 4e-3)
        assert ok, worst


def test_host_degenerate_sizes():
    A = torch.zeros((0, 5))
    B = torch.zeros((5, 3))
    assert g14.gemm(A, B).shape == (0, 3)
    A, B = torch.zeros((4, 0)), torch.zeros((0, 3))
    got = g14.gemm(A, B)
    assert torch.equal(got, torch.zeros((4, 3)))


def test_async_products_in_flight_match_the_blocking_call():
    """Several products issued with gemm_async before any is waited for (their
    copies and kernels overlap one another): each result has the bits of the
    same product run through the blocking call."""
    cases = [(3000, 520, 700, "bf16", 4), (1500, 1024, 512, "f32", 2), (300, 200, 100, "f16", 1),
             (4096, 256, 1024, "bf16", 8), (2048, 300, 257, "f32", 3)]
    ins = [inputs.make(M, N, K, dt, "normal", 0.1, seed=50 + i)
           for i, (M, N, K, dt, _) in enumerate(cases)]
    hs = [g14.gemm_async(A, B, panels=P) for (A, B), (_, _, _, _, P) in zip(ins, cases)]
    got = [h.wait() for h in hs]
    for (A, B), (_, _, _, _, P), C in zip(ins, cases, got):
        assert torch.equal(C, g14.gemm(A, B, panels=P))


def test_async_result_fed_back_as_an_operand():
    """The second product reads the first one's host result before the caller
    waited for it: the library orders the two (exact integer products)."""
    M, N, K = 4096, 512, 1024
    A, B = inputs.make_integer(M, N, K, 3, "f32", seed=61)
    W = torch.from_numpy(np.random.default_rng(62).integers(-1, 2, (N, 64)).astype(np.float32))
    out1 = torch.full((M, N), float("nan"), pin_memory=True)
    h1 = g14.gemm_async(A, B, out=out1, panels=4)
    h2 = g14.gemm_async(out1, W, panels=4)
    C1 = A.double() @ B.double()
    assert torch.equal(h2.wait().double(), C1 @ W.double())
    assert torch.equal(h1.wait().double(), C1)


def test_async_accumulations_into_one_out():
    """Two products with beta = 1 into the same pinned out, both in flight:
    the second sends out to the GPU only after the first's result is back."""
    M, N, K = 2048, 512, 512
    A1, B1 = inputs.make_integer(M, N, K, 2, "f32", seed=63)
    A2, B2 = inputs.make_integer(M, N, K, 2, "f32", seed=64)
    C0 = torch.from_numpy(np.random.default_rng(65).integers(-9, 10, (M, N)).astype(np.float32))
    out = C0.clone().pin_memory()
    g14.gemm_async(A1, B1, out=out, beta=1.0, panels=2)
    g14.gemm_async(A2, B2, out=out, beta=1.0, panels=4).wait()
    want = C0.double() + A1.double() @ B1.double() + A2.double() @ B2.double()
    assert torch.equal(out.double(), want)


def test_gemm_async_takes_host_tensors_only():
    with pytest.raises(ValueError):
        g14.gemm_async(torch.ones(4, 4, device="cuda"), torch.ones(4, 4, device="cuda"))


def _padded_host(x: torch.Tensor, ld: int, fill: float = 0.0) -> tuple[torch.Tensor, torch.Tensor]:
    rows, cols = x.shape
    buf = torch.full((max(rows, 1) * ld + 8,), fill, dtype=x.dtype).pin_memory()
    view = buf[:rows * ld].view(rows, ld)[:, :cols]
    view.copy_(x)
    return buf, view


@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_c_abi_host_entry_pitched_and_transposed(oracle_mod, dt, ta, tb):
    """gemm14_gemm_host on raw host pointers with padded pitches, stored
    transposes and odd 16-bit row lengths (the device copies are re-pitched
    to 16 bytes), against the oracle; then waited twice."""
    M, N, K = 777, 301, 259
    A, B = inputs.make(M, N, K, dt, "normal", 0.2, seed=70 + 2 * ta + tb)
    As = A.t().contiguous() if ta else A
    Bs = B.t().contiguous() if tb else B
    abuf, a = _padded_host(As, As.shape[1] + 3)
    bbuf, b = _padded_host(Bs, Bs.shape[1] + 5)
    cbuf, c = _padded_host(torch.full((M, N), float("nan")), N + 7, fill=float("nan"))
    code = {"f32": g14.GEMM14_DTYPE_F32, "bf16": g14.GEMM14_DTYPE_BF16}[dt]
    t = g14.gemm_host(code, ta, tb, M, N, K, 1.0, a.data_ptr(), a.stride(0), b.data_ptr(),
                      b.stride(0), 0.0, c.data_ptr(), c.stride(0), panels=3)
    assert g14.host_wait(t) == 0
    assert g14.host_wait(t) == 0
    oracle_check(oracle_mod, A, B, c.clone())
    # the padding of C is untouched
    assert torch.isnan(cbuf[:M * (N + 7)].view(M, N + 7)[:, N:]).all()


def test_c_abi_host_entry_degenerate_calls():
    P = torch.zeros(64, pin_memory=True)
    # M == 0: nothing to do, a ticket all the same
    t = g14.gemm_host(g14.GEMM14_DTYPE_F32, 0, 0, 0, 4, 4, 1.0, P.data_ptr(), 4, P.data_ptr(), 4,
                      0.0, P.data_ptr(), 4)
    assert t > 0 and g14.host_wait(t) == 0
    # K == 0: C = beta * C (beta 0.5), sent in and back
    C = torch.arange(12, dtype=torch.float32).view(3, 4).pin_memory()
    t = g14.gemm_host(g14.GEMM14_DTYPE_BF16, 0, 0, 3, 4, 0, 1.0, None, 1, None, 4, 0.5,
                      C.data_ptr(), 4)
    assert g14.host_wait(t) == 0
    assert torch.equal(C, torch.arange(12, dtype=torch.float32).view(3, 4) * 0.5)
    assert g14.host_synchronize() == 0


def test_host_calls_from_several_threads():
    """Four threads issue and wait for host-buffer products at the same time
    (ctypes releases the GIL around each call): each result is the bits of
    the same product issued alone."""
    import threading
    cases = [inputs.make(700 + 64 * t, 300 + 32 * t, 257, "f32", "normal", 0.2, seed=80 + t)
             for t in range(4)]
    want = [g14.gemm(A, B) for A, B in cases]
    got = [[None] * 5 for _ in range(4)]
    errors = []

    def work(t):
        try:
            A, B = cases[t]
            hs = [g14.gemm_async(A, B) for _ in range(5)]
            for i, h in enumerate(hs):
                got[t][i] = h.wait()
        except Exception as e:  # reported by the main thread
            errors.append(repr(e))

    threads = [threading.Thread(target=work, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    for t in range(4):
        for i in range(5):
            assert torch.equal(got[t][i], want[t]), (t, i)
