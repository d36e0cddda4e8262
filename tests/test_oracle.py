"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle -- a transposed
operand, a wrong index or leading dimension, a dropped or repeated k term, a
sign error, a wrong 16-bit decoder, a wrong |A||B| -- fails at least one of
them. None of them re-types the oracle's own loop.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from dense_gemm_14_gb300 import inputs


def f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


# ----------------------------------------------------------------- decoders

def test_decode_f16_all_patterns_match_numpy(oracle_mod):
    """Every binary16 pattern, including subnormals, infinities and NaN, decodes
    like numpy's independent float16 implementation."""
    bits = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    got = oracle_mod.decode(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    m = ~np.isnan(want)
    assert np.array_equal(got[m], want[m])
    assert np.array_equal(np.signbit(got[m]), np.signbit(want[m]))


def test_decode_bf16_all_patterns_match_torch(oracle_mod):
    """Every bfloat16 pattern decodes like torch's bfloat16 -> float32 cast."""
    bits = np.arange(65536, dtype=np.uint16).reshape(256, 256)
    got = oracle_mod.decode(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    m = ~np.isnan(want)
    assert np.array_equal(got[m], want[m])


@pytest.mark.parametrize("bits,value", [
    (0x3C00, 1.0), (0xC000, -2.0), (0x0001, 2.0 ** -24), (0x03FF, 1023 * 2.0 ** -24),
    (0x0400, 2.0 ** -14), (0x7BFF, 65504.0), (0x3555, 0.333251953125),
])
def test_decode_f16_textbook_values(oracle_mod, bits, value):
    got = oracle_mod.decode(np.array([[bits]], dtype=np.uint16), "f16")[0, 0]
    assert got == value


@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x4049, 3.140625), (0x0001, 2.0 ** -133),
    (0x7F7F, 3.3895313892515355e38),
])
def test_decode_bf16_textbook_values(oracle_mod, bits, value):
    got = oracle_mod.decode(np.array([[bits]], dtype=np.uint16), "bf16")[0, 0]
    assert got == value


# ----------------------------------------------------------------- structure

def test_identity_right_and_left(oracle_mod):
    g = np.random.default_rng(1)
    A = f32(g.uniform(-1, 1, (7, 5)))
    C, _ = oracle_mod.gemm(A, f32(np.eye(5)))
    assert np.array_equal(C, A.astype(np.float64))
    B = f32(g.uniform(-1, 1, (5, 9)))
    C, _ = oracle_mod.gemm(f32(np.eye(5)), B)
    assert np.array_equal(C, B.astype(np.float64))


def test_permutation_rows_and_columns(oracle_mod):
    """P @ B permutes the rows of B; A @ Q permutes the columns of A. An operand
    transposed or an index swapped inside the oracle breaks this."""
    g = np.random.default_rng(2)
    perm = g.permutation(6)
    P = np.zeros((6, 6), np.float32)
    P[np.arange(6), perm] = 1
    B = f32(g.uniform(-1, 1, (6, 11)))
    C, _ = oracle_mod.gemm(P, B)
    assert np.array_equal(C, B[perm].astype(np.float64))
    A = f32(g.uniform(-1, 1, (4, 6)))
    Q = np.zeros((6, 6), np.float32)
    Q[perm, np.arange(6)] = 1
    C, _ = oracle_mod.gemm(A, Q)
    assert np.array_equal(C, A[:, perm].astype(np.float64))


def test_selection_non_square(oracle_mod):
    """A @ S with S picking column sel[j] of A into column j (K != N)."""
    g = np.random.default_rng(3)
    A = f32(g.uniform(-1, 1, (5, 8)))
    sel = np.array([7, 0, 3, 3, 1])
    S = np.zeros((8, 5), np.float32)
    S[sel, np.arange(5)] = 1
    C, _ = oracle_mod.gemm(A, S)
    assert np.array_equal(C, A[:, sel].astype(np.float64))


def test_diagonal_scaling_is_one_product(oracle_mod):
    g = np.random.default_rng(4)
    d = f32(g.uniform(-2, 2, 6))
    B = f32(g.uniform(-1, 1, (6, 7)))
    C, _ = oracle_mod.gemm(f32(np.diag(d)), B)
    assert np.array_equal(C, d.astype(np.float64)[:, None] * B.astype(np.float64))


# ----------------------------------------------------------------- exact sums

@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_integer_matrices_exact(oracle_mod, dtype):
    """Integer entries in [-4, 4]: the exact product is the int64 matmul."""
    A_t, B_t = inputs.make_integer(37, 29, 53, 4, dtype=dtype, seed=5)
    A_i = A_t.to(torch.int64).numpy()
    B_i = B_t.to(torch.int64).numpy()
    C, Cabs = oracle_mod.gemm(inputs.host_view(A_t), inputs.host_view(B_t), dtype)
    assert np.array_equal(C, (A_i @ B_i).astype(np.float64))
    assert np.array_equal(Cabs, (np.abs(A_i) @ np.abs(B_i)).astype(np.float64))


def test_closed_forms(oracle_mod):
    M, N, K = 9, 13, 17
    C, Cabs = oracle_mod.gemm(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
    assert np.all(C == K) and np.all(Cabs == K)
    a = (np.arange(M) % 7 + 1).astype(np.float32)
    b = (np.arange(N) % 5 + 1).astype(np.float32)
    A = np.repeat(a[:, None], K, axis=1)
    B = np.repeat(b[None, :], K, axis=0)
    C, _ = oracle_mod.gemm(f32(A), f32(B))
    assert np.array_equal(C, K * np.outer(a, b).astype(np.float64))
    # alternating signs cancel exactly: row i of A = (-1)^k, B = ones
    A = f32(np.tile((-1.0) ** np.arange(16), (3, 1)))
    C, Cabs = oracle_mod.gemm(A, np.ones((16, 4), np.float32))
    assert np.all(C == 0) and np.all(Cabs == 16)


def test_brute_force_tiny_shapes_fraction(oracle_mod):
    """All shapes in {1..4}^3 with dyadic entries k/8: compared with exact
    rational sums (fractions.Fraction), so any rounding, missing term or
    mis-indexing shows."""
    g = np.random.default_rng(6)
    for M, N, K in itertools.product(range(1, 5), repeat=3):
        A = g.integers(-16, 17, (M, K)) / 8.0
        B = g.integers(-16, 17, (K, N)) / 8.0
        C, Cabs = oracle_mod.gemm(f32(A), f32(B))
        for i in range(M):
            for j in range(N):
                exact = sum(Fraction(A[i, k]) * Fraction(B[k, j]) for k in range(K))
                exact_abs = sum(abs(Fraction(A[i, k]) * Fraction(B[k, j])) for k in range(K))
                assert C[i, j] == float(exact)
                assert Cabs[i, j] == float(exact_abs)


def test_empty_inner_dimension_is_zero(oracle_mod):
    C, Cabs = oracle_mod.gemm(np.zeros((3, 0), np.float32), np.zeros((0, 4), np.float32))
    assert C.shape == (3, 4) and np.all(C == 0) and np.all(Cabs == 0)
    C, _ = oracle_mod.gemm(np.zeros((0, 5), np.float32), np.zeros((5, 4), np.float32))
    assert C.shape == (0, 4)


def test_leading_dimension_views(oracle_mod):
    """Strided views (lda > K, ldb > N) give the same result as compact copies."""
    g = np.random.default_rng(7)
    Abig = f32(g.uniform(-1, 1, (10, 20)))
    Bbig = f32(g.uniform(-1, 1, (12, 30)))
    A, B = Abig[:, :12], Bbig[:, 5:19]
    C1, _ = oracle_mod.gemm(A, B)
    C2, _ = oracle_mod.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B))
    assert np.array_equal(C1, C2)


# ----------------------------------------------------------------- library cross-check

@pytest.mark.parametrize("shape", [(64, 96, 128), (257, 129, 300), (512, 64, 513)])
def test_matches_numpy_float64(oracle_mod, shape):
    """numpy's float64 matmul is an independent evaluation of the same sum;
    the two agree to within fp64 rounding of a length-K sum."""
    M, N, K = shape
    A_t, B_t = inputs.make(M, N, K, "f32", "normal", 1.0, seed=8)
    A, B = A_t.numpy(), B_t.numpy()
    C, Cabs = oracle_mod.gemm(A, B)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    assert np.all(np.abs(C - ref) <= 1e-12 * Cabs)
    assert np.array_equal(Cabs, np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))) or \
        np.all(np.abs(Cabs - np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))) <= 1e-12 * Cabs)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_16bit_matches_numpy_on_decoded_values(oracle_mod, dtype):
    A_t, B_t = inputs.make(96, 80, 257, dtype, "normal", 1.0 / 16, seed=9)
    A64 = A_t.to(torch.float64).numpy()
    B64 = B_t.to(torch.float64).numpy()
    C, Cabs = oracle_mod.gemm(inputs.host_view(A_t), inputs.host_view(B_t), dtype)
    assert np.all(np.abs(C - A64 @ B64) <= 1e-12 * Cabs)


def test_entries_agree_with_full_product(oracle_mod):
    A_t, B_t = inputs.make(70, 90, 110, "f32", "uniform", 1.0, seed=10)
    A, B = A_t.numpy(), B_t.numpy()
    C, Cabs = oracle_mod.gemm(A, B)
    g = np.random.default_rng(11)
    rows, cols = g.integers(0, 70, 200), g.integers(0, 90, 200)
    e, ea = oracle_mod.gemm_entries(A, B, rows, cols)
    assert np.array_equal(e, C[rows, cols]) and np.array_equal(ea, Cabs[rows, cols])


def test_thread_count_does_not_change_results(oracle_mod):
    A_t, B_t = inputs.make(65, 33, 129, "f32", "normal", 1.0, seed=12)
    C1, _ = oracle_mod.gemm(A_t.numpy(), B_t.numpy(), threads=1)
    C4, _ = oracle_mod.gemm(A_t.numpy(), B_t.numpy(), threads=4)
    assert np.array_equal(C1, C4)


# ----------------------------------------------------------------- the acceptance check

def test_within_bound_accepts_rounded_oracle_and_rejects_perturbation(oracle_mod):
    A_t, B_t = inputs.make(40, 50, 300, "f32", "uniform", 1.0, seed=13)
    C, Cabs = oracle_mod.gemm(A_t.numpy(), B_t.numpy())
    ok, worst = oracle_mod.within_bound(C.astype(np.float32), C, Cabs, 1e-5)
    assert ok and worst < 1e-7
    bad = C.astype(np.float32).astype(np.float64)
    bad[3, 4] += 2e-5 * Cabs[3, 4]
    ok, _ = oracle_mod.within_bound(bad, C, Cabs, 1e-5)
    assert not ok
    nan = C.copy()
    nan[0, 0] = np.nan
    ok, _ = oracle_mod.within_bound(nan, C, Cabs, 1e-5)
    assert not ok


def test_sequential_fp32_sum_fits_the_fp32_bound(oracle_mod):
    """The fp32 bound 1e-5 * (|A||B|)_ij leaves room for any plain fp32
    summation order: a sequential float32 sum (the worst common order) over
    K = 3072 stays well inside it."""
    A_t, B_t = inputs.make(16, 16, 3072, "f32", "uniform", 1.0, seed=14)
    A, B = A_t.numpy(), B_t.numpy()
    C, Cabs = oracle_mod.gemm(A, B)
    seq = np.zeros((16, 16), np.float32)
    for k in range(3072):
        seq = (seq + np.outer(A[:, k], B[k, :]).astype(np.float32)).astype(np.float32)
    ok, worst = oracle_mod.within_bound(seq, C, Cabs, 1e-5)
    assert ok and worst < 1e-6


def test_inputs_are_seeded_and_shaped():
    A1, B1 = inputs.make_workload("f32_ragged", M=33, N=17, K=9)
    A2, B2 = inputs.make_workload("f32_ragged", M=33, N=17, K=9)
    assert torch.equal(A1, A2) and torch.equal(B1, B2)
    assert A1.shape == (33, 9) and B1.shape == (9, 17) and A1.dtype == torch.float32
    A, B = inputs.make_workload("bf16_8192", M=8, N=8, K=8)
    assert A.dtype == torch.bfloat16
    A16, _ = inputs.make_workload("f16_8192", M=8, N=8, K=8)
    assert torch.equal(A.float().half().float() - A16.float(), A.float().half().float() - A16.float())
    w = inputs.WORKLOADS["bf16_8192"]
    assert math.isclose(w.sigma, 1 / math.sqrt(8192))


# ----------------------------------------------------------------- the extended product
# C = alpha * op(A) @ op(B) + beta * C0 (the pages' wgmma: D = A*B + D with
# transposable, negatable operands and D scaled by 0 or 1; generalised).

@pytest.mark.parametrize("transa,transb", [(False, False), (True, False), (False, True),
                                           (True, True)])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ex_transposes_match_plain_product(oracle_mod, transa, transb, dtype):
    """Stored transposes (made by numpy) give exactly the plain product."""
    A_t, B_t = inputs.make(23, 17, 31, dtype, "normal", 1.0, seed=51)
    A, B = inputs.host_view(A_t), inputs.host_view(B_t)
    C, Cabs = oracle_mod.gemm(A, B, dtype)
    As = np.ascontiguousarray(A.T) if transa else A
    Bs = np.ascontiguousarray(B.T) if transb else B
    C2, Cabs2 = oracle_mod.gemm_ex(As, Bs, dtype, transa, transb)
    assert np.array_equal(C, C2) and np.array_equal(Cabs, Cabs2)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.0, 1.0), (-1.0, 1.0), (2.0, -3.0),
                                        (0.5, 0.25), (0.0, 1.0), (-1.0, 0.0)])
def test_ex_alpha_beta_integer_exact(oracle_mod, alpha, beta):
    """Integer matrices and dyadic scalars: the exact result, computed with
    Python fractions, including the |alpha||A||B| + |beta||C0| scale."""
    from fractions import Fraction as F
    A_t, B_t = inputs.make_integer(9, 11, 13, 4, "f32", seed=52)
    g = np.random.default_rng(53)
    C0 = g.integers(-50, 51, (9, 11)).astype(np.float32)
    A, B = A_t.numpy(), B_t.numpy()
    C, Cabs = oracle_mod.gemm_ex(A, B, "f32", alpha=alpha, beta=beta, C0=C0)
    AB = A.astype(np.int64) @ B.astype(np.int64)
    AbsAB = np.abs(A.astype(np.int64)) @ np.abs(B.astype(np.int64))
    for i in range(9):
        for j in range(11):
            want = F(alpha) * int(AB[i, j]) + F(beta) * F(float(C0[i, j]))
            want_abs = abs(F(alpha)) * int(AbsAB[i, j]) + abs(F(beta)) * abs(F(float(C0[i, j])))
            assert C[i, j] == float(want) and Cabs[i, j] == float(want_abs)


def test_ex_beta_zero_does_not_read_c0(oracle_mod):
    A_t, B_t = inputs.make(8, 8, 8, "f32", "uniform", 1.0, seed=54)
    C0 = np.full((8, 8), np.nan, np.float32)
    C, Cabs = oracle_mod.gemm_ex(A_t.numpy(), B_t.numpy(), "f32", alpha=2.0, beta=0.0, C0=C0)
    ref, refabs = oracle_mod.gemm(A_t.numpy(), B_t.numpy())
    assert not np.isnan(C).any()
    assert np.array_equal(C, 2.0 * ref) and np.array_equal(Cabs, 2.0 * refabs)


def test_ex_brute_force_tiny_fraction(oracle_mod):
    """All shapes in {1..3}^3, every transpose combination, dyadic entries and
    scalars: exact rational sums."""
    from fractions import Fraction as F
    g = np.random.default_rng(55)
    for M, N, K in itertools.product(range(1, 4), repeat=3):
        for ta, tb in itertools.product([False, True], repeat=2):
            A = (g.integers(-16, 17, (M, K)) / 8.0).astype(np.float32)
            B = (g.integers(-16, 17, (K, N)) / 8.0).astype(np.float32)
            C0 = (g.integers(-16, 17, (M, N)) / 4.0).astype(np.float32)
            alpha, beta = float(g.integers(-4, 5)) / 2, float(g.integers(-4, 5)) / 2
            As = np.ascontiguousarray(A.T) if ta else A
            Bs = np.ascontiguousarray(B.T) if tb else B
            C, _ = oracle_mod.gemm_ex(As, Bs, "f32", ta, tb, alpha, beta, C0)
            for i in range(M):
                for j in range(N):
                    s = sum(F(float(A[i, k])) * F(float(B[k, j])) for k in range(K))
                    want = F(alpha) * s + (F(beta) * F(float(C0[i, j])) if beta else 0)
                    assert C[i, j] == float(want)


# ----------------------------------------------------------------- tf32 truncation
# TF32 ([book] "Tensor Cores" -> "TF32 (TensorFloat-32) 精度"): fp32's 8-bit
# exponent with 10 fraction bits. The page fixes the format, not how an fp32
# value is brought into it; the tensor cores read an fp32 operand by clearing
# its 13 low fraction bits (truncation toward zero), and so does the oracle.

def _tf32_trunc_reference(x: float) -> float:
    """Largest-magnitude value with 11 significant bits not above |x| (fp32's
    exponent range), sign kept: truncation toward zero, by exact rationals."""
    if x == 0 or math.isinf(x) or math.isnan(x):
        return x
    s = -1 if x < 0 else 1
    a = Fraction(abs(x))
    _, e = math.frexp(abs(x))
    e = max(e, -125)
    unit = Fraction(2) ** (e - 11)
    return s * float((a // unit) * unit)


@pytest.mark.parametrize("x,want", [
    (1.0, 1.0), (1 + 2.0 ** -10, 1 + 2.0 ** -10),
    (1 + 2.0 ** -11, 1.0), (1 + 2.0 ** -10 - 2.0 ** -23, 1.0),    # toward zero, never up
    (-(1 + 2.0 ** -10 - 2.0 ** -23), -1.0),
    (2 - 2.0 ** -23, 2 - 2.0 ** -10),                               # no carry
    (3.4028234663852886e38, (2 - 2.0 ** -10) * 2.0 ** 127),         # stays finite
    (2.0 ** -149, 0.0), (2.0 ** -136 + 2.0 ** -149, 2.0 ** -136),
    (math.inf, math.inf), (-math.inf, -math.inf),
])
def test_truncate_tf32_textbook_values(oracle_mod, x, want):
    got = oracle_mod.truncate_tf32(np.array([[x]], np.float32))[0, 0]
    assert got == np.float32(want) and np.signbit(got) == np.signbit(np.float32(want))


def test_truncate_tf32_matches_exact_rational_truncation(oracle_mod):
    g = np.random.default_rng(61)
    x = g.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32)
    x = x[np.isfinite(x)].reshape(1, -1)
    got = oracle_mod.truncate_tf32(x)[0]
    for xi, gi in zip(x[0], got):
        assert gi == np.float32(_tf32_trunc_reference(float(xi))), (xi, gi)
    # a quiet NaN stays NaN; truncation never moves a value away from zero
    assert np.isnan(oracle_mod.truncate_tf32(np.array([[np.nan]], np.float32))[0, 0])
    assert (np.abs(got) <= np.abs(x[0])).all()


# 3xTF32 (reading R14: the split of Ootomo and Yokota, 2022): x = hi + lo with
# hi = tf32(x) and lo = x - hi, and A B ~ hi(A) hi(B) + hi(A) lo(B) + lo(A) hi(B).
# The bound the kernels are held to rests on the split being exact, lo being
# below 2^-10 |x|, and the dropped and truncated terms each staying below
# 2^-20 |a||b| per product; these pins check those facts on the oracle's
# truncation and its products.

def _split(oracle_mod, X):
    hi = oracle_mod.truncate_tf32(X)
    return hi, (X - hi).astype(np.float32)


def test_tf32_split_is_exact_and_lo_is_small(oracle_mod):
    g = np.random.default_rng(62)
    x = (g.standard_normal(20000) * np.exp2(g.integers(-60, 61, 20000))).astype(np.float32)
    x = x.reshape(1, -1)
    hi, lo = _split(oracle_mod, x)
    # the fp32 subtraction is exact: hi + lo is x, compared in float64
    assert np.array_equal(hi.astype(np.float64) + lo.astype(np.float64), x.astype(np.float64))
    # lo is below 2^-10 |x| (normal x: 10 fraction bits kept), with x's sign or zero
    assert (np.abs(lo) < np.abs(x) * 2.0 ** -10).all()
    assert ((lo == 0) | (np.sign(lo) == np.sign(x))).all()
    # truncation is idempotent and hi is already a tf32 value
    assert np.array_equal(oracle_mod.truncate_tf32(hi), hi)


def test_3xtf32_terms_against_the_exact_product(oracle_mod):
    """The three-term sum misses the exact product of the fp32 inputs by the
    dropped lo(A) lo(B) term alone, below 2^-20 (|A||B|); reading each lo part
    as tf32 too (the tensor cores' reading) stays below 3 * 2^-20 (|A||B|),
    the bound the fp32 tolerance 1e-5 covers."""
    g = np.random.default_rng(63)
    A = (g.random((48, 96)) * 2 - 1).astype(np.float32)
    B = (g.random((96, 40)) * 2 - 1).astype(np.float32)
    hA, lA = _split(oracle_mod, A)
    hB, lB = _split(oracle_mod, B)
    exact, absAB = oracle_mod.gemm(A, B)
    hh, _ = oracle_mod.gemm(hA, hB)
    hl, _ = oracle_mod.gemm(hA, lB)
    lh, _ = oracle_mod.gemm(lA, hB)
    ll, _ = oracle_mod.gemm(lA, lB)
    slack = 1e-12 * absAB  # the oracle's own float64 sums
    # exact split: the four terms give the product
    assert (np.abs(hh + hl + lh + ll - exact) <= slack).all()
    err3 = np.abs(hh + hl + lh - exact)
    assert (err3 <= 2.0 ** -20 * absAB + slack).all()
    assert err3.max() > 0  # the dropped term is not always zero
    tl, _ = oracle_mod.gemm(hA, oracle_mod.truncate_tf32(lB))
    lt, _ = oracle_mod.gemm(oracle_mod.truncate_tf32(lA), hB)
    assert (np.abs(hh + tl + lt - exact) <= 3 * 2.0 ** -20 * absAB + slack).all()
    # and a single tf32 product is far outside that bound somewhere
    assert (np.abs(hh - exact) > 3 * 2.0 ** -20 * absAB).any()
