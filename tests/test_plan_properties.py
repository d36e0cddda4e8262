"""Properties of the launch planner over random calls (host only, no GPU):
whatever the shape, storage, alignment and SM count, a plan launches a kernel
the dtype has, with a tile count and grid that follow from its tile shape,
within the shared-memory limit, with the thread count of the variant it picks,
and with loaders that follow TMA's 16-byte rules operand by operand."""
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import dense_gemm_14_gb300 as g14  # noqa: E402

F32, BF16, F16 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16, g14.GEMM14_DTYPE_F16
TF32, X3 = g14.GEMM14_DTYPE_TF32, g14.GEMM14_DTYPE_F32_3XTF32
ELEM = {F32: 4, BF16: 2, F16: 2, TF32: 4, X3: 4}
BASE = 1 << 40  # a 256-byte-aligned device-like address (never dereferenced)

dims = st.one_of(st.integers(1, 300), st.integers(300, 20000))


def cdiv(a, b):
    return -(-a // b)


def leading_dim(cols, eb, aligned, extra):
    """A pitch TMA can take (a multiple of 16 bytes) or any pitch >= cols."""
    q = 16 // eb
    return cdiv(cols, q) * q + q * (extra % 2) if aligned else cols + extra


@settings(max_examples=600, deadline=None)
@given(dtype=st.sampled_from([F32, BF16, F16, TF32, X3]), ta=st.integers(0, 1),
       tb=st.integers(0, 1), M=dims, N=dims, K=dims, a_al=st.booleans(), b_al=st.booleans(),
       xa=st.integers(0, 9), xb=st.integers(0, 9), oa=st.integers(0, 7), ob=st.integers(0, 7),
       xc=st.integers(0, 5), oc=st.integers(0, 3), sms=st.sampled_from([8, 132, 148, 152]))
def test_plan_invariants(dtype, ta, tb, M, N, K, a_al, b_al, xa, xb, oa, ob, xc, oc, sms):
    eb = ELEM[dtype]
    a_cols, b_cols = (M if ta else K), (K if tb else N)
    lda, ldb, ldc = leading_dim(a_cols, eb, a_al, xa), leading_dim(b_cols, eb, b_al, xb), N + xc
    oa, ob = (0 if a_al else oa), (0 if b_al else ob)
    A, B, C = BASE + eb * oa, BASE + (1 << 32) + eb * ob, BASE + (2 << 32) + 4 * oc
    st_, p = g14.plan_ex(dtype, ta, tb, M, N, K, A, lda, B, ldb, C, ldc, sms)
    assert st_ == 0
    assert p.smem_bytes <= 227 * 1024 and p.smem_bytes > 0
    assert p.vec_store == int(C % 16 == 0 and ldc % 4 == 0)
    assert p.tiles == cdiv(M, p.bm) * cdiv(N, p.bn)
    q = 16 // eb
    a_tma = A % 16 == 0 and lda % q == 0
    b_tma = B % 16 == 0 and ldb % q == 0
    if dtype in (F32, TF32, X3):
        assert p.kernel in (1, 4, 5, 6)
    else:
        assert p.kernel in (2, 3)
    if p.kernel == 1:
        assert (p.bm, p.bn, p.bk, p.threads) == (128, 256, 32, 256)
        assert p.grid == min(p.tiles, sms)
        assert p.loader == (1 if a_tma and b_tma else 2)
        assert p.stages == (3 if p.loader == 1 and tb else 4)
    elif p.kernel == 6:
        assert (p.bm, p.bn, p.threads) == (64, 64, 128)
        split = p.grid // p.tiles
        assert p.grid == split * p.tiles and split in (1, 2, 4, 8)
        assert split == 1 or (p.grid <= 4 * sms and split <= cdiv(K, 32))
        assert 2 * cdiv(M, 128) * cdiv(N, 256) <= sms  # few large tiles
    elif p.kernel in (3, 4, 5):
        assert (p.bm, p.bn) == (256, 256) and p.grid % 2 == 0
        assert p.grid == 2 * min(p.tiles, sms // 2)
        assert p.loader == 1 and a_tma and b_tma
        if p.kernel == 3:
            assert M > 128 and N > 128 and p.threads == 192
        if p.kernel == 5:
            assert dtype == TF32 and not ta and tb
        if p.kernel == 4:
            # TF32: two announcer warps, 4 operand stages of copies; 3xTF32:
            # its converters announce themselves, 2 operand stages
            assert (p.threads, p.stages) == ((384, 4) if dtype == TF32 else (320, 2))
    else:  # kernel 2: one SM per tile, each operand by TMA where it can be
        assert p.bm in (64, 128) and p.bn in (64, 128, 256) and p.bk == 64
        assert p.grid == min(p.tiles, sms)
        want = 1 if a_tma and b_tma else 2 if not (a_tma or b_tma) else 3 if not a_tma else 4
        assert p.loader == want
        assert p.threads == (192 if p.loader == 1 else 448)
        if p.loader == 1 and M > 128 and N > 128:
            pytest.fail("a wide product with TMA-addressable operands belongs on CTA pairs")
