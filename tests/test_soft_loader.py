"""The 16-bit software loader: operands that TMA cannot read (row pitches that
are not multiples of 8 elements, bases off a 16-byte boundary) are copied into
shared memory by loader warps in the same swizzled layout the TMA boxes give,
so the one-SM kernel must return the TMA path's very bits. The cases mix row
segments that start on either half of a 4-byte word (odd pitches alternate
them row by row; a 2-byte offset with an even pitch makes them all start on
the upper half), ragged k and column edges, both tile heights, every stored
transpose, and calls where only one operand breaks TMA's rules (TMA loads the
other in the same stages). The tensor-core MMA of the pages' "Tensor Cores" section
reads its operand tiles from shared memory in a fixed layout; how the tiles
get there must not change the product.
"""
import pytest
import torch

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import inputs

from gpu_util import oracle_check_ex, run_ex

pytestmark = pytest.mark.gpu

TRANS = [(0, 0), (1, 0), (0, 1), (1, 1)]

# (M, N, K): 64-row tiles with 256-column tiles and a k tail of 60; 128-row
# tiles (102 tiles of 128 x 256); 64-row tiles with 64 columns and an odd K;
# more tiles than SMs (264 tiles of 128 x 256: CTAs run two tiles in turn)
SHAPES = [(300, 520, 700), (2100, 1300, 300), (200, 64, 333), (4100, 2100, 200)]

# (extra pitch of A, offset of A, extra pitch of B, offset of B), in elements;
# None: that operand on a 16-byte pitch (TMA reads it, the software loader the
# other one)
PITCHES = [(1, 0, 3, 0), (2, 1, 1, 1), (3, 1, 2, 0), (6, 0, 5, 1),
           (None, None, 1, 0), (1, 0, None, None), (None, None, 2, 1), (3, 1, None, None)]


def rup(x, m):
    return (x + m - 1) // m * m


@pytest.fixture(autouse=True)
def one_sm_kernel():
    """The TMA reference runs on the one-SM kernel too (same tiles, same bits)."""
    prev = g14.set_pair_kernel(False)
    yield
    g14.set_pair_kernel(prev)


@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_software_loader_gives_the_tma_bits(oracle_mod, M, N, K, ta, tb):
    A, B = inputs.make(M, N, K, "bf16", "normal", 1.0 / K ** 0.5,
                       seed=11 * M + 7 * N + 3 * K + 2 * ta + tb)
    a_cols, b_cols = (M if ta else K), (K if tb else N)
    C_tma = run_ex(A, B, ta, tb, lda=rup(a_cols, 8), ldb=rup(b_cols, 8))
    for i, (da, oa, db, ob) in enumerate(PITCHES):
        lda = rup(a_cols, 8) if da is None else a_cols + da
        ldb = rup(b_cols, 8) if db is None else b_cols + db
        C = run_ex(A, B, ta, tb, lda=lda, ldb=ldb, ldc=N + 1, a_off=oa or 0, b_off=ob or 0,
                   c_off=1)
        if i == 0:
            oracle_check_ex(oracle_mod, A, B, C, ta, tb)
        assert torch.equal(C, C_tma), (da, oa, db, ob)


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 1)])
def test_software_loader_f16(oracle_mod, ta, tb):
    M, N, K = 300, 520, 700
    A, B = inputs.make(M, N, K, "f16", "normal", 1.0 / K ** 0.5, seed=5 + ta)
    a_cols, b_cols = (M if ta else K), (K if tb else N)
    C_tma = run_ex(A, B, ta, tb, lda=rup(a_cols, 8), ldb=rup(b_cols, 8))
    C = run_ex(A, B, ta, tb, lda=a_cols + 1, ldb=b_cols + 1, a_off=1, b_off=1)
    oracle_check_ex(oracle_mod, A, B, C, ta, tb)
    assert torch.equal(C, C_tma)


def test_software_loader_one_k_block_and_tiny():
    """K = 1 and K = 64 (the first k block is also the last) and a 1 x 1 x 1
    product, with odd pitches."""
    for M, N, K in [(130, 70, 1), (130, 70, 64), (1, 1, 1), (65, 3, 65)]:
        A, B = inputs.make(M, N, K, "bf16", "uniform", 1.0, seed=M + N + K)
        C_tma = run_ex(A, B, lda=rup(K, 8), ldb=rup(N, 8))
        C = run_ex(A, B, lda=K + 1, ldb=N + 1, a_off=1)
        assert torch.equal(C, C_tma), (M, N, K)
