"""The C ABI on the host: the library loads, exports every symbol the header
declares, validates arguments before touching CUDA, and plans launches.
No GPU needed (nothing here enqueues work)."""
import ctypes
import os
import re

import pytest

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm14.h")

F32, BF16, F16 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16, g14.GEMM14_DTYPE_F16


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_14_gb300 import build
    build.build()
    return g14.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("gemm_f32", "gemm_bf16_f32acc", "gemm_f16_f32acc"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"


def test_exports_are_exactly_the_header(lib):
    """The library's dynamic symbol table holds the header's functions and
    nothing else: the kernels' C++ internals and the statically linked CUDA
    runtime stay local (a linker version script)."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", g14.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({line.split()[-1] for line in out.splitlines() if line.strip()})
    assert exported == declared_functions()


def test_status_strings(lib):
    assert g14.status_string(0) == "ok"
    for s in range(1, 6):
        assert g14.status_string(s) and g14.status_string(s) != "unknown status"
    assert g14.status_string(99) == "unknown status"
    assert g14.version() >= 100


P = 0x10000  # a 64 KiB-aligned fake device address (never dereferenced)


@pytest.mark.parametrize("fn", [g14.gemm_f32, g14.gemm_bf16_f32acc, g14.gemm_f16_f32acc])
@pytest.mark.parametrize("args", [
    (-1, 4, 4, P, 4, P, 4, P, 4),        # negative M
    (4, -1, 4, P, 4, P, 4, P, 4),        # negative N
    (4, 4, -2, P, 4, P, 4, P, 4),        # negative K
    (1 << 31, 4, 4, P, 4, P, 4, P, 4),   # M beyond int32
    (4, 4, 8, P, 4, P, 4, P, 4),         # lda < K
    (4, 8, 4, P, 8, P, 4, P, 8),         # ldb < N
    (4, 8, 4, P, 8, P, 8, P, 4),         # ldc < N
    (4, 4, 4, 0, 8, P, 8, P, 8),         # A NULL
    (4, 4, 4, P, 8, 0, 8, P, 8),         # B NULL
    (4, 4, 4, P, 8, P, 8, 0, 8),         # C NULL
    (4, 4, 4, P, 8, P, 8, P + 2, 8),     # C misaligned
])
def test_invalid_arguments_rejected_before_cuda(lib, fn, args):
    assert fn(*args, None, check=False) == _lib.GEMM14_ERR_INVALID_ARG


def test_loader_choice_follows_tma_rules(lib):
    # 16-bit operands: TMA needs 16-byte bases and pitches (multiples of 8 elements)
    st, p = g14.plan(BF16, 4, 8, 4, P, 8, P, 8, P, 8, 152)
    assert st == 0 and p.loader == 1
    # each operand on its own: 3 = software A and TMA B, 4 = the reverse, 2 = both
    st, p = g14.plan(BF16, 4, 8, 4, P, 12, P, 8, P, 8, 152)
    assert st == 0 and p.loader == 3
    st, p = g14.plan(F16, 4, 8, 4, P + 8, 8, P, 8, P, 8, 152)
    assert st == 0 and p.loader == 3
    st, p = g14.plan(BF16, 4, 8, 4, P, 8, P + 2, 8, P, 8, 152)
    assert st == 0 and p.loader == 4
    st, p = g14.plan(BF16, 4, 8, 4, P, 12, P, 9, P, 8, 152)
    assert st == 0 and p.loader == 2
    # an odd byte address is not an element address
    assert g14.gemm_bf16_f32acc(4, 8, 4, P + 1, 8, P, 8, P, 8, None, check=False) == 1
    # fp32: any 4-byte aligned pointer/pitch (cp.async loader)
    st, p = g14.plan(F32, 4, 8, 5, P + 4, 5, P + 4, 9, P, 8, 152)
    assert st == 0 and p.loader == 2
    assert g14.gemm_f32(4, 8, 4, P + 2, 8, P, 8, P, 8, None, check=False) == 1


def test_empty_product_is_a_no_op(lib):
    # M == 0 or N == 0: OK without any CUDA call (works without a GPU)
    assert g14.gemm_f32(0, 4, 4, 0, 4, 0, 4, 0, 4, None, check=False) == 0
    assert g14.gemm_bf16_f32acc(4, 0, 4, 0, 8, 0, 8, 0, 1, None, check=False) == 0


def test_plan_fp32_tma_and_fallback(lib):
    st, p = g14.plan(F32, 3072, 3072, 3072, P, 3072, P, 3072, P, 3072, 152)
    assert st == 0
    assert (p.kernel, p.loader, p.bm, p.bn, p.bk) == (1, 1, 128, 256, 32)
    assert p.tiles == 24 * 12 and p.grid == 152 and p.vec_store == 1
    assert p.smem_bytes <= 227 * 1024 and p.threads == 256
    # the ragged workload breaks TMA's 16-byte pitch rule -> cp.async loader, scalar stores
    st, p = g14.plan(F32, 4097, 3001, 513, P, 513, P, 3001, P, 3001, 152)
    assert st == 0 and p.loader == 2 and p.vec_store == 0
    assert p.tiles == 33 * 12
    # just over half the SMs' worth of 128 x 256 tiles: still the large kernel
    st, p = g14.plan(F32, 1280, 2048, 256, P, 256, P, 2048, P, 2048, 152)
    assert (p.kernel, p.tiles, p.grid) == (1, 80, 80)


# fp32 products whose 128 x 256 tiles would fill at most half the SMs: 64 x 64
# tiles, k split over a cluster of 2-8 CTAs while the grid stays within four
# CTAs per SM and each CTA has a k-block.
@pytest.mark.parametrize("M,N,K,tiles,split", [
    (256, 256, 256, 16, 8),      # the 256^3 workload: 8 k-blocks, one per CTA
    (512, 512, 512, 64, 8),      # 8 x 64 CTAs <= 4 x 152
    (1024, 1024, 1024, 256, 2),  # 4 x 256 would pass four CTAs per SM
    (256, 256, 64, 16, 2),       # 2 k-blocks: split 2
    (1, 1, 1, 1, 1),
    (64, 64, 65536, 1, 8),       # a cluster is at most 8 CTAs
    (1280, 1024, 256, 320, 1),   # 40 large tiles <= 76
])
def test_plan_fp32_small_products(lib, M, N, K, tiles, split):
    st, p = g14.plan(F32, M, N, K, P, K, P, N, P, N, 152)
    assert st == 0 and p.kernel == 6 and (p.bm, p.bn, p.bk) == (64, 64, 32)
    assert p.tiles == tiles and p.grid == split * tiles
    assert p.threads == 128 and p.smem_bytes <= 227 * 1024
    assert p.loader == (1 if K % 4 == 0 and N % 4 == 0 else 2)
    # no stream-K workspace and no operand copies: the split is added up on
    # chip; but a call with a workspace runs products above 2^30 FLOP on the
    # large kernel, split over every SM
    if 2 * M * N * K <= 1 << 30:
        assert g14.workspace_bytes(F32, M, N, K, 152) == 0
        assert g14.workspace_bytes_ex(F32, 0, 1, M, N, K, P, K, P, K, P, N, 152) == 0
    else:
        assert g14.workspace_bytes(F32, M, N, K, 152) == 768 + 152 * 128 * 256 * 4


def test_plan_fp32_small_product_loaders(lib):
    # 16-byte copies need A stored M x K, B stored K x N, aligned, pitches % 4 == 0
    st, p = g14.plan(F32, 256, 256, 256, P + 4, 256, P, 256, P, 256, 152)
    assert p.kernel == 6 and p.loader == 2
    st, p = g14.plan(F32, 256, 256, 256, P, 257, P, 256, P, 256, 152)
    assert p.kernel == 6 and p.loader == 2
    for ta, tb in ((1, 0), (0, 1), (1, 1)):
        st, p = g14.plan_ex(F32, ta, tb, 256, 256, 256, P, 256, P, 256, P, 256, 152)
        assert st == 0 and p.kernel == 6 and p.loader == 2


def _bm_for(M, N, bn, sms=152):
    """One-SM tile rows: 64 when the 64-row tiles fit in one wave."""
    return 64 if 2 * ((M + 127) // 128) * ((N + bn - 1) // bn) <= sms else 128


@pytest.mark.parametrize("M,N,bn", [(16384, 1, 64), (16384, 64, 64), (16384, 65, 128),
                                    (16384, 128, 128), (32768, 64, 64), (19457, 64, 64),
                                    (64, 64, 64), (100, 128, 128)])
def test_plan_tensor_core_tile_width(lib, M, N, bn):
    st, p = g14.plan(BF16, M, N, 4096, P, 4096, P, ((N + 7) // 8) * 8, P, N, 152)
    bm = _bm_for(M, N, bn)
    assert st == 0 and p.kernel == 2 and p.bn == bn and p.bm == bm and p.bk == 64
    assert p.smem_bytes <= 227 * 1024
    assert p.tiles == ((M + bm - 1) // bm) * ((N + bn - 1) // bn)
    assert p.grid == min(p.tiles, 152)


@pytest.mark.parametrize("M,N", [(16384, 129), (16384, 11008), (8192, 8192), (129, 300)])
def test_plan_pair_kernel_for_wide_products(lib, M, N):
    ldb = ((N + 7) // 8) * 8
    st, p = g14.plan(BF16, M, N, 4096, P, 4096, P, ldb, P, N, 152)
    assert st == 0 and p.kernel == 3 and (p.bm, p.bn, p.bk) == (256, 256, 64)
    tiles = ((M + 255) // 256) * ((N + 255) // 256)
    assert p.tiles == tiles and p.grid == 2 * min(tiles, 76) and p.grid % 2 == 0
    assert p.smem_bytes <= 227 * 1024 and p.threads == 192
    prev = g14.set_pair_kernel(False)
    try:
        st, p1 = g14.plan(BF16, M, N, 4096, P, 4096, P, ldb, P, N, 152)
        assert p1.kernel == 2 and p1.bm == _bm_for(M, N, 256)
    finally:
        g14.set_pair_kernel(prev)
    # operands TMA cannot address stay on the one-SM kernel with the software loader
    st, p2 = g14.plan(BF16, M, N, 4096, P, 4097, P, ldb, P, N, 152)
    assert p2.kernel == 2 and p2.loader == (3 if ldb % 8 == 0 else 2)


def test_plan_k_zero_launches_nothing(lib):
    st, p = g14.plan(F16, 10, 10, 0, 0, 1, 0, 16, P, 16, 152)
    assert st == 0 and p.kernel == 0


def test_no_gpu_gives_a_status_not_a_crash(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = g14.gemm_f32(4, 4, 4, P, 4, P, 4, P, 4, None, check=False)
    assert st in (_lib.GEMM14_ERR_UNSUPPORTED_DEVICE, _lib.GEMM14_ERR_CUDA)
    with pytest.raises(g14.Gemm14Error):
        g14.gemm_f32(4, 4, 4, P, 4, P, 4, P, 4, None)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setenv("GEMM14_LIB", str(tmp_path / "nope.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.load()


# ----------------------------------------------------------------- the extended call

def _ex(dtype, ta, tb, M, N, K, A, lda, B, ldb, C, ldc, alpha=1.0, beta=0.0):
    return g14.gemm_ex(dtype, ta, tb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, None, 0,
                       None, check=False)


@pytest.mark.parametrize("dtype", [F32, BF16, F16])
def test_ex_leading_dimensions_follow_storage(lib, dtype):
    """lda >= K when A is stored M x K, >= M when stored K x M; likewise ldb."""
    M, N, K = 8, 16, 24
    bad = _lib.GEMM14_ERR_INVALID_ARG
    st, _ = g14.plan_ex(dtype, 1, 0, M, N, K, P, M, P, N, P, N, 152)
    assert st == 0
    st, _ = g14.plan_ex(dtype, 1, 0, M, N, K, P, M - 1, P, N, P, N, 152)
    assert st == bad
    st, _ = g14.plan_ex(dtype, 0, 1, M, N, K, P, K, P, K, P, N, 152)
    assert st == 0
    st, _ = g14.plan_ex(dtype, 0, 1, M, N, K, P, K, P, K - 1, P, N, 152)
    assert st == bad
    st, _ = g14.plan_ex(dtype, 0, 0, M, N, K, P, K, P, N - 1, P, N, 152)
    assert st == bad
    st, _ = g14.plan_ex(dtype, 0, 0, M, N, K, P, K - 1, P, N, P, N, 152)
    assert st == bad


@pytest.mark.parametrize("ta,tb", [(2, 0), (0, 2), (-1, 0), (0, -1)])
def test_ex_invalid_transpose_flags(lib, ta, tb):
    assert _ex(F32, ta, tb, 4, 4, 4, P, 4, P, 4, P, 4) == _lib.GEMM14_ERR_INVALID_ARG
    st, _ = g14.plan_ex(F32, ta, tb, 4, 4, 4, P, 4, P, 4, P, 4, 152)
    assert st == _lib.GEMM14_ERR_INVALID_ARG


def test_ex_plan_loaders(lib):
    """TMA in every storage for aligned operands (same tiles), the software
    loader for unaligned ones; 16-bit transposes on pairs too."""
    st, nn = g14.plan_ex(F32, 0, 0, 2048, 2048, 512, P, 2048, P, 2048, P, 2048, 152)
    assert st == 0 and nn.loader == 1 and nn.kernel == 1
    for ta, tb in ((1, 0), (0, 1), (1, 1)):
        st, p = g14.plan_ex(F32, ta, tb, 2048, 2048, 512, P, 2048, P, 2048, P, 2048, 152)
        assert st == 0 and p.loader == 1 and p.tiles == nn.tiles and p.grid == nn.grid
        # B stored N x K is transposed in shared memory: two 32 KB buffers take
        # one ring stage's place
        assert p.stages == (3 if tb else nn.stages) and p.smem_bytes <= 227 * 1024
        assert p.smem_bytes == nn.smem_bytes + (32768 * 2 - 49152 if tb else 0)
        st, p = g14.plan_ex(F32, ta, tb, 2048, 2048, 512, P, 2049, P, 2048, P, 2048, 152)
        assert st == 0 and p.loader == 2
        st, p = g14.plan_ex(BF16, ta, tb, 512, 512, 512, P, 512, P, 512, P, 512, 152)
        assert st == 0 and p.loader == 1 and p.kernel == 3
        st, p = g14.plan_ex(F16, ta, tb, 100, 512, 512, P, 512, P, 512, P, 512, 152)
        assert st == 0 and p.loader == 1 and p.kernel == 2
    # the plain planner is the extended one without transposes
    st, p0 = g14.plan(BF16, 300, 700, 200, P, 200, P, 704, P, 700, 152)
    st1, p1 = g14.plan_ex(BF16, 0, 0, 300, 700, 200, P, 200, P, 704, P, 700, 152)
    assert st == st1 == 0 and p0 == p1


def test_ex_empty_product_is_a_no_op(lib):
    assert _ex(BF16, 1, 1, 0, 4, 4, 0, 1, 0, 4, 0, 4, 2.0, 3.0) == 0
    assert _ex(F32, 0, 1, 4, 0, 4, 0, 4, 0, 4, 0, 1, 2.0, 3.0) == 0


# ----------------------------------------------------------------- fp32 on the tensor cores

TF32, X3 = g14.GEMM14_DTYPE_TF32, g14.GEMM14_DTYPE_F32_3XTF32


@pytest.mark.parametrize("dtype", [TF32, X3])
def test_plan_tf32_pairs_and_fallback(lib, dtype):
    st, p = g14.plan(dtype, 3072, 3072, 3072, P, 3072, P, 3072, P, 3072, 152)
    assert st == 0 and p.kernel == 4 and (p.bm, p.bn, p.bk) == (256, 256, 32)
    assert p.tiles == 144 and p.grid == 152
    # TF32: 12 warps (two announcers), 4 compact operand stages; 3xTF32: 10
    # warps, 2 operand stages (copies and lo tiles)
    assert (p.threads, p.stages) == ((384, 4) if dtype == TF32 else (320, 2))
    assert p.smem_bytes <= 227 * 1024
    for ta, tb in ((1, 0), (0, 1), (1, 1)):
        st, pt = g14.plan_ex(dtype, ta, tb, 3072, 3072, 3072, P, 3072, P, 3072, P, 3072, 152)
        if dtype == TF32 and (ta, tb) == (0, 1):
            # both operands K-major as stored: the 16-bit pair kernel with
            # kind::tf32 MMAs, k-blocks of 32 fp32, no converter warps
            assert st == 0 and pt.kernel == 5 and (pt.bm, pt.bn, pt.bk) == (256, 256, 32)
            assert pt.tiles == 144 and pt.grid == 152 and pt.threads == 192
            # 144 tiles on 76 clusters (1.89 waves, the last more than half
            # full): not split, no workspace
            assert g14.workspace_bytes_ex(dtype, 0, 1, 3072, 3072, 3072, P, 3072, P, 3072, P,
                                          3072, 152) == 0
            # 90 tiles (1.18 waves), 128 k-blocks: split, one 128 x 256 slot an SM
            assert g14.workspace_bytes_ex(dtype, 0, 1, 2304, 2560, 4096, P, 4096, P, 4096, P,
                                          2560, 152) == 768 + 152 * 128 * 256 * 4
        else:
            assert st == 0 and pt == p
    # pitches TMA cannot take: the fp32 SIMT kernel (cp.async loader)
    st, p2 = g14.plan(dtype, 4097, 3001, 513, P, 513, P, 3001, P, 3001, 152)
    assert st == 0 and p2.kernel == 1 and p2.loader == 2
    # no workspace: the pair kernel does not split tiles
    assert g14.workspace_bytes(dtype, 3072, 3072, 3072, 152) == 0


def test_tf32_entry_points_validate(lib):
    for fn in (g14.gemm_tf32_f32acc, g14.gemm_f32_3xtf32):
        assert fn(4, 4, 8, P, 4, P, 4, P, 4, None, check=False) == _lib.GEMM14_ERR_INVALID_ARG
        assert fn(0, 4, 4, 0, 4, 0, 4, 0, 4, None, check=False) == 0
    assert _ex(5, 0, 0, 4, 4, 4, P, 4, P, 4, P, 4) == _lib.GEMM14_ERR_INVALID_ARG  # no dtype 5


def test_host_entry_points_validate_before_any_cuda_call():
    """gemm14_gemm_host / gemm14_host_wait reject bad arguments on the host."""
    import ctypes
    lib = g14.load()
    F32 = g14.GEMM14_DTYPE_F32
    P = 1 << 16
    t = ctypes.c_uint64(0)
    args = (0, 0, 8, 8, 8, 1.0, P, 8, P, 8, 0.0, P, 8)
    assert lib.gemm14_gemm_host(F32, *args, 0, None) == _lib.GEMM14_ERR_INVALID_ARG
    assert lib.gemm14_gemm_host(F32, *args, -1, ctypes.byref(t)) == _lib.GEMM14_ERR_INVALID_ARG
    assert lib.gemm14_gemm_host(99, *args, 0, ctypes.byref(t)) == _lib.GEMM14_ERR_INVALID_ARG
    # lda < K, NULL A with K > 0, transa = 2
    bad = [(0, 0, 8, 8, 8, 1.0, P, 7, P, 8, 0.0, P, 8), (0, 0, 8, 8, 8, 1.0, 0, 8, P, 8, 0.0, P, 8),
           (2, 0, 8, 8, 8, 1.0, P, 8, P, 8, 0.0, P, 8)]
    for a in bad:
        assert lib.gemm14_gemm_host(F32, *a, 0, ctypes.byref(t)) == _lib.GEMM14_ERR_INVALID_ARG
    assert t.value == 0  # untouched by failed calls
    # tickets never issued
    assert g14.host_wait(0, check=False) == _lib.GEMM14_ERR_INVALID_ARG
    assert g14.host_wait(1 << 60, check=False) == _lib.GEMM14_ERR_INVALID_ARG
    # nothing in flight
    assert g14.host_synchronize(check=False) == 0


def test_status_constants_match_the_header():
    """The binding's status constants are the header's enum values."""
    import os
    import re
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "include", "gemm14.h")).read()
    enum = dict((m.group(1), int(m.group(2)))
                for m in re.finditer(r"\b(GEMM14_(?:OK|ERR_[A-Z_]+))\s*=\s*(\d+)", hdr))
    assert set(enum) == {"GEMM14_OK", "GEMM14_ERR_INVALID_ARG", "GEMM14_ERR_UNSUPPORTED_DEVICE",
                         "GEMM14_ERR_CUDA", "GEMM14_ERR_TIMEOUT", "GEMM14_ERR_DEVICE_CHECK"}
    for name, value in enum.items():
        assert getattr(g14, name) == value, name
