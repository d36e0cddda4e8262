"""Host-side checks of the stream-K schedule and the workspace entry points."""
import os
import subprocess

import pytest

import dense_gemm_14_gb300 as g14
from dense_gemm_14_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "dense_gemm_14_gb300", "csrc")


def test_schedule_covers_every_k_block_once(tmp_path):
    exe = tmp_path / "sk_check"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe),
                    os.path.join(ROOT, "tests", "streamk_schedule_check.cpp")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout[-2000:]
    assert "bad = 0" in out.stdout


def test_workspace_bytes():
    g14.load()
    F32, BF16 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16
    # fp32: the flags (one word per SM, 256-byte aligned), then one 128 x 256
    # slot per worker (for its PARTIAL; a HEAD adds into its accumulators)
    want = 768 + 152 * 128 * 256 * 4
    assert g14.workspace_bytes(F32, 3072, 3072, 3072, 152) == want
    assert g14.workspace_bytes(F32, 4097, 3001, 513, 152) == want
    # skinny bf16: 128 tiles of 128 x 64 (64-row tiles would spill past one
    # wave) -- between half and one wave: not split
    assert g14.workspace_bytes(BF16, 16384, 64, 4096, 152) == 0
    # 16-bit one-SM tiles between one and two waves: split with the last wave
    # under half full (180 tiles), not above (284 tiles); beyond two waves the
    # last one and a half (320 tiles)
    assert g14.workspace_bytes(BF16, 23040, 64, 4096, 152) == 768 + 152 * 128 * 64 * 4
    assert g14.workspace_bytes(BF16, 36352, 64, 4096, 152) == 0
    assert g14.workspace_bytes(BF16, 40960, 64, 4096, 152) == 768 + 152 * 128 * 64 * 4
    # few tiles (fewer than half a wave; 64-row tiles since those fit in one
    # wave): split, one 64 x 64 slot per worker
    assert g14.workspace_bytes(BF16, 1024, 64, 4096, 152) == 768 + 152 * 64 * 64 * 4
    # ... but a 16-bit tile takes at most 4 workers, each with at least 16 of
    # its k-blocks: two tiles of 64 k-blocks split 4 ways each, of 8 or 16 not
    assert g14.workspace_bytes(BF16, 128, 64, 4096, 152) == 768 + 152 * 64 * 64 * 4
    assert g14.workspace_bytes(BF16, 128, 64, 512, 152) == 0
    assert g14.workspace_bytes(BF16, 128, 64, 1024, 152) == 0
    # fp32 products of few 128 x 256 tiles run 64 x 64 tiles split over
    # clusters, added up in shared memory: no workspace
    assert g14.workspace_bytes(F32, 256, 256, 256, 152) == 0
    # ... from more than half the SMs' worth of tiles the large kernel, whose
    # long k-blocks spread over every SM past a whole wave (160 tiles of 8
    # k-blocks), not within one (80 tiles)
    assert g14.workspace_bytes(F32, 2560, 2048, 256, 152) == want
    assert g14.workspace_bytes(F32, 1280, 2048, 256, 152) == 0
    # the CTA-pair kernel (a cluster of two per worker): one 128 x 256 slot per
    # SM when it splits -- between one and two waves with long k (90 tiles on
    # 76 clusters), or few tiles with long k (4 tiles, 16 workers) ...
    pair_ws = 768 + 152 * 128 * 256 * 4
    assert g14.workspace_bytes(BF16, 2304, 2560, 8192, 152) == pair_ws
    assert g14.workspace_bytes(BF16, 512, 512, 16384, 152) == pair_ws
    # ... beyond two waves that are not whole, the last one and a half waves
    # (8192^3: 1024 tiles = 13.47 waves on 76 clusters) ...
    assert g14.workspace_bytes(BF16, 8192, 8192, 8192, 152) == pair_ws
    # ... but not a last wave more than half full below two waves (144 tiles =
    # 1.89 waves), nor whole waves (152 tiles on 76 clusters), nor short k
    assert g14.workspace_bytes(BF16, 3072, 3072, 8192, 152) == 0
    assert g14.workspace_bytes(BF16, 2048, 4864, 8192, 152) == 0
    assert g14.workspace_bytes(BF16, 2304, 2560, 2000, 152) == 0
    assert g14.workspace_bytes(BF16, 1000, 776, 1000, 152) == 0
    # whole waves use none; invalid args -> 0
    assert g14.workspace_bytes(F32, 128 * 152, 256, 64, 152) == 0
    assert g14.workspace_bytes(F32, -1, 4, 4, 152) == 0


def test_ws_entry_points_validate_workspace():
    g14.load()
    P = 1 << 16
    for fn in (g14.gemm_f32_ws, g14.gemm_bf16_f32acc_ws, g14.gemm_f16_f32acc_ws):
        # misaligned workspace
        assert fn(4, 8, 8, P, 8, P, 8, P, 8, P + 4, 1 << 20, None, check=False) == \
            _lib.GEMM14_ERR_INVALID_ARG
        # the usual argument checks still apply
        assert fn(-1, 8, 8, P, 8, P, 8, P, 8, P, 1 << 20, None, check=False) == \
            _lib.GEMM14_ERR_INVALID_ARG
        # empty products need nothing
        assert fn(0, 8, 8, P, 8, P, 8, P, 8, 0, 0, None, check=False) == 0


def _r256(x):
    return (x + 255) // 256 * 256


def test_workspace_bytes_ex_adds_room_to_repitch():
    """Aligned operands need what gemm14_workspace_bytes gives; an operand TMA
    cannot read adds its copy with a 16-byte pitch after the stream-K region
    (which keeps the workspace's start), A's copy first."""
    g14.load()
    F32, BF16 = g14.GEMM14_DTYPE_F32, g14.GEMM14_DTYPE_BF16
    P = 1 << 20
    ex = g14.workspace_bytes_ex
    # aligned: the same as the shape-only query (fp32 narrower than 2048
    # columns: no transposed copy of A, below)
    for dt, M, N, K in ((F32, 3072, 2000, 3072), (F32, 4097, 1001, 516), (BF16, 1024, 64, 4096),
                        (BF16, 16384, 64, 4096), (BF16, 2304, 2560, 8192), (BF16, 3072, 3072, 3072)):
        lda, ldb = (K + 7) // 8 * 8, (N + 7) // 8 * 8
        assert ex(dt, 0, 0, M, N, K, P, lda, P, ldb, P, ldb, 152) == \
            g14.workspace_bytes(dt, M, N, K, 152)
    # fp32 4097 x 3001 x 513 (pitches 2052 and 12004 bytes): both copied, A
    # transposed into K x M (N >= 2048) with a pitch of 4100 floats
    M, N, K = 4097, 3001, 513
    sk = 768 + 152 * 128 * 256 * 4              # 396 tiles: split, one fp32 slot per SM
    a_off = _r256(sk)
    b_off = _r256(a_off + K * 4100 * 4)
    assert ex(F32, 0, 0, M, N, K, P, K, P, N, P, N, 152) == b_off + K * 3004 * 4
    # only B unaligned (bf16, ldb odd), 128 tiles (not split): the copy after the flags
    M, N, K = 16384, 64, 4096
    assert ex(BF16, 0, 0, M, N, K, P, K, P, 65, P, N, 152) == 768 + K * 64 * 2
    # a misaligned base with an aligned pitch is copied too (A stored K x M)
    M, N, K = 2000, 2000, 777
    sk = g14.workspace_bytes(F32, M, N, K, 152)
    assert ex(F32, 1, 0, M, N, K, P + 4, 2000, P, N, P, N, 152) == _r256(max(sk, 768)) + K * 2000 * 4
    # ... but not for the small-product kernel (18 tiles of 128 x 256, under
    # 2^30 FLOP), which reads any base, pitch and storage as it is
    M, N, K = 700, 530, 333
    assert ex(F32, 1, 0, M, N, K, P + 4, 700, P, N, P, N, 152) == 0
    assert ex(F32, 0, 1, M, N, K, P, 333, P + 4, 333, P, N, 152) == 0
    # ... which a call with a workspace leaves above 2^30 FLOP (1000 x 1000 x
    # 777: 1.55 GFLOP): the large kernel, A copied, split over every SM
    M, N, K = 1000, 1000, 777
    assert ex(F32, 1, 0, M, N, K, P + 4, 1000, P, N, P, N, 152) == \
        _r256(768 + 152 * 128 * 256 * 4) + K * 1000 * 4
    # nothing to compute, or invalid arguments: 0
    assert ex(F32, 0, 0, 8, 8, 0, 0, 1, 0, 8, P, 8, 152) == 0
    assert ex(F32, 0, 0, 8, 8, 8, P, 7, P, 8, P, 8, 152) == 0


def test_workspace_bytes_ex_tf32_transposes_into_k_major():
    """TF32 reads fp32 operands straight from TMA only K-major (A stored M x K,
    B stored N x K): other storages get K-major copies in the workspace, after
    the stream-K region of the pair kernel's split (plan kernel 5). 3xTF32 on
    that kernel also needs lo(A) and lo(B), written after the copies."""
    g14.load()
    TF32, X3 = g14.GEMM14_DTYPE_TF32, g14.GEMM14_DTYPE_F32_3XTF32
    P = 1 << 20
    n = 3072
    flags = 768                            # 144 pair tiles = 1.89 waves: not split
    ex = g14.workspace_bytes_ex
    assert ex(TF32, 0, 1, n, n, n, P, n, P, n, P, n, 152) == 0                   # NT: as stored
    assert ex(TF32, 0, 0, n, n, n, P, n, P, n, P, n, 152) == flags + n * n * 4   # B^T
    assert ex(TF32, 1, 1, n, n, n, P, n, P, n, P, n, 152) == flags + n * n * 4   # A^T
    assert ex(TF32, 1, 0, n, n, n, P, n, P, n, P, n, 152) == flags + 2 * n * n * 4
    # 2304 x 2560 (90 tiles, 1.18 waves, 128 k-blocks) is split: copies after the slots
    M, N, K = 2304, 2560, 4096
    sk = 768 + 152 * 128 * 256 * 4
    assert ex(TF32, 0, 0, M, N, K, P, K, P, N, P, N, 152) == sk + N * K * 4
    # 3xTF32 takes the same K-major copies and lo(A), lo(B) after them (both
    # K-major, pitch K rounded up to 4 floats), in every storage
    lo = 2 * n * n * 4
    assert ex(X3, 0, 1, n, n, n, P, n, P, n, P, n, 152) == flags + lo
    assert ex(X3, 0, 0, n, n, n, P, n, P, n, P, n, 152) == flags + n * n * 4 + lo
    assert ex(X3, 1, 0, n, n, n, P, n, P, n, P, n, 152) == flags + 2 * n * n * 4 + lo
    # its 3 x 128 k-blocks at 1.18 waves are split like TF32's
    M, N, K = 2304, 2560, 4096
    assert ex(X3, 0, 1, M, N, K, P, K, P, K, P, N, 152) == sk + (M + N) * K * 4
    # 4 pair tiles of 3 x 32 k-blocks: split over 12 clusters (3 terms make k
    # long enough where TF32's 32 k-blocks stay unsplit); K rounded up to 1004
    M, N, K = 512, 384, 1001
    assert ex(X3, 0, 1, M, N, K, P, 1004, P, 1004, P, N, 152) == \
        _r256(sk + M * 1004 * 4) + N * 1004 * 4
    # without the pair kernel 3xTF32 runs on the converter kernel: no copies
    prev = g14.set_pair_kernel(False)
    try:
        assert ex(X3, 0, 0, n, n, n, P, n, P, n, P, n, 152) == 0
    finally:
        g14.set_pair_kernel(prev)
    # a transposed copy has K rounded up to 4 floats: B (K x N) -> N x round4(K);
    # 4 pair tiles of 32 k-blocks are not split, so the copy follows the flags
    M, N, K = 512, 384, 1001
    assert ex(TF32, 0, 0, M, N, K, P, 1004, P, N, P, N, 152) == 768 + N * 1004 * 4


def test_workspace_bytes_ex_fp32_b_stored_n_by_k():
    """fp32 FFMA with B stored N x K gets a K x N copy of B (its fast storage)."""
    g14.load()
    F32 = g14.GEMM14_DTYPE_F32
    P = 1 << 20
    n = 3072
    sk = g14.workspace_bytes(F32, n, n, n, 152)
    ex = g14.workspace_bytes_ex
    assert ex(F32, 1, 0, n, n, n, P, n, P, n, P, n, 152) == sk
    assert ex(F32, 1, 1, n, n, n, P, n, P, n, P, n, 152) == sk + n * n * 4
    # A stored M x K is transposed into K x M when N >= 2048 (5 % faster kernel)
    assert ex(F32, 0, 0, n, n, n, P, n, P, n, P, n, 152) == sk + n * n * 4
    assert ex(F32, 0, 1, n, n, n, P, n, P, n, P, n, 152) == sk + 2 * n * n * 4
    # ... not for narrower products
    assert ex(F32, 0, 0, n, 2047, n, P, n, P, 2048, P, 2048, 152) == \
        g14.workspace_bytes(F32, n, 2047, n, 152)


def test_device_check_predicates(tmp_path):
    """The predicates of the device-side bounds checks (csrc/checks.h), on
    the host: in-bounds accesses pass, one element outside fails."""
    exe = tmp_path / "checks_predicates"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe),
                    os.path.join(ROOT, "tests", "checks_predicates.cpp")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout
