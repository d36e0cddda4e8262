"""The C ABI from C: tests/c_abi_consumer.c includes only include/gemm14.h
and links libgemm14.so (and libcudart). The CPU test compiles and links it as
C; the GPU test runs it (exact integer products through the device-pointer,
workspace and host-buffer calls)."""
import os
import subprocess

import pytest

import dense_gemm_14_gb300 as g14

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_consumer(tmp_path) -> str:
    lib = g14.lib_path()
    exe = str(tmp_path / "c_abi_consumer")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           os.path.join(ROOT, "tests", "c_abi_consumer.c"), "-o", exe,
           lib, "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(CUDA, "lib64")]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_header_compiles_and_links_as_c(tmp_path):
    g14.load()
    assert os.path.exists(build_consumer(tmp_path))


@pytest.mark.gpu
def test_c_consumer_runs(tmp_path):
    exe = build_consumer(tmp_path)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr[-2000:]
    assert "all checks passed" in out.stdout
