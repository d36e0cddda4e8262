"""Builds libgemm14.so in-tree (dense_gemm_14_gb300/_build/) with nvcc for sm_103a.

The translation units are compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically, so the library depends on
nothing but the driver (libcuda, reached at run time) and libc/libstdc++.

    python -m dense_gemm_14_gb300.build [--force] [--verbose] [--checked]

--checked builds the variant with the device-side bounds checks
(-DGEMM14_DEVICE_CHECKS, csrc/checks.h) into _build_checked/; select it at run
time with GEMM14_LIB=<path of its libgemm14.so>.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
CHECKED_BUILD_DIR = os.path.join(HERE, "_build_checked")
CHECKED_FLAGS = ["-DGEMM14_DEVICE_CHECKS"]
LIB_NAME = "libgemm14.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["api.cu", "sgemm_simt.cu", "sgemm_small.cu", "hgemm_tc.cu", "hgemm_tc2.cu",
           "sgemm_tc3.cu", "epilogue.cu", "host_path.cu", "copy.cu", "plan.cu"]
HEADERS = ["ptx.cuh", "kernels.h", "streamk.cuh", "api_internal.h", "plan.h", "checks.h",
           "libgemm14.map"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-lineinfo", "-O3", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-Xptxas", "-v",
    "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put it on PATH)")


def _stale(lib: str, inputs) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in inputs)


def build(force: bool = False, verbose: bool = False, extra_flags=(), out_dir: str | None = None,
          checked: bool = False) -> str:
    """Compiles every .cu and links libgemm14.so; returns its path.

    extra_flags (e.g. schedule macros such as -DSGEMM_UNROLL=2) and out_dir
    allow building variants side by side; the default build is the product.
    checked: the variant with the device-side bounds checks, in its own folder
    (rebuilt only when a source changed, like the product).
    """
    if checked:
        extra_flags = list(extra_flags) + CHECKED_FLAGS
        out_dir = out_dir or CHECKED_BUILD_DIR
    build_dir = out_dir or BUILD_DIR
    lib_path = os.path.join(build_dir, LIB_NAME)
    os.makedirs(build_dir, exist_ok=True)
    inputs = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    inputs.append(os.path.join(INCLUDE, "gemm14.h"))
    inputs.append(os.path.abspath(__file__))
    if not force and (checked or not extra_flags) and not _stale(lib_path, inputs):
        return lib_path
    cc = nvcc()
    procs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        log = os.path.join(build_dir, src.replace(".cu", ".ptxas.log"))
        cmd = [cc, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-c", os.path.join(CSRC, src),
               "-o", obj]
        fh = open(log, "w")
        procs.append((src, obj, log, fh, subprocess.Popen(cmd, stdout=fh, stderr=subprocess.STDOUT)))
    failed = []
    for src, obj, log, fh, p in procs:
        rc = p.wait()
        fh.close()
        if rc != 0:
            failed.append((src, log))
        elif verbose:
            sys.stdout.write(open(log).read())
    if failed:
        msgs = "\n".join(f"--- {s} ---\n{open(l).read()}" for s, l in failed)
        raise RuntimeError(f"nvcc failed for {[s for s, _ in failed]}:\n{msgs}")
    tmp = lib_path + f".tmp{os.getpid()}"
    objs = [o for _, o, _, _, _ in procs]
    subprocess.run([cc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-Xlinker", "--version-script=" + os.path.join(CSRC, "libgemm14.map"),
                    "-o", tmp, *objs], check=True)
    os.replace(tmp, lib_path)
    return lib_path


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true",
                    help="the variant with device-side bounds checks, in _build_checked/")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose, checked=a.checked))


if __name__ == "__main__":
    main()
