"""Build the CUDA library (libgemm12.so) in-tree with nvcc, for sm_103a only.

Each translation unit under ``csrc/`` is compiled in parallel to an object in
``_build/``, then linked into ``_build/libgemm12.so`` with the CUDA runtime
linked statically (the library needs no libcuda at link time: the one driver
entry point it uses, cuTensorMapEncodeTiled, is looked up at run time).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libgemm12.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

SOURCES = ["api.cu", "sgemm_simt.cu", "bf16_tc.cu", "bf16_decode.cu", "decode_noalloc.cu"]
HEADERS = ["ptx.cuh", "internal.h", "epilogue.cuh", "dispatch_table.inc"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc_path() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _newest_input() -> float:
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    paths.append(os.path.join(INCLUDE, "gemm12.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def _compile(nvcc: str, src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, proc.stdout, proc.stderr))
    return obj, proc.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libgemm12.so if any source is newer; return its path.

    The ptxas resource report (registers, spills, shared memory per kernel)
    is written to ``_build/ptxas.log``.
    """
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _newest_input():
        return LIB_PATH
    nvcc = nvcc_path()
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s), SOURCES))
    objs = [r[0] for r in results]
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        for src, (_, log) in zip(SOURCES, results):
            f.write("==== %s\n%s\n" % (src, log))
    if verbose:
        for _, log in results:
            print(log)
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    proc = subprocess.run(cmd, capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (proc.stdout, proc.stderr))
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
