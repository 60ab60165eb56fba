"""Build libkvq.so (the C-ABI CUDA library) in-tree for sm_103a.

Each CUDA translation unit is compiled by its own nvcc process (in parallel),
then linked into ``decode_attention_quantized_gb300/lib/libkvq.so``.  A stamp
of the sources and flags skips rebuilds when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libkvq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I" + INCLUDE, "-I" + CSRC] + ARCH
SOURCES = ["api.cu", "append.cu", "combine.cu", "decode_int8.cu", "decode_fp8.cu", "decode_int4.cu",
           "decode_tc_int8.cu", "decode_tc_fp8.cu", "decode_tc_int4.cu", "decode_tc_grp_int8.cu",
           "decode_tc_grp_fp8.cu", "decode_tc_grp_int4.cu", "decode_qt_int8.cu", "decode_qt_fp8.cu",
           "decode_qt_int4.cu", "noalloc.cu"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")


HEADERS = ["kvq_internal.h", "ptx.cuh", "pipeline.cuh", "decode.cuh", "decode_tc.cuh", "decode_qt.cuh"]


def _stamp() -> str:
    """Digest of the library's own source files (a fixed list, so stray files
    in the folders change nothing) and the compiler flags, with the flags'
    machine-specific include paths left out."""
    h = hashlib.sha256()
    h.update(" ".join(f for f in NVCC_FLAGS if not f.startswith("-I")).encode())
    files = [os.path.join(CSRC, n) for n in SOURCES + HEADERS] + [os.path.join(INCLUDE, "kvq.h")]
    for path in files:
        with open(path, "rb") as f:
            h.update(os.path.basename(path).encode())
            h.update(f.read().replace(b"\r\n", b"\n"))
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libkvq.so; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    stamp_path = os.path.join(BUILD_DIR, "stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return LIB_PATH
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for (_, log), src in zip(results, SOURCES):
            if log.strip():
                print(f"--- {src}\n{log}", file=sys.stderr)
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
