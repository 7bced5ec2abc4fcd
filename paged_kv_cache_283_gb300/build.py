"""Builds libpa.so (CUDA kernels for sm_103a + the C ABI + the host block
allocator) in-tree with nvcc.  No torch extension machinery: the library is
a plain shared object that the ctypes binding in ``pa.py`` loads.

Objects and the ptxas report (registers, spills, shared memory per kernel)
go to ``_build/``; the library goes next to this file.  Sources compile in
parallel; an unchanged tree is not rebuilt.
"""
import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpa.so")

SOURCES = ["api.cu", "decode.cu", "splitk_reduce.cu", "reshape_and_cache.cu", "copy_blocks.cu",
           "noalloc.cu", "prefill.cu", "allocator.cpp", "sha256.cpp",
           "scheduler.cpp", "splitk_plan.cpp"]
HEADERS = [os.path.join(ROOT, "include", "pa.h"), os.path.join(CSRC, "internal.h"),
           os.path.join(CSRC, "device.cuh"), os.path.join(CSRC, "decode_tile.cuh"),
           os.path.join(CSRC, "sha256.h"), os.path.join(CSRC, "cache_row.cuh")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CU_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-Xptxas", "-v", "--expt-relaxed-constexpr"]
CPP_FLAGS = ["-O2", "-std=c++17", "-Xcompiler", "-fPIC"]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: set NVCC or put CUDA's bin directory on PATH")


def _stamp():
    h = hashlib.sha256()
    h.update(" ".join(CU_FLAGS + CPP_FLAGS).encode())
    for f in [os.path.join(CSRC, s) for s in SOURCES] + HEADERS:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _compile(src):
    path = os.path.join(CSRC, src)
    obj = os.path.join(BUILD, src + ".o")
    flags = CU_FLAGS if src.endswith(".cu") else CPP_FLAGS
    cmd = [nvcc()] + flags + ["-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(BUILD, src + ".log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
    return obj


def build(force=False, verbose=False):
    """Compile and link libpa.so if anything changed; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp_file = os.path.join(BUILD, "stamp")
    stamp = _stamp()
    if not force and os.path.exists(LIB) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read() == stamp:
                return LIB
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(_compile, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    if verbose:
        for src in SOURCES:
            with open(os.path.join(BUILD, src + ".log")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
