"""Build of libmcemu.so: nvcc for sm_103a, one object per translation unit, in parallel.

The library is built in-tree (next to this file) and loaded by ``binding``; nothing is
installed.  ``build()`` is what the package's entry point and the tests call.
"""
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_PATH = os.path.join(HERE, "libmcemu.so")
SOURCES = ["api.cu", "stream.cu", "stream_fp8.cu", "gemm.cu", "gemm_fast.cu", "gemm_fast_sw.cu", "gemm_exact.cu", "sparse.cu", "multiword.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(HERE, "..", "include")]


def _nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmcemu.so")
    return exe


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(HERE, "..", "include", "mcemu.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        build_peak()
        return LIB_PATH
    nvcc = _nvcc()
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    build_peak()
    return LIB_PATH


PEAK_PATH = os.path.join(HERE, "libmcpeak.so")


def build_peak() -> str:
    """The pipe-peak microbenchmark (csrc/peak.cu) that the benchmark uses for its
    integer rooflines; a library of its own, not part of the emulator."""
    src = os.path.join(CSRC, "peak.cu")
    if os.path.exists(PEAK_PATH) and os.path.getmtime(PEAK_PATH) >= os.path.getmtime(src):
        return PEAK_PATH
    tmp = PEAK_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([_nvcc(), *ARCH, *FLAGS, "-shared", "-o", tmp, src, "-lcudart"], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on peak.cu:\n{r.stderr}")
    os.replace(tmp, PEAK_PATH)
    return PEAK_PATH


if __name__ == "__main__":
    import sys
    import time
    t = time.time()
    print(build(force=True, verbose="-v" in sys.argv), f"{time.time() - t:.1f}s")
