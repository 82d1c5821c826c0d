"""Build libgemm_gb300.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Translation units compile in parallel; the link uses nvcc's static CUDA runtime,
so the library depends only on the driver (loaded lazily by the runtime).
Beside it, gcc builds _gemm_pycall (CPython entry points for the per-call
functions; the binding uses ctypes for them when it cannot be built).
"""
from __future__ import annotations

import os
import subprocess
import sys
import sysconfig
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libgemm_gb300.so")

SOURCES = ["gemm_api.cu", "gemm_aux.cu", "gemm_inst_f16.cu", "gemm_inst_bf16.cu",
           "gemm_inst_i32.cu", "gemm_inst_f16_pair.cu", "gemm_inst_bf16_pair.cu",
           "gemm_inst_i32_pair.cu", "gemm_noalloc.cu", "gemm_probe.cu", "tma_intensity.cu"]
PYCALL_SRC = os.path.join(CSRC, "gemm_pycall.c")
PYCALL_PATH = os.path.join(PKG, "_gemm_pycall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-I", CSRC, *extra]


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if not f.endswith(".c")]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(f) > t for f in _deps())


def build_library(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library if any source is newer than it; return its path."""
    if not force and not ptxas_info and not _stale(LIB_PATH):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc(), *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            if err.strip():
                sys.stderr.write(err)
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def build_pycall(force: bool = False) -> str | None:
    """Compile the CPython entry-point module; None (with a note on stderr) if this
    interpreter's headers or a C compiler are missing."""
    if (not force and os.path.exists(PYCALL_PATH)
            and os.path.getmtime(PYCALL_PATH) >= os.path.getmtime(PYCALL_SRC)):
        return PYCALL_PATH
    inc = sysconfig.get_paths().get("include", "")
    if not os.path.exists(os.path.join(inc, "Python.h")):
        sys.stderr.write("_gemm_pycall not built: no Python.h in %s\n" % inc)
        return None
    tmp = PYCALL_PATH + ".tmp.%d" % os.getpid()
    cmd = [os.environ.get("CC", "gcc"), "-O2", "-shared", "-fPIC", "-I", inc, PYCALL_SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write("_gemm_pycall not built:\n%s\n%s" % (" ".join(cmd), r.stderr))
        return None
    os.replace(tmp, PYCALL_PATH)
    return PYCALL_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True,
                        ptxas_info="--ptxas-info" in sys.argv))
    print(build_pycall(force="--force" in sys.argv))
