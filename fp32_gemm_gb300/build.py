"""Builds the gx_gemm CUDA library (libsdm_gx_gemm.so) in-tree for sm_103a with nvcc.

Translation units are compiled in parallel, then linked into one shared library with the CUDA runtime linked
statically. Nothing is installed: the library lands in fp32_gemm_gb300/lib/. build(trace=True) builds the timeline
variant (libsdm_gx_gemm_trace.so: the same kernels with per-CTA global-timer stamps, sdm_gx_gemm_plan_set_trace), which
the binding loads when SDM_GX_TRACE_BUILD=1 is set.
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libsdm_gx_gemm.so")
TRACE_LIB = os.path.join(LIBDIR, "libsdm_gx_gemm_trace.so")
SOURCES = ("gx_host.cu", "gx_tma.cu", "gx_generic.cu")
HEADERS = ("gx_internal.h", "gx_device.cuh")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-Xcompiler", "-fvisibility=hidden",
              "-diag-suppress", "1160", "-diag-suppress", "177"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Compile (if stale) and link the library (trace=True: its timeline variant); returns its path. Raises
    CalledProcessError on a compiler error."""
    obj_dir = os.path.join(OBJ, "trace") if trace else OBJ
    lib = TRACE_LIB if trace else LIB
    defines = ["-DSDMGX_TRACE"] if trace else []
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    inc = ["-I", os.path.join(ROOT, "include"), "-I", CSRC]
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "sdm_gx_gemm.h")]
    nvcc = _nvcc()

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src.replace(".cu", ".o"))
        if force or _stale(o, [s, *hdrs]):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, *defines, *inc, "-c", s, "-o", o + ".tmp"]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            subprocess.run(cmd, check=True)
            os.replace(o + ".tmp", o)
        return o

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, trace="--trace" in sys.argv))
