"""CPU oracle of the gx_gemm step update -- TEST INFRASTRUCTURE ONLY.

Only the tests, `__graft_entry__.smoke()` and the bench's `cpu_baseline` / reference leg may import this package.
The product path (the CUDA library and its Python binding) never imports it and shares no code with it.

The arithmetic lives in `gx_gemm_oracle.c` (plain C: the defining loop nest with fmaf in j order and one separately
rounded add; sparse_delta_memory/cuda/gx_gemm_cuda.py, module docstring formula and gx_gemm_kernel's chain and
epilogue). This module compiles it with gcc (`-O2 -ffp-contract=off`, no fast-math) and wraps it with ctypes.

The synthetic producer (`producer_step`) is not on the pages: it stands in for the kernel that writes d_dv(ti) right
before each step (our reading): d_dv slice ti = S slice ti, negated when ti is odd (exact).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gx_gemm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_gx_gemm.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]
_lock = threading.Lock()
_lib = None

__all__ = ["build", "lib", "fp_env_ok", "step", "run_steps", "points", "producer_step", "chunk_strides",
           "successor_rows"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc) if it is missing or older than its source. Returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, fp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            L.oracle_fp_env_ok.restype = ctypes.c_int
            L.oracle_gx_gemm_step.restype = ctypes.c_int
            L.oracle_gx_gemm_step.argtypes = [fp, fp, fp] + [i64] * 10
            L.oracle_gx_gemm_points.restype = ctypes.c_int
            L.oracle_gx_gemm_points.argtypes = [fp, fp, fp, fp, ip, ip, ip] + [i64] * 7
            L.oracle_gx_gemm_element.restype = ctypes.c_float
            L.oracle_gx_gemm_element.argtypes = [fp, fp, ctypes.c_float] + [i64] * 8
            _lib = L
    return _lib


def fp_env_ok() -> bool:
    return bool(lib().oracle_fp_env_ok())


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def chunk_strides(x: np.ndarray, d_dv: np.ndarray, d_u: np.ndarray):
    """Element strides (x_sn, x_sj, dv_sn, dv_sj, du_sn, du_si) of 3-D float32 arrays with unit innermost stride."""
    for a in (x, d_dv, d_u):
        assert a.dtype == np.float32 and a.ndim == 3 and a.strides[2] == 4, "float32 [N, rows, cols], unit inner stride"
    e = 4
    return (x.strides[0] // e, x.strides[1] // e, d_dv.strides[0] // e, d_dv.strides[1] // e,
            d_u.strides[0] // e, d_u.strides[1] // e)


def step(d_u: np.ndarray, x: np.ndarray, d_dv: np.ndarray, ti: int, P: int) -> None:
    """One step ti in place on d_u: chunks n = ti*P + p, p < P. Arrays are float32 [N, C, C] / [N, C, hd] views with
    unit innermost stride (other strides arbitrary)."""
    N, C, _ = x.shape
    hd = d_u.shape[2]
    assert x.shape[2] == C and d_u.shape[:2] == (N, C) and d_dv.shape == (N, C, hd)
    assert 0 <= ti and (ti + 1) * P <= N
    assert d_u.flags.writeable
    s = chunk_strides(x, d_dv, d_u)
    rc = lib().oracle_gx_gemm_step(_ptr(d_u), _ptr(x), _ptr(d_dv), ti, P, C, hd, *s)
    if rc != 0:
        raise RuntimeError("oracle: floating-point environment flushes subnormals or fmaf is not fused")


def run_steps(d_u, x, d_dv, P: int, order=None, producer_src=None) -> None:
    """Apply the steps in `order` (default: ti = 0 .. N/P - 1). With `producer_src`, the synthetic producer rewrites
    d_dv(ti) from it right before each step."""
    T = x.shape[0] // P
    for ti in (range(T) if order is None else order):
        if producer_src is not None:
            producer_step(d_dv, producer_src, ti, P)
        step(d_u, x, d_dv, ti, P)


def points(d_u, x, d_dv, n, i, c) -> np.ndarray:
    """The updated values of d_u[n[k], i[k], c[k]] (d_u itself untouched), float32 [len(n)]."""
    n = np.ascontiguousarray(n, np.int64)
    i = np.ascontiguousarray(i, np.int64)
    c = np.ascontiguousarray(c, np.int64)
    assert n.shape == i.shape == c.shape and n.ndim == 1
    C = x.shape[1]
    out = np.empty(n.shape[0], np.float32)
    s = chunk_strides(x, d_dv, d_u)
    rc = lib().oracle_gx_gemm_points(_ptr(out), _ptr(d_u), _ptr(x), _ptr(d_dv), _ptr(n), _ptr(i), _ptr(c),
                                     n.shape[0], C, *s)
    if rc != 0:
        raise RuntimeError("oracle: floating-point environment flushes subnormals or fmaf is not fused")
    return out


def producer_step(d_dv: np.ndarray, S: np.ndarray, ti: int, P: int) -> None:
    """The synthetic producer (not on the pages; our stand-in for the kernel that writes d_dv(ti)): d_dv chunks of step
    ti = S chunks of step ti, negated when ti is odd. Negation is exact (sign bit only)."""
    sl = slice(ti * P, (ti + 1) * P)
    if ti % 2:
        np.negative(S[sl], out=d_dv[sl])
    else:
        d_dv[sl] = S[sl]


def successor_rows(d_u: np.ndarray, ti: int, P: int) -> np.ndarray:
    """The synthetic successor (not on the pages; a stand-in for the next kernel of the backward step, which reads d_u
    after the step): for each chunk n of step ti, the sum of its leading row d_u[n, 0, :] in this fixed order: 32
    partial sums, partial l = d_u[n, 0, l] + d_u[n, 0, l + 32] + ... added left to right from +0, then for offsets 16,
    8, 4, 2, 1: partial[l] = partial[l] + partial[l ^ offset] for all l at once; the result is partial[0]. Every add
    is one float32 rounding. Returns float32 [P]."""
    rows = d_u[ti * P:(ti + 1) * P, 0, :]
    hd = rows.shape[1]
    part = np.zeros((rows.shape[0], 32), np.float32)
    for c in range(hd):
        part[:, c % 32] = part[:, c % 32] + rows[:, c]
    lanes = np.arange(32)
    for off in (16, 8, 4, 2, 1):
        part = part + part[:, lanes ^ off]
    return part[:, 0].copy()
