"""Seeded synthetic inputs for the gx_gemm step update (shared by the tests, the bench and the oracle checks).

This module holds no arithmetic of the method itself: it only draws numbers. Both sides of every parity check (the
CUDA library and the CPU oracle) receive the very same arrays from here.

Generator (our own definition; the pages name none): SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) run in counter mode. The key of a stream is derived from (seed, workload id, tensor
id, value-set id, sub-stream id) by repeated SplitMix64 mixing; element k of a stream is mix(key + (k + 1) * golden).
Normals use the Box-Muller transform in float64 on the uniforms of elements 2k and 2k + 1, then one rounding to float32.

Workloads: the five configurations of the gx_gemm page (sparse_delta_memory/cuda/gx_gemm_cuda.py, the module
docstring's step formula) as used for parity and measurement; see `WORKLOADS`.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = ["Workload", "WORKLOADS", "VALUE_SETS", "uniform01", "normal", "fill_normal", "make_inputs",
           "make_source", "misaligned_copy"]

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_S30, _S27, _S31, _S11 = np.uint64(30), np.uint64(27), np.uint64(31), np.uint64(11)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (wrapping uint64 arithmetic)."""
    z = (z ^ (z >> _S30)) * _M1
    z = (z ^ (z >> _S27)) * _M2
    return z ^ (z >> _S31)


def _mix_int(v: int) -> int:
    m = (1 << 64) - 1
    v &= m
    v = ((v ^ (v >> 30)) * 0xBF58476D1CE4E5B9) & m
    v = ((v ^ (v >> 27)) * 0x94D049BB133111EB) & m
    return v ^ (v >> 31)


def stream_key(*fields: int) -> int:
    """64-bit key of one counter stream, from integer fields (seed, workload, tensor, value set, sub-stream)."""
    k = 0
    for f in fields:
        k = _mix_int(k + 0x9E3779B97F4A7C15 + (int(f) & ((1 << 64) - 1)))
    return k


def _raw(key: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(key) + idx * _G)


def uniform01(key: int, start: int, count: int) -> np.ndarray:
    """Uniforms in (0, 1]: ((u64 >> 11) + 1) * 2^-53, float64."""
    return ((_raw(key, start, count) >> _S11).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(key: int, start: int, count: int) -> np.ndarray:
    """Standard normals (float64) of elements start .. start + count - 1 of the stream: Box-Muller (cosine branch) on
    uniforms 2k and 2k + 1."""
    u = uniform01(key, 2 * start, 2 * count)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos((2.0 * np.pi) * u2)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _fill(out: np.ndarray, fn) -> None:
    """out (flat float32) [a:b] = fn(a, b - a), in parallel chunks (numpy releases the GIL)."""
    n = out.size
    spans = [(a, min(n, a + _CHUNK)) for a in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for a, b in spans:
            out[a:b] = fn(a, b - a)
        return

    def work(ab):
        a, b = ab
        out[a:b] = fn(a, b - a)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, spans))


def fill_normal(out: np.ndarray, key: int, scale: float = 1.0) -> None:
    """Fill the flat float32 array `out` with float32(scale * N(0,1)) of stream `key`."""
    flat = out.reshape(-1)
    _fill(flat, lambda a, c: (normal(key, a, c) * scale).astype(np.float32))


# ---------------------------------------------------------------------------------------------------------------------
# Value sets (edge-pattern workload). The fractions and scales are our reading of "six seeded value sets: all zeros,
# +-1e30 magnitudes, denormals (~1e-40), mixed +-Inf, NaN sprinkled at 1%, and N(0,1)", plus three extra variants.
VALUE_SETS = ("normal", "zeros", "zeros_signed", "big", "wide", "denormal", "denormal_all", "inf", "nan")
_SET_ID = {s: i + 1 for i, s in enumerate(VALUE_SETS)}
_TENSOR_ID = {"x": 1, "d_dv": 2, "d_u": 3, "S": 4}
_SUB_NORMAL, _SUB_MASK, _SUB_SIGN, _SUB_EXP = 0, 1, 2, 3


def _value_set_fn(vset: str, tensor: str, keyf, scale: float):
    kn = keyf(_SUB_NORMAL)
    km = keyf(_SUB_MASK)
    ks = keyf(_SUB_SIGN)
    ke = keyf(_SUB_EXP)

    def f(a, c):
        if vset == "normal":
            return (normal(kn, a, c) * scale).astype(np.float32)
        if vset == "zeros":
            return np.zeros(c, np.float32)
        if vset == "zeros_signed":
            neg = uniform01(ks, a, c) <= 0.5
            return np.where(neg, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
        if vset == "big":
            return (normal(kn, a, c) * 1e30).astype(np.float32)
        if vset == "wide":
            e = np.floor(uniform01(ke, a, c) * 121.0 - 1e-12).astype(np.int64) - 60   # integer in [-60, 60]
            return np.ldexp(normal(kn, a, c), e).astype(np.float32)
        if vset == "denormal":
            s = 1e-40 if tensor == "d_u" else 1e-20
            return (normal(kn, a, c) * s).astype(np.float32)
        if vset == "denormal_all":
            return np.full(c, 1e-40, np.float64).astype(np.float32)
        if vset in ("inf", "nan"):
            v = normal(kn, a, c).astype(np.float32)
            hit = uniform01(km, a, c) <= 0.01
            if vset == "inf":
                sgn = uniform01(ks, a, c) <= 0.5
                v[hit] = np.where(sgn[hit], np.float32(-np.inf), np.float32(np.inf))
            else:
                v[hit] = np.float32(np.nan)
            return v
        raise ValueError(f"unknown value set {vset!r}")

    return f


@dataclass(frozen=True)
class Workload:
    """One gx_gemm workload: T steps of P chunks, chunk size C, head dim hd (x [N,C,C], d_dv / d_u [N,C,hd], N = T*P).

    x_scale: 'unit' (x ~ N(0,1)) or 'inv_sqrt_c' (x ~ N(0, 1/C)). producer: d_dv(ti) is rewritten before every step by
    the synthetic producer (d_dv slice = +-S slice). pdl: steps are chained with programmatic dependent launch."""

    name: str
    wid: int
    T: int
    P: int
    C: int
    hd: int
    x_scale: str = "inv_sqrt_c"
    producer: bool = False
    pdl: bool = True
    value_sets: tuple = ("normal",)
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return self.T * self.P

    def flops_per_step(self) -> int:
        return 2 * self.C * self.C * self.hd * self.P

    def bytes_per_step(self) -> int:
        return (self.C * self.C + 3 * self.C * self.hd) * 4 * self.P


WORKLOADS = {
    "tiny": Workload("tiny", 1, T=4, P=2, C=16, hd=32, x_scale="unit", pdl=False,
                     note="T=4, P=2 (N=8), C=16, hd=32; all N(0,1)"),
    "producer_chain": Workload("producer_chain", 2, T=64, P=8, C=64, hd=64, producer=True,
                               note="T=64, P=8 (batch 2 x 4 heads), C=64, hd=64; d_dv rewritten per step by a "
                                    "synthetic producer kernel"),
    "pdl_chain": Workload("pdl_chain", 3, T=128, P=32, C=64, hd=128,
                          note="T=128, P=32 (batch 4 x 8 heads), C=64, hd=128; PDL-chained steps"),
    "edge": Workload("edge", 4, T=8, P=4, C=48, hd=100, x_scale="unit", pdl=False, value_sets=VALUE_SETS,
                     note="T=8, P=4, C=48; hd in {100, 99, 128 misaligned base, 128 with row stride 129}; value sets"),
    "large": Workload("large", 5, T=32, P=256, C=128, hd=128,
                      note="T=32, P=256 (batch 16 x 16 heads), C=128, hd=128; multi-wave"),
}


def make_inputs(w: Workload, seed: int = 0, value_set: str = "normal", hd: int | None = None,
                N: int | None = None, out: dict | None = None) -> dict:
    """x [N,C,C], d_dv [N,C,hd], d_u [N,C,hd] (float32, C-contiguous numpy) for workload `w`.

    `hd` / `N` override the workload's (edge variants, reduced parity sizes); the streams are keyed by the workload id,
    so a reduced N is a prefix of the full-size arrays. `out` may hold preallocated float32 arrays (e.g. pinned host
    memory) to fill in place."""
    hd = w.hd if hd is None else int(hd)
    N = w.N if N is None else int(N)
    C = w.C
    shapes = {"x": (N, C, C), "d_dv": (N, C, hd), "d_u": (N, C, hd)}
    res = {}
    for t, shp in shapes.items():
        arr = out[t] if out is not None and t in out else np.empty(shp, np.float32)
        assert arr.shape == shp and arr.dtype == np.float32
        scale = 1.0
        if t == "x" and w.x_scale == "inv_sqrt_c":
            scale = 1.0 / np.sqrt(C)
        keyf = (lambda sub, t=t: stream_key(seed, w.wid, _TENSOR_ID[t], _SET_ID[value_set], hd, sub))
        _fill(arr.reshape(-1), _value_set_fn(value_set, t, keyf, scale))
        res[t] = arr
    return res


def make_source(w: Workload, seed: int = 0, N: int | None = None) -> np.ndarray:
    """The producer's pre-generated source S [N, C, hd] ~ N(0,1) (the synthetic producer writes +-S into d_dv)."""
    N = w.N if N is None else int(N)
    S = np.empty((N, w.C, w.hd), np.float32)
    fill_normal(S, stream_key(seed, w.wid, _TENSOR_ID["S"], _SET_ID["normal"], w.hd, _SUB_NORMAL))
    return S


def misaligned_copy(a: np.ndarray, offset_bytes: int = 4) -> np.ndarray:
    """A C-contiguous copy of `a` whose data pointer sits `offset_bytes` past a 64-byte boundary (host memory)."""
    nbytes = a.nbytes
    buf = np.empty(nbytes + 128, np.uint8)
    base = buf.ctypes.data
    off = (-base) % 64 + offset_bytes
    view = buf[off:off + nbytes].view(a.dtype).reshape(a.shape)
    view[...] = a
    return view
