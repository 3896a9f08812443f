"""The oracle's pins must catch plausible mistakes: each mutant below is the oracle's C source with one slip planted
(on the CPU, in a temporary copy), and at least one pin has to reject it."""

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth
from tests.ieee32 import chain_element

SRC = open(os.path.join(os.path.dirname(oracle.__file__), "gx_gemm_oracle.c")).read()

MUTANTS = {
    "x_untransposed": ("x[n * x_sn + j * x_sj + i]", "x[n * x_sn + i * x_sj + j]"),
    "j_reversed": ("for (int64_t j = 0; j < C; ++j) {\n        acc = fmaf(x[n * x_sn + j * x_sj + i], "
                   "d_dv[n * dv_sn + j * dv_sj + c], acc);",
                   "for (int64_t jj = 0; jj < C; ++jj) {\n        const int64_t j = C - 1 - jj;\n"
                   "        acc = fmaf(x[n * x_sn + j * x_sj + i], d_dv[n * dv_sn + j * dv_sj + c], acc);"),
    "chain_from_du": ("float acc = 0.0f;\n    for", "float acc = du_old;\n    du_old = 0.0f;\n    for"),
    "unfused": ("acc = fmaf(x[n * x_sn + j * x_sj + i], d_dv[n * dv_sn + j * dv_sj + c], acc);",
                "{ volatile float pr = x[n * x_sn + j * x_sj + i] * d_dv[n * dv_sn + j * dv_sj + c]; acc = acc + pr; }"),
    "last_term_dropped": ("for (int64_t j = 0; j < C; ++j) {", "for (int64_t j = 0; j < C - 1; ++j) {"),
    "wrong_sign": ("return du_old + acc;", "return du_old - acc;"),
    "start_negative_zero": ("float acc = 0.0f;", "float acc = -0.0f;"),
    "wrong_chunk": ("const int64_t n = ti * P + p;", "const int64_t n = ti + p;"),
    "d_dv_row_col_swapped": ("d_dv[n * dv_sn + j * dv_sj + c]", "d_dv[n * dv_sn + c * dv_sj + j]"),
}


def _build_mutant(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) >= 1, name
    src = SRC.replace(old, new)
    # keep the environment self-check from rejecting the unfused mutant before the pins can
    src = src.replace("if (!oracle_fp_env_ok()) return -1;", "")
    # scratch inside the repository (the oracle's own git-ignored build folder), one folder per mutant
    d = os.path.join(os.path.dirname(oracle.__file__), "_build", "mutants", name)
    os.makedirs(d, exist_ok=True)
    c = os.path.join(d, "m.c")
    so = os.path.join(d, "m.so")
    open(c, "w").write(src)
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, c, "-lm"], check=True)
    L = ctypes.CDLL(so)
    L.oracle_gx_gemm_step.restype = ctypes.c_int
    L.oracle_gx_gemm_step.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 10
    return L


def _step(L, d_u, x, d_dv, ti, P):
    out = d_u.copy()
    N, C, _ = x.shape
    hd = d_u.shape[2]
    s = oracle.chunk_strides(x, d_dv, out)
    L.oracle_gx_gemm_step(out.ctypes.data, x.ctypes.data, d_dv.ctypes.data, ti, P, C, hd, *s)
    return out


def _pins_pass(L) -> bool:
    """A compact run of the pins (integer exactness, permutation x, j order, final add, fusion, signed zero,
    brute force); False as soon as one rejects the library."""
    bits = lambda a: np.ascontiguousarray(a, np.float32).view(np.uint32)  # noqa: E731
    rng = np.random.default_rng(5)
    C, hd, P = 12, 7, 2
    x = rng.integers(-4, 5, (2 * P, C, C)).astype(np.float32)
    dv = rng.integers(-4, 5, (2 * P, C, hd)).astype(np.float32)
    du = rng.integers(-100, 101, (2 * P, C, hd)).astype(np.float32)
    got = _step(L, du, x, dv, 1, P)
    want = du.astype(np.int64).copy()
    want[P:] += np.einsum("nji,njc->nic", x[P:].astype(np.int64), dv[P:].astype(np.int64))
    if not np.array_equal(got.astype(np.int64), want):
        return False
    # permutation x (not an involution)
    pi = np.roll(np.arange(C), 1)
    xp = np.zeros((2, C, C), np.float32)
    for i in range(C):
        xp[:, pi[i], i] = 1.0
    dvp = rng.standard_normal((2, C, hd)).astype(np.float32)
    dup = rng.standard_normal((2, C, hd)).astype(np.float32)
    gp = _step(L, dup, xp, dvp, 0, 2)
    if not np.array_equal(bits(gp), bits(dup + dvp[:, pi, :])):
        return False
    # j order
    xj = np.zeros((1, 3, 3), np.float32)
    xj[0, :, 0] = [1.0, 1e8, -1e8]
    gj = _step(L, np.zeros((1, 3, 1), np.float32), xj, np.ones((1, 3, 1), np.float32), 0, 1)
    if gj[0, 0, 0] != 0.0:
        return False
    # final add separate
    gf = _step(L, np.full((1, 8, 1), 1e8, np.float32), np.ones((1, 8, 8), np.float32), np.ones((1, 8, 1), np.float32),
               0, 1)
    if not np.all(gf == np.float32(1e8 + 8)):
        return False
    # fusion
    xf = np.zeros((1, 2, 2), np.float32)
    xf[0, :, 0] = [1.0, 1.0 + 2 ** -23]
    gfu = _step(L, np.zeros((1, 2, 1), np.float32), xf, np.array([[[-1.0], [1.0 - 2 ** -23]]], np.float32), 0, 1)
    if gfu[0, 0, 0] != np.float32(-(2.0 ** -46)):
        return False
    # signed zero: all-zero inputs give +0
    z = np.zeros((2, 4, 4), np.float32)
    gz = _step(L, -z, z, -z[:, :, :4], 0, 2)
    if np.any(bits(gz) != 0):
        return False
    # brute force against exact rational arithmetic
    w = synth.Workload("mut", 99, T=2, P=2, C=4, hd=3, x_scale="unit")
    inp = synth.make_inputs(w, seed=1, value_set="wide")
    gb = _step(L, inp["d_u"], inp["x"], inp["d_dv"], 1, 2)
    for n in (2, 3):
        for i in range(4):
            for c in range(3):
                e = chain_element(inp["x"][n, :, i], inp["d_dv"][n, :, c], inp["d_u"][n, i, c])
                if bits(gb[n, i, c]) != bits(e):
                    return False
    return True


def test_unmutated_source_passes():
    L = ctypes.CDLL(oracle.build())
    L.oracle_gx_gemm_step.restype = ctypes.c_int
    L.oracle_gx_gemm_step.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 10
    assert _pins_pass(L)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert not _pins_pass(_build_mutant(name)), f"mutant {name} slipped through the pins"
