"""Pins of the CPU oracle against facts fixed by the mathematics, independent of the oracle's own code.

The step update (sparse_delta_memory/cuda/gx_gemm_cuda.py, module docstring formula; gx_gemm_kernel's chain and
epilogue): acc = +0; acc = fmaf(x[n,j,i], d_dv[n,j,c], acc) for j = 0..C-1; d_u[n,i,c] = d_u[n,i,c] + acc.

Each test below would fail for a plausible slip in the oracle: a dropped or extra term, a wrong sign, x used
untransposed (x[n,i,j]), a reversed or reordered j loop, the chain started from d_u instead of +0, a product rounded
before the add (no fusion), flushed subnormals, a double rounding of the final add, or a wrong chunk / step offset.
"""

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests.ieee32 import add32, chain_element, fma32, round_f32

RNG_SEED = 20261202


def bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def assert_bitwise(got, want, allow_nan_class=True):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape
    gn, wn = np.isnan(got), np.isnan(want)
    assert np.array_equal(gn, wn), f"NaN positions differ: {np.argwhere(gn != wn)[:5]}"
    m = ~gn
    bad = np.flatnonzero(bits(got)[m] != bits(want)[m])
    assert bad.size == 0, f"{bad.size} mismatches, first: got {got[m][bad[:4]]} want {want[m][bad[:4]]}"


def run_oracle_step(x, d_dv, d_u, ti, P):
    out = d_u.copy()
    oracle.step(out, x, d_dv, ti, P)
    return out


def test_fp_environment():
    assert oracle.fp_env_ok()


def test_ieee32_helper_self_check():
    # the exact-rational helper against hardware float32 on operations that have a single rounding in numpy
    rng = np.random.default_rng(RNG_SEED)
    a = (rng.standard_normal(300) * np.exp2(rng.integers(-140, 120, 300))).astype(np.float32)
    b = (rng.standard_normal(300) * np.exp2(rng.integers(-140, 120, 300))).astype(np.float32)
    with np.errstate(all="ignore"):
        s = a + b
    for k in range(300):
        assert bits(add32(a[k], b[k])) == bits(s[k])
    # rounding boundaries: halfway cases tie to even (1 + 2^-24 -> 1; 1 + 3 * 2^-24 -> 1 + 2^-22)
    assert float(round_f32(Fraction(1) + Fraction(1, 2 ** 24))) == 1.0
    assert float(round_f32(Fraction(1) + Fraction(3, 2 ** 24))) == 1.0 + 2.0 ** -22
    # overflow threshold and the smallest subnormal
    assert np.isinf(round_f32(Fraction(2) ** 128 - Fraction(2) ** 103))
    assert float(round_f32(Fraction(2) ** 128 - Fraction(2) ** 103 - 1)) == float(np.finfo(np.float32).max)
    assert float(round_f32(Fraction(1, 2 ** 149))) == 2.0 ** -149
    assert float(round_f32(Fraction(1, 2 ** 150))) == 0.0               # tie to even: down to 0
    assert float(round_f32(Fraction(3, 2 ** 151))) == 2.0 ** -149
    assert float(fma32(1.0 + 2 ** -23, 1.0 - 2 ** -23, -1.0)) == -(2.0 ** -46)


@pytest.mark.parametrize("vset", ["normal", "wide", "denormal", "zeros_signed", "big", "inf", "nan"])
@pytest.mark.parametrize("C,hd", [(1, 3), (2, 4), (3, 1), (5, 3), (8, 2)])
def test_brute_force_exact_rational(vset, C, hd):
    """Every output bit equals the chain evaluated with exact rational arithmetic and explicit binary32 rounding."""
    P, T = 2, 2
    w = synth.Workload("bf", 90 + C, T=T, P=P, C=C, hd=hd, x_scale="unit")
    inp = synth.make_inputs(w, seed=7, value_set=vset)
    x, dv, du = inp["x"], inp["d_dv"], inp["d_u"]
    ti = 1
    got = run_oracle_step(x, dv, du, ti, P)
    want = du.copy()
    for p in range(P):
        n = ti * P + p
        for i in range(C):
            for c in range(hd):
                want[n, i, c] = chain_element(x[n, :, i], dv[n, :, c], du[n, i, c])
    assert_bitwise(got, want)


@pytest.mark.parametrize("C,hd", [(16, 32), (64, 17), (48, 100)])
def test_error_bound_against_exact_sum(C, hd):
    """|oracle - exact| <= gamma_{C+1} * (|d_u| + sum_j |x d|) (recursive summation bound, u = 2^-24)."""
    P = 2
    w = synth.Workload("eb", 80, T=1, P=P, C=C, hd=hd, x_scale="unit")
    inp = synth.make_inputs(w, seed=3)
    x, dv, du = inp["x"], inp["d_dv"], inp["d_u"]
    got = run_oracle_step(x, dv, du, 0, P)
    x64, d64, u64 = x.astype(np.float64), dv.astype(np.float64), du.astype(np.float64)
    prods = np.einsum("nji,njc->nijc", x64, d64)          # each product exact in float64 (24 + 24 <= 53 bits)
    exact = np.empty_like(u64)
    for n in range(P):
        for i in range(C):
            for c in range(hd):
                exact[n, i, c] = math.fsum([u64[n, i, c], *prods[n, i, :, c]])
    absum = np.abs(u64) + np.abs(prods).sum(axis=2)
    k = C + 1
    u = 2.0 ** -24
    gamma = k * u / (1 - k * u)
    err = np.abs(got.astype(np.float64) - exact)
    assert np.all(err <= gamma * absum * (1 + 1e-12) + 1e-300)
    # and the error is not identically zero (the chain really rounds: a fake exact-sum oracle would fail this)
    assert np.count_nonzero(got.astype(np.float64) != exact) > 0


@pytest.mark.parametrize("C,hd,P", [(16, 32, 2), (64, 64, 3), (48, 99, 2), (64, 1, 1)])
def test_small_integers_exact(C, hd, P):
    """Integer entries in [-4, 4]: every partial sum is an integer below 2^24, so the result is exactly
    d_u + x^T d_dv (computed here with int64 arithmetic)."""
    rng = np.random.default_rng(RNG_SEED + C)
    N = 2 * P
    x = rng.integers(-4, 5, (N, C, C)).astype(np.float32)
    dv = rng.integers(-4, 5, (N, C, hd)).astype(np.float32)
    du = rng.integers(-1000, 1001, (N, C, hd)).astype(np.float32)
    ti = 1
    got = run_oracle_step(x, dv, du, ti, P)
    xi, di, ui = x.astype(np.int64), dv.astype(np.int64), du.astype(np.int64)
    want = ui.copy()
    sl = slice(ti * P, (ti + 1) * P)
    want[sl] = ui[sl] + np.einsum("nji,njc->nic", xi[sl], di[sl])
    assert np.array_equal(got.astype(np.int64), want)
    # -0 never appears (integer zero results are +0)
    assert not np.any(np.signbit(got) & (got == 0))


def test_j_order():
    """Products (1, 1e8, -1e8) summed in j order give 0 (1 + 1e8 rounds to 1e8); the order (1e8, -1e8, 1) gives 1."""
    C, hd = 3, 2
    x = np.zeros((1, C, C), np.float32)
    dv = np.ones((1, C, hd), np.float32)
    du = np.zeros((1, C, hd), np.float32)
    x[0, :, 0] = [1.0, 1e8, -1e8]          # output row i = 0
    x[0, :, 1] = [1e8, -1e8, 1.0]          # output row i = 1
    x[0, :, 2] = [-1e8, 1e8, 1.0]          # row 2: the reversed order of row 0
    got = run_oracle_step(x, dv, du, 0, 1)
    assert got[0, 0, 0] == 0.0 and not np.signbit(got[0, 0, 0])
    assert got[0, 1, 0] == 1.0
    assert got[0, 2, 0] == 1.0


def test_final_add_is_separate_from_chain():
    """d_u = 1e8 and eight unit products: the chain gives 8 and 1e8 + 8 is exact. Starting the chain from d_u would
    lose every +1 (1e8 + 1 rounds to 1e8)."""
    C = 8
    x = np.ones((1, C, C), np.float32)
    dv = np.ones((1, C, 1), np.float32)
    du = np.full((1, C, 1), 1e8, np.float32)
    got = run_oracle_step(x, dv, du, 0, 1)
    assert np.all(got == np.float32(1e8 + 8))


def test_fused_not_two_roundings():
    """j = 0 gives acc = -1; j = 1 adds the product (1 + 2^-23)(1 - 2^-23) = 1 - 2^-46. Fused, the sum is -2^-46
    exactly; a product rounded first (to 1) would give 0."""
    x = np.zeros((1, 2, 2), np.float32)
    x[0, :, 0] = [1.0, 1.0 + 2 ** -23]
    dv = np.array([[[-1.0], [1.0 - 2 ** -23]]], np.float32)
    du = np.zeros((1, 2, 1), np.float32)
    got = run_oracle_step(x, dv, du, 0, 1)
    assert got[0, 0, 0] == np.float32(-(2.0 ** -46))


@pytest.mark.parametrize("vset", ["normal", "wide", "denormal", "big", "zeros_signed"])
def test_c_equals_one(vset):
    """C = 1: d_u + RN(x d), where a -0 product becomes +0 (fma from +0)."""
    w = synth.Workload("c1", 70, T=3, P=2, C=1, hd=37, x_scale="unit")
    inp = synth.make_inputs(w, seed=11, value_set=vset)
    x, dv, du = inp["x"], inp["d_dv"], inp["d_u"]
    got = run_oracle_step(x, dv, du, 2, 2)
    want = du.copy()
    with np.errstate(all="ignore"):
        prod = x[4:6, 0, 0][:, None] * dv[4:6, 0, :]          # float32 multiply: one rounding
        acc = prod + np.float32(0.0)                          # -0 + +0 = +0
        want[4:6, 0, :] = du[4:6, 0, :] + acc
    assert_bitwise(got, want)


def _finite_normal(shape, key):
    a = np.empty(shape, np.float32)
    synth.fill_normal(a, key)
    return a


@pytest.mark.parametrize("vset", ["normal", "denormal", "wide", "zeros_signed"])
def test_identity_x(vset):
    """x[n] = I: d_u + d_dv[n, i, c] with one rounding (d_dv = -0 contributes +0)."""
    w = synth.Workload("idx", 71, T=2, P=3, C=24, hd=19, x_scale="unit")
    inp = synth.make_inputs(w, seed=5, value_set=vset)
    dv, du = inp["d_dv"], inp["d_u"]
    x = np.broadcast_to(np.eye(24, dtype=np.float32), (6, 24, 24)).copy()
    got = run_oracle_step(x, dv, du, 1, 3)
    want = du.copy()
    with np.errstate(all="ignore"):
        want[3:6] = du[3:6] + (dv[3:6] + np.float32(0.0))
    assert_bitwise(got, want)


def test_permutation_x():
    """x[n, j, i] = [j == pi(i)]: d_u + d_dv[n, pi(i), c]. A transposed x would give pi^-1 instead."""
    C, hd, P = 32, 21, 2
    rng = np.random.default_rng(RNG_SEED + 1)
    pi = rng.permutation(C)
    while np.array_equal(pi[pi], np.arange(C)):       # not an involution, so pi != pi^-1
        pi = rng.permutation(C)
    x = np.zeros((2 * P, C, C), np.float32)
    for i in range(C):
        x[:, pi[i], i] = 1.0
    dv = _finite_normal((2 * P, C, hd), synth.stream_key(1, 2, 3))
    du = _finite_normal((2 * P, C, hd), synth.stream_key(1, 2, 4))
    got = run_oracle_step(x, dv, du, 0, P)
    want = du.copy()
    want[:P] = du[:P] + dv[:P][:, pi, :]
    assert_bitwise(got, want)


@pytest.mark.parametrize("vset", ["normal", "denormal", "zeros_signed", "denormal_all"])
def test_zero_x_keeps_d_u(vset):
    """x = 0 with finite d_dv: every product is a zero, acc = +0, and d_u comes back bit for bit except -0 -> +0.
    With subnormal d_u this is the subnormal-survival check (a flush to zero would lose them)."""
    w = synth.Workload("zx", 72, T=2, P=2, C=16, hd=33, x_scale="unit")
    inp = synth.make_inputs(w, seed=9, value_set=vset)
    dv, du = inp["d_dv"], inp["d_u"]
    x = np.zeros((4, 16, 16), np.float32)
    got = run_oracle_step(x, dv, du, 1, 2)
    want = du.copy()
    want[2:4] = np.where(du[2:4] == 0, np.float32(0.0), du[2:4])
    assert_bitwise(got, want)
    if vset.startswith("denormal"):
        sub = np.abs(du[2:4]) < np.finfo(np.float32).tiny
        assert np.count_nonzero(sub & (du[2:4] != 0)) > 0
        assert np.array_equal(bits(got[2:4])[sub & (du[2:4] != 0)], bits(du[2:4])[sub & (du[2:4] != 0)])


@pytest.mark.parametrize("vset", ["inf", "nan"])
def test_ieee_special_rules(vset):
    """With N(0,1) data (no finite overflow) and sprinkled Inf / NaN: NaN if any NaN input of the element, any 0*Inf
    product, or both signs of infinity among the Inf products and d_u; else that single-signed infinity; else finite."""
    C, hd, P = 48, 40, 2
    w = synth.Workload("sp", 73, T=1, P=P, C=C, hd=hd, x_scale="unit")
    inp = synth.make_inputs(w, seed=13, value_set=vset)
    x, dv, du = inp["x"], inp["d_dv"], inp["d_u"]
    got = run_oracle_step(x, dv, du, 0, P)
    n_nan = n_inf = 0
    for n in range(P):
        for i in range(C):
            a = x[n, :, i].astype(np.float64)
            for c in range(hd):
                b = dv[n, :, c].astype(np.float64)
                u = float(du[n, i, c])
                g = float(got[n, i, c])
                if np.isnan(a).any() or np.isnan(b).any() or math.isnan(u):
                    assert math.isnan(g)
                    n_nan += 1
                    continue
                inf_a, inf_b = np.isinf(a), np.isinf(b)
                if np.any((inf_a & (b == 0)) | (inf_b & (a == 0))):
                    assert math.isnan(g)
                    n_nan += 1
                    continue
                with np.errstate(all="ignore"):
                    signs = set(np.sign(a[inf_a | inf_b] * b[inf_a | inf_b]).tolist())
                if math.isinf(u):
                    signs.add(math.copysign(1.0, u))
                if len(signs) == 2:
                    assert math.isnan(g)
                    n_nan += 1
                elif len(signs) == 1:
                    assert math.isinf(g) and math.copysign(1.0, g) == signs.pop()
                    n_inf += 1
                else:
                    assert math.isfinite(g)
    assert n_nan > 0
    if vset == "inf":
        assert n_inf > 0


@pytest.mark.parametrize("vset", ["zeros", "zeros_signed", "normal", "wide", "denormal", "big", "inf"])
def test_no_negative_zero_output(vset):
    """acc starts at +0 and a -0 product plus +0 is +0, so no non-NaN output is -0; all-zero inputs give +0."""
    w = synth.Workload("nz", 74, T=2, P=2, C=16, hd=24, x_scale="unit")
    inp = synth.make_inputs(w, seed=17, value_set=vset)
    got = run_oracle_step(inp["x"], inp["d_dv"], inp["d_u"], 1, 2)[2:4]
    zero = (got == 0) & ~np.isnan(got)
    assert not np.any(np.signbit(got[zero]))
    if vset.startswith("zeros"):
        assert np.all(bits(got) == 0)


def test_step_touches_only_its_chunks():
    """Step ti writes chunks ti*P .. ti*P + P - 1 and nothing else; x and d_dv are not modified."""
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w)
    x0, dv0, du0 = (inp[k].copy() for k in ("x", "d_dv", "d_u"))
    for ti in range(w.T):
        du = du0.copy()
        oracle.step(du, inp["x"], inp["d_dv"], ti, w.P)
        mask = np.zeros(w.N, bool)
        mask[ti * w.P:(ti + 1) * w.P] = True
        assert np.array_equal(bits(du[~mask]), bits(du0[~mask]))
        assert np.count_nonzero(bits(du[mask]) != bits(du0[mask])) > 0
    assert np.array_equal(bits(inp["x"]), bits(x0)) and np.array_equal(bits(inp["d_dv"]), bits(dv0))


def test_strided_views_equal_contiguous():
    """Row strides (d_dv and d_u rows of hd + 1 floats, x rows of C + 3) give the same bits as contiguous arrays."""
    w = synth.WORKLOADS["edge"]
    C, hd, P = w.C, 128, w.P
    inp = synth.make_inputs(w, hd=hd, N=2 * P)
    x, dv, du = inp["x"], inp["d_dv"], inp["d_u"]
    xs = np.zeros((2 * P, C, C + 3), np.float32)[:, :, :C]
    xs[...] = x
    dvs = np.zeros((2 * P, C, hd + 1), np.float32)[:, :, :hd]
    dvs[...] = dv
    dus = np.zeros((2 * P, C, hd + 1), np.float32)[:, :, :hd]
    dus[...] = du
    want = run_oracle_step(x, dv, du, 1, P)
    oracle.step(dus, xs, dvs, 1, P)
    assert_bitwise(dus, want)


def test_points_match_step():
    w = synth.WORKLOADS["pdl_chain"]
    inp = synth.make_inputs(w, N=64)
    x, dv, du = inp["x"], inp["d_dv"], inp["d_u"]
    full = run_oracle_step(x, dv, du, 1, w.P)
    rng = np.random.default_rng(1)
    n = rng.integers(w.P, 2 * w.P, 200)
    i = rng.integers(0, w.C, 200)
    c = rng.integers(0, w.hd, 200)
    pts = oracle.points(du, x, dv, n, i, c)
    assert_bitwise(pts, full[n, i, c])


def test_steps_commute():
    """Steps touch disjoint chunks: any order of the T steps gives the same bits."""
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w)
    a = inp["d_u"].copy()
    b = inp["d_u"].copy()
    oracle.run_steps(a, inp["x"], inp["d_dv"], w.P)
    oracle.run_steps(b, inp["x"], inp["d_dv"], w.P, order=reversed(range(w.T)))
    assert_bitwise(a, b)


def test_producer_sign_flip():
    w = synth.WORKLOADS["producer_chain"]
    S = synth.make_source(w, N=4 * w.P)
    dv = np.zeros_like(S)
    for ti in range(4):
        oracle.producer_step(dv, S, ti, w.P)
    for ti in range(4):
        sl = slice(ti * w.P, (ti + 1) * w.P)
        want = -S[sl] if ti % 2 else S[sl]
        assert np.array_equal(bits(dv[sl]), bits(want))


def test_golden_tiny_matches_stored_bits():
    """The stored tiny-workload result (written by tests/golden/make_golden.py from the oracle) still matches, so an
    accidental change of the oracle's arithmetic shows up."""
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_seed0_after_4_steps.txt")
    lines = [ln for ln in open(path) if not ln.startswith("#")]
    stored = np.array([int(t, 16) for ln in lines for t in ln.split()], np.uint32)
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w)
    du = inp["d_u"].copy()
    oracle.run_steps(du, inp["x"], inp["d_dv"], w.P)
    assert np.array_equal(bits(du).reshape(-1), stored)


def test_successor_rows_pins():
    """The synthetic successor's reference: integer rows sum exactly; for a row of 33 floats the order is written out by
    hand: lane 0 holds d[0] + d[32], every other lane l one value, and lane 0's butterfly result is
    ((((p0 + p16) + (p8 + p24)) + ((p4 + p20) + (p12 + p28))) + ...) with each add rounded to float32."""
    rng = np.random.default_rng(3)
    d = rng.integers(-1000, 1000, (4, 3, 70)).astype(np.float32)
    got = oracle.successor_rows(d, 1, 2)
    assert np.array_equal(got.astype(np.int64), d[2:4, 0].astype(np.int64).sum(axis=1))
    f = (rng.standard_normal((1, 1, 33)) * np.exp2(rng.integers(-20, 20, (1, 1, 33)))).astype(np.float32)
    r = f[0, 0]
    add = lambda a, b: np.float32(float(a) + float(b))   # noqa: E731 (exact double sum of two floats, one rounding)
    p = [add(np.float32(0.0), r[k]) for k in range(32)]
    p[0] = add(p[0], r[32])

    def level(v, off):
        return [add(v[k], v[k ^ off]) for k in range(32)]
    v = p
    for off in (16, 8, 4, 2, 1):
        v = level(v, off)
    assert oracle.successor_rows(f, 0, 1)[0] == v[0]
