"""The C ABI without a GPU: the library loads, exports every symbol include/sdm_gx_gemm.h declares, and rejects bad
arguments with the documented status codes before making any CUDA call (fake pointers are never dereferenced)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdm_gx_gemm.h")

gx = pytest.importorskip("fp32_gemm_gb300")
L = gx.lib()
CODE = gx._binding.CODE


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^SDM_GX_API\s+[\w\s\*]*?\b(sdm_gx_\w+)\(", src, re.M)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(L, n), f"missing export {n}"
    assert set(names) == set(gx._binding.SIGNATURES), "binding signatures and header declarations differ"


def test_header_constants_match_binding():
    """Every flag and error-word bit the header defines has the same value in the Python binding."""
    src = open(HEADER).read()
    defs = re.findall(r"#define SDM_GX_((?:FLAG|ERR)_\w+)\s+(0x[0-9A-Fa-f]+|\d+)u?\b", src)
    assert len(defs) >= 10
    for name, value in defs:
        assert getattr(gx._binding, name) == int(value, 0), name


def test_version_and_strerror():
    assert gx.abi_version() == 1
    for code, name in gx._binding.STATUS.items():
        s = gx.strerror(code)
        assert isinstance(s, str) and s and s != "unknown status", name
    assert gx.strerror(12345) == "unknown status"


# Fake, 16-byte aligned, non-overlapping "device" addresses: argument checks must fail before any use of them.
U, X, V = 0x10000000, 0x20000000, 0x30000000


def step(du=U, x=X, dv=V, ti=0, P=2, C=16, hd=32):
    return L.sdm_gx_gemm_step(du, x, dv, ti, P, C, hd, None, 0)


def step_ex(du=U, x=X, dv=V, ti=0, N=8, P=2, C=16, hd=32, strides=None, flags=0):
    sp = ctypes.byref(strides) if strides is not None else None
    return L.sdm_gx_gemm_step_ex(du, x, dv, ti, N, P, C, hd, sp, None, 0, flags)


@pytest.mark.parametrize("kw,code", [
    (dict(du=0), "SDM_GX_E_NULL"), (dict(x=0), "SDM_GX_E_NULL"), (dict(dv=0), "SDM_GX_E_NULL"),
    (dict(C=0), "SDM_GX_E_SHAPE"), (dict(C=257), "SDM_GX_E_SHAPE"), (dict(hd=0), "SDM_GX_E_SHAPE"),
    (dict(hd=1 << 20), "SDM_GX_E_SHAPE"), (dict(P=0), "SDM_GX_E_RANGE"), (dict(ti=-1), "SDM_GX_E_RANGE"),
    (dict(P=1 << 31), "SDM_GX_E_RANGE"), (dict(ti=(1 << 30), P=2), "SDM_GX_E_RANGE"),
    (dict(du=U + 2), "SDM_GX_E_ALIGN"), (dict(x=X + 1), "SDM_GX_E_ALIGN"), (dict(dv=V + 3), "SDM_GX_E_ALIGN"),
    (dict(x=U + 64), "SDM_GX_E_OVERLAP"), (dict(dv=U - 4), "SDM_GX_E_OVERLAP"),
])
def test_step_argument_errors(kw, code):
    assert step(**kw) == CODE[code]


def test_step_overlap_is_per_step_span():
    """sdm_gx_gemm_step checks the spans of the chunks the step touches: for ti = 1, P = 2 those are chunks 2..3."""
    cu, cx = 16 * 32 * 4, 16 * 16 * 4            # bytes per d_u / x chunk
    assert step(ti=1, dv=U) == CODE["SDM_GX_E_OVERLAP"]
    assert step(ti=1, x=U + 4 * cu - 2 * cx - 4) == CODE["SDM_GX_E_OVERLAP"]
    # x's step span starting exactly where d_u's ends passes the argument checks (then fails later: no GPU here)
    assert step(ti=1, x=U + 4 * cu - 2 * cx) not in (CODE["SDM_GX_E_OVERLAP"], 0)


@pytest.mark.parametrize("kw,code", [
    (dict(N=0), "SDM_GX_E_RANGE"), (dict(N=1 << 31), "SDM_GX_E_RANGE"), (dict(P=9), "SDM_GX_E_RANGE"),
    (dict(ti=4), "SDM_GX_E_RANGE"), (dict(ti=3, N=7), "SDM_GX_E_RANGE"), (dict(ti=-1), "SDM_GX_E_RANGE"),
    (dict(dv=U + 8 * 16 * 32 * 4 - 4), "SDM_GX_E_OVERLAP"), (dict(x=U + 100), "SDM_GX_E_OVERLAP"),
])
def test_step_ex_argument_errors(kw, code):
    assert step_ex(**kw) == CODE[code]


@pytest.mark.parametrize("field,value", [
    ("x_sj", 15), ("x_sn", 16 * 16 - 1), ("dv_sj", 31), ("dv_sn", 16 * 32 - 1), ("du_si", 31), ("du_sn", 100),
    ("du_si", 1 << 41),
])
def test_stride_errors(field, value):
    s = gx.Strides(16 * 16, 16, 16 * 32, 32, 16 * 32, 32)
    setattr(s, field, value)
    assert step_ex(strides=s) == CODE["SDM_GX_E_STRIDE"]


def test_plan_errors_without_gpu():
    h = ctypes.c_void_p()
    assert L.sdm_gx_gemm_plan_create(ctypes.byref(h), U, X, V, 8, 2, 0, 32, None, 3, 0) == CODE["SDM_GX_E_SHAPE"]
    assert L.sdm_gx_gemm_plan_create(ctypes.byref(h), U, X, V, 8, 2, 16, 32, None, 4, 0) == CODE["SDM_GX_E_RANGE"]
    assert L.sdm_gx_gemm_plan_create(None, U, X, V, 8, 2, 16, 32, None, 3, 0) == CODE["SDM_GX_E_NULL"]
    assert h.value is None
    assert L.sdm_gx_gemm_plan_step(None, 0, None, 0) == CODE["SDM_GX_E_PLAN"]
    assert L.sdm_gx_gemm_plan_run(None, 0, 4, None, 1) == CODE["SDM_GX_E_PLAN"]
    assert L.sdm_gx_gemm_plan_run_producer(None, V, 0, 4, None, 1) == CODE["SDM_GX_E_PLAN"]
    g = gx.Geom()
    assert L.sdm_gx_gemm_plan_geometry(None, ctypes.byref(g)) == CODE["SDM_GX_E_PLAN"]
    # a corrupt plan: arbitrary bytes are not a plan
    junk = ctypes.create_string_buffer(b"\x47" * 4096)
    assert L.sdm_gx_gemm_plan_step(ctypes.cast(junk, ctypes.c_void_p), 0, None, 0) == CODE["SDM_GX_E_PLAN"]
    L.sdm_gx_gemm_plan_destroy(None)
    L.sdm_gx_gemm_plan_destroy(ctypes.cast(junk, ctypes.c_void_p))   # not a plan: ignored


def test_autotune_argument_errors():
    f = L.sdm_gx_gemm_autotune
    fo, co, us = ctypes.c_uint(7), ctypes.c_int32(-1), ctypes.c_float(0.0)

    def call(flags_out=ctypes.byref(fo), steps=8, flags=0, N=8, P=2, C=16, hd=32, du=U):
        return f(du, X, V, N, P, C, hd, None, flags, None, 0, steps, None, flags_out, ctypes.byref(co),
                 ctypes.byref(us))

    assert call(flags_out=None) == CODE["SDM_GX_E_NULL"]
    assert call(steps=0) == CODE["SDM_GX_E_RANGE"]
    assert call(steps=4097) == CODE["SDM_GX_E_RANGE"]
    assert call(flags=gx.config_flag(3)) == CODE["SDM_GX_E_FLAGS"]       # a forced configuration is the output
    assert call(flags=gx._binding.FLAG_TEST_STALL) == CODE["SDM_GX_E_FLAGS"]
    assert call(P=0) == CODE["SDM_GX_E_RANGE"]
    assert call(N=1) == CODE["SDM_GX_E_RANGE"]
    assert call(C=0) == CODE["SDM_GX_E_SHAPE"]                            # the plan's own checks
    assert call(du=0) == CODE["SDM_GX_E_NULL"]
    assert fo.value == 7 and co.value == -1                                  # outputs untouched on error


def test_producer_argument_errors():
    f = L.sdm_gx_producer_step
    assert f(0, V, 0, 2, 16, 32, None, 0) == CODE["SDM_GX_E_NULL"]
    assert f(U, V, 0, 2, 0, 32, None, 0) == CODE["SDM_GX_E_SHAPE"]
    assert f(U, V, -1, 2, 16, 32, None, 0) == CODE["SDM_GX_E_RANGE"]
    assert f(U + 1, V, 0, 2, 16, 32, None, 0) == CODE["SDM_GX_E_ALIGN"]
    assert f(U, U + 64, 0, 2, 16, 32, None, 0) == CODE["SDM_GX_E_OVERLAP"]


def test_unknown_flags_rejected_before_cuda():
    # unknown flag bits are checked in build_launch after validation; on a machine without a GPU the call must
    # still end in an error status, never a crash
    rc = step_ex(flags=0x80000)
    assert rc < 0


def test_missing_library_fails_loudly(monkeypatch):
    import fp32_gemm_gb300._binding as b
    missing = os.path.join(ROOT, "fp32_gemm_gb300", "lib", "no_such_library.so")
    assert not os.path.exists(missing)
    monkeypatch.setattr(b, "LIB_PATH", missing)
    with pytest.raises(ImportError):
        b._load()


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++17")])
def test_header_compiles_as_c_and_cpp(lang, std):
    """include/sdm_gx_gemm.h is a C ABI: it must compile as strict C99 and as C++ (syntax only; nothing is written)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("no host compiler or CUDA headers")
    r = subprocess.run([cc, "-x", lang, std, "-Wall", "-Wextra", "-pedantic", "-fsyntax-only", "-I", cuda_inc, HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_binding_has_no_cpu_fallback():
    import fp32_gemm_gb300._binding as b
    src = open(b.__file__).read()
    assert "oracle" not in src and "numpy" not in src


def test_set_trace_rejects_a_bad_plan():
    n = ctypes.c_int32(-1)
    assert L.sdm_gx_gemm_plan_set_trace(None, None, 0, ctypes.byref(n)) == CODE["SDM_GX_E_PLAN"]
    fake = (ctypes.c_uint64 * 64)()   # host memory that is not a plan (bad magic)
    assert L.sdm_gx_gemm_plan_set_trace(ctypes.addressof(fake), None, 0, None) == CODE["SDM_GX_E_PLAN"]
    assert n.value == -1
