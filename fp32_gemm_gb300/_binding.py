"""ctypes binding of the gx_gemm C ABI (include/sdm_gx_gemm.h). Argument marshalling only: torch tensors are turned
into device pointers, element strides and the current CUDA stream; every step of the update runs in the library's
kernels. There is no CPU fallback: if the library is not built, importing this module raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# SDM_GX_TRACE_BUILD=1: the timeline build of the same library (build(trace=True); sdm_gx_gemm_plan_set_trace works
# there only)
LIB_PATH = os.path.join(HERE, "lib", "libsdm_gx_gemm_trace.so" if os.environ.get("SDM_GX_TRACE_BUILD") == "1"
                        else "libsdm_gx_gemm.so")

FLAG_GENERIC = 0x100
FLAG_NO_PREFETCH = 0x200
FLAG_TEST_STALL = 0x400
FLAG_TEST_NO_HANDOFF = 0x20000
FLAG_NOALLOC = 0x800   # geometry(): the launch sdm_gx_gemm_step_noalloc would make
FLAG_X_TRANSPOSED = 0x10000   # x stored [n][i][j] (passed here as a transpose(1, 2) view; set automatically)
FLAG_CONFIG_MASK = 0x0FF
FLAG_CTAS_SHIFT = 12
FLAG_CTAS_MASK = 0xF000

# bits of the device error word (sdm_gx_device_error)
ERR_FATAL_MASK = 0x7              # bits 0-2: a kernel gave up a bounded wait, its step is incomplete
ERR_HANDOFF_RECOMPUTED = 0x8      # bit 3, informational: a tile's chain recomputed after a late hand-off (exact)

STATUS = {
    0: "SDM_GX_OK", -1: "SDM_GX_E_NULL", -2: "SDM_GX_E_SHAPE", -3: "SDM_GX_E_RANGE", -4: "SDM_GX_E_ALIGN",
    -5: "SDM_GX_E_OVERLAP", -6: "SDM_GX_E_STRIDE", -7: "SDM_GX_E_GRID", -8: "SDM_GX_E_SMEM", -9: "SDM_GX_E_DEVICE",
    -10: "SDM_GX_E_PLAN", -11: "SDM_GX_E_PLAN_TI", -12: "SDM_GX_E_PLAN_DEVICE", -13: "SDM_GX_E_FLAGS",
    -14: "SDM_GX_E_CUDA", -15: "SDM_GX_E_DEVICE_FAULT", -16: "SDM_GX_E_UNSUPPORTED", -17: "SDM_GX_E_ALLOC",
    -18: "SDM_GX_E_CAPTURE",
}
CODE = {v: k for k, v in STATUS.items()}


class Strides(ctypes.Structure):
    _fields_ = [("x_sn", ctypes.c_int64), ("x_sj", ctypes.c_int64), ("dv_sn", ctypes.c_int64),
                ("dv_sj", ctypes.c_int64), ("du_sn", ctypes.c_int64), ("du_si", ctypes.c_int64)]


class Geom(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("config", ctypes.c_int32), ("TI", ctypes.c_int32),
                ("TC", ctypes.c_int32), ("KB", ctypes.c_int32), ("stages", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("smem_bytes", ctypes.c_int32), ("tiles", ctypes.c_int64),
                ("ctas", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32), ("sms", ctypes.c_int32),
                ("one_wave", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {k: int(getattr(self, k)) for k, _ in self._fields_}


class GxGemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.name = STATUS.get(self.status, str(status))
        msg = f"{where}: {self.name} ({_lib.sdm_gx_strerror(status).decode()})"
        if self.status == CODE["SDM_GX_E_CUDA"]:
            msg += f" [cudaError {_lib.sdm_gx_last_cuda_error()}]"
        super().__init__(msg)


SIGNATURES = {
    # name: (restype, argtypes)
    "sdm_gx_gemm_step": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 4 + [ctypes.c_void_p, ctypes.c_int]),
    "sdm_gx_gemm_step_noalloc": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 4 +
                                 [ctypes.c_void_p, ctypes.c_int]),
    "sdm_gx_gemm_step_ex": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 5 +
                            [ctypes.POINTER(Strides), ctypes.c_void_p, ctypes.c_int, ctypes.c_uint]),
    "sdm_gx_gemm_geometry": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 4 +
                             [ctypes.POINTER(Strides), ctypes.c_uint, ctypes.POINTER(Geom)]),
    "sdm_gx_gemm_plan_create": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p)] + [ctypes.c_void_p] * 3 +
                                [ctypes.c_int64] * 4 + [ctypes.POINTER(Strides), ctypes.c_int64, ctypes.c_uint]),
    "sdm_gx_gemm_plan_create_ws": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p)] + [ctypes.c_void_p] * 3 +
                                   [ctypes.c_int64] * 4 + [ctypes.POINTER(Strides), ctypes.c_int64, ctypes.c_uint,
                                                           ctypes.c_void_p, ctypes.c_size_t]),
    "sdm_gx_gemm_plan_workspace_size": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 4 +
                                        [ctypes.POINTER(Strides), ctypes.c_uint, ctypes.POINTER(ctypes.c_size_t)]),
    "sdm_gx_gemm_autotune": (ctypes.c_int, [ctypes.c_void_p] * 3 + [ctypes.c_int64] * 4 +
                             [ctypes.POINTER(Strides), ctypes.c_uint, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int,
                              ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_int32),
                              ctypes.POINTER(ctypes.c_float)]),
    "sdm_gx_gemm_plan_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]),
    "sdm_gx_gemm_plan_run": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                            ctypes.c_int]),
    "sdm_gx_gemm_plan_run_producer": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                     ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]),
    "sdm_gx_gemm_plan_geometry": (ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(Geom)]),
    "sdm_gx_gemm_plan_set_trace": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                  ctypes.POINTER(ctypes.c_int32)]),
    "sdm_gx_gemm_plan_graph_create": (ctypes.c_int, [ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]),
    "sdm_gx_gemm_plan_run_successor": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                                      ctypes.c_int64, ctypes.c_void_p, ctypes.c_int]),
    "sdm_gx_gemm_plan_run_host": (ctypes.c_int, [ctypes.c_void_p] * 4 + [ctypes.c_int64] * 2 + [ctypes.c_void_p] * 3),
    "sdm_gx_graph_launch": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "sdm_gx_graph_destroy": (None, [ctypes.c_void_p]),
    "sdm_gx_gemm_plan_destroy": (None, [ctypes.c_void_p]),
    "sdm_gx_producer_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int64] * 4 +
                             [ctypes.c_void_p, ctypes.c_int]),
    "sdm_gx_gemm_kernel_attrs": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64)]),
    "sdm_gx_gemm_num_configs": (ctypes.c_int, [ctypes.c_int32]),
    "sdm_gx_gemm_choose_config": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32),
                                                 ctypes.c_int32, ctypes.c_int32] + [ctypes.c_int64] * 3 +
                                  [ctypes.c_size_t]),
    "sdm_gx_gemm_config_info": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "sdm_gx_gemm_stream_piece": (ctypes.c_int, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]),
    "sdm_gx_device_error": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
    "sdm_gx_launch_counts": (None, [ctypes.POINTER(ctypes.c_int64)]),
    "sdm_gx_last_cuda_error": (ctypes.c_int, []),
    "sdm_gx_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "sdm_gx_abi_version": (ctypes.c_int, []),
}


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"gx_gemm CUDA library not built ({LIB_PATH} missing): run fp32_gemm_gb300.build.build() "
                          "or __graft_entry__.build(); there is no CPU fallback")
    L = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


_lib = _load()


def lib():
    return _lib


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise GxGemmError(rc, where)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


def _as3(t: torch.Tensor, rows: int, cols: int, N: int) -> torch.Tensor:
    """A [N, rows, cols] view of a float32 CUDA tensor with unit innermost stride (no copy)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32:
        raise TypeError("gx_gemm: operands are float32 CUDA tensors")
    if t.is_neg() or t.is_conj():
        raise TypeError("gx_gemm: lazy negative / conjugate views are not supported (materialise them first)")
    if t.dim() == 3:
        v = t
    elif t.dim() == 2 and t.shape[0] == N * rows:
        v = t.view(N, rows, cols) if t.is_contiguous() else t.unflatten(0, (N, rows))
    else:
        raise ValueError(f"gx_gemm: expected [N, {rows}, {cols}] (or [N*{rows}, {cols}]), got {tuple(t.shape)}")
    if tuple(v.shape) != (N, rows, cols):
        raise ValueError(f"gx_gemm: expected shape {(N, rows, cols)}, got {tuple(v.shape)}")
    if v.stride(2) != 1:
        raise ValueError("gx_gemm: the innermost stride must be 1")
    return v


def _operands(d_u, x, d_dv):
    """Views, sizes and strides of the three operands. x is the logical [N, C, C] tensor x[n, j, i]; a view with unit
    stride along j instead of i (e.g. stored.transpose(1, 2) of a [N, C(i), C(j)] tensor) is passed as stored
    transposed (SDM_GX_FLAG_X_TRANSPOSED, returned in the last element as the flag to add)."""
    if x.dim() != 3:
        raise ValueError("gx_gemm: x is [N, C, C]")
    N, C = int(x.shape[0]), int(x.shape[1])
    hd = int(d_u.shape[-1])
    xflag = 0
    if C > 1 and x.stride(2) != 1 and x.stride(1) == 1:
        if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32:
            raise TypeError("gx_gemm: operands are float32 CUDA tensors")
        xv = x
        xs = (x.stride(0), x.stride(2))   # chunk stride, stride between the stored rows i
        xflag = FLAG_X_TRANSPOSED
    else:
        xv = _as3(x, C, C, N)
        xs = (xv.stride(0), xv.stride(1))
    uv = _as3(d_u, C, hd, N)
    vv = _as3(d_dv, C, hd, N)
    s = Strides(xs[0], xs[1], vv.stride(0), vv.stride(1), uv.stride(0), uv.stride(1))
    return uv, xv, vv, N, C, hd, s, xflag


def step(d_u, x, d_dv, ti: int, P: int, pdl: bool = False, stream=None) -> None:
    """sdm_gx_gemm_step: one step on contiguous operands (d_u updated in place)."""
    if not (d_u.is_contiguous() and x.is_contiguous() and d_dv.is_contiguous()):
        raise ValueError("gx_gemm.step: contiguous operands (use step_ex for strided views)")
    C = int(x.shape[1])
    hd = int(d_u.shape[-1])
    _check(_lib.sdm_gx_gemm_step(d_u.data_ptr(), x.data_ptr(), d_dv.data_ptr(), int(ti), int(P), C, hd,
                                 _stream(stream), int(bool(pdl))), "sdm_gx_gemm_step")


def step_noalloc(d_u, x, d_dv, ti: int, P: int, pdl: bool = False, stream=None) -> None:
    """sdm_gx_gemm_step_noalloc: one step like step(), with the library's static scratch as the stream kernel's
    workspace (allocates nothing; calls on one device must not overlap in time)."""
    if not (d_u.is_contiguous() and x.is_contiguous() and d_dv.is_contiguous()):
        raise ValueError("gx_gemm.step_noalloc: contiguous operands")
    C = int(x.shape[1])
    hd = int(d_u.shape[-1])
    _check(_lib.sdm_gx_gemm_step_noalloc(d_u.data_ptr(), x.data_ptr(), d_dv.data_ptr(), int(ti), int(P), C, hd,
                                         _stream(stream), int(bool(pdl))), "sdm_gx_gemm_step_noalloc")


def step_ex(d_u, x, d_dv, ti: int, P: int, pdl: bool = False, flags: int = 0, stream=None) -> None:
    """sdm_gx_gemm_step_ex: one step on strided [N, ...] operands."""
    uv, xv, vv, N, C, hd, s, xflag = _operands(d_u, x, d_dv)
    _check(_lib.sdm_gx_gemm_step_ex(uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), int(ti), N, int(P), C, hd,
                                    ctypes.byref(s), _stream(stream), int(bool(pdl)), int(flags) | xflag),
           "sdm_gx_gemm_step_ex")


def geometry(d_u, x, d_dv, P: int, flags: int = 0) -> dict:
    uv, xv, vv, N, C, hd, s, xflag = _operands(d_u, x, d_dv)
    g = Geom()
    _check(_lib.sdm_gx_gemm_geometry(uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), N, int(P), C, hd,
                                     ctypes.byref(s), int(flags) | xflag, ctypes.byref(g)), "sdm_gx_gemm_geometry")
    return g.as_dict()


def noalloc_geometry(d_u, x, d_dv, P: int) -> dict:
    """sdm_gx_gemm_geometry with SDM_GX_FLAG_NOALLOC: the geometry sdm_gx_gemm_step_noalloc uses for a step of this
    shape (contiguous operands)."""
    return geometry(d_u, x, d_dv, P, flags=FLAG_NOALLOC)


def workspace_size(d_u, x, d_dv, P: int, flags: int = 0) -> int:
    """sdm_gx_gemm_plan_workspace_size: bytes of plan workspace that let this shape use the stream kernel (0: none)."""
    uv, xv, vv, N, C, hd, s, xflag = _operands(d_u, x, d_dv)
    n = ctypes.c_size_t(0)
    _check(_lib.sdm_gx_gemm_plan_workspace_size(uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), N, int(P), C, hd,
                                                ctypes.byref(s), int(flags) | xflag, ctypes.byref(n)),
           "sdm_gx_gemm_plan_workspace_size")
    return int(n.value)


def autotune(d_u_scratch, x, d_dv, P: int, steps: int = 20, flags: int = 0, workspace: bool = True,
             stream=None) -> dict:
    """sdm_gx_gemm_autotune: time every configuration that this shape and layout admit, on these buffers, and return
    {"flags", "config", "us"} of the fastest; Plan(d_u, x, d_dv, P, flags=result["flags"]) then uses it. d_u_scratch
    is updated by the timed steps: pass a copy of d_u (same shape and strides), never d_u itself. workspace=True lets
    the stream configurations take part (a temporary allocation of the size a Plan's workspace has; the Plan must then
    have its workspace too, the default)."""
    uv, xv, vv, N, C, hd, s, xflag = _operands(d_u_scratch, x, d_dv)
    nws = workspace_size(d_u_scratch, x, d_dv, P, flags) if workspace else 0
    ws = torch.empty(nws, dtype=torch.uint8, device=uv.device) if nws > 0 else None
    fo, co, us = ctypes.c_uint(0), ctypes.c_int32(-1), ctypes.c_float(0.0)
    _check(_lib.sdm_gx_gemm_autotune(uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), N, int(P), C, hd, ctypes.byref(s),
                                     int(flags) | xflag, ws.data_ptr() if ws is not None else None, nws, int(steps),
                                     _stream(stream), ctypes.byref(fo), ctypes.byref(co), ctypes.byref(us)),
           "sdm_gx_gemm_autotune")
    return {"flags": int(fo.value), "config": int(co.value), "us": float(us.value)}


class Plan:
    """sdm_gx_gemm_plan_*: validated once, launched per step with only ti changing. Keeps references to the tensors
    so that their memory outlives the plan. workspace=True (default) gives the plan the device workspace
    sdm_gx_gemm_plan_workspace_size asks for (a torch allocation held by the plan), so it may use the stream kernel;
    workspace=False creates it without one (sdm_gx_gemm_plan_create)."""

    def __init__(self, d_u, x, d_dv, P: int, ti_max: int | None = None, flags: int = 0, workspace: bool = True):
        uv, xv, vv, N, C, hd, s, xflag = _operands(d_u, x, d_dv)
        self._keep = (d_u, x, d_dv)
        self.N, self.P, self.C, self.hd = N, int(P), C, hd
        self.T = N // int(P) if P >= 1 else 0
        self.ti_max = self.T - 1 if ti_max is None else int(ti_max)
        h = ctypes.c_void_p()
        nws = workspace_size(d_u, x, d_dv, P, flags) if workspace else 0
        if nws > 0:
            self._ws = torch.empty(nws, dtype=torch.uint8, device=uv.device)
            _check(_lib.sdm_gx_gemm_plan_create_ws(ctypes.byref(h), uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), N,
                                                   int(P), C, hd, ctypes.byref(s), self.ti_max, int(flags) | xflag,
                                                   self._ws.data_ptr(), nws), "sdm_gx_gemm_plan_create_ws")
        else:
            self._ws = None
            _check(_lib.sdm_gx_gemm_plan_create(ctypes.byref(h), uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), N,
                                                int(P), C, hd, ctypes.byref(s), self.ti_max, int(flags) | xflag),
                   "sdm_gx_gemm_plan_create")
        self._h = h

    @property
    def workspace_bytes(self) -> int:
        return 0 if self._ws is None else int(self._ws.numel())

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def step(self, ti: int, pdl: bool = False, stream=None) -> None:
        _check(_lib.sdm_gx_gemm_plan_step(self._h, int(ti), _stream(stream), int(bool(pdl))),
               "sdm_gx_gemm_plan_step")

    def run(self, ti_begin: int = 0, ti_end: int | None = None, pdl: bool = True, stream=None) -> None:
        """Steps ti_begin, ti_begin +- 1, ... stopping before ti_end (default: all steps ascending)."""
        ti_end = self.T if ti_end is None else int(ti_end)
        _check(_lib.sdm_gx_gemm_plan_run(self._h, int(ti_begin), ti_end, _stream(stream), int(bool(pdl))),
               "sdm_gx_gemm_plan_run")

    def run_producer(self, S, ti_begin: int = 0, ti_end: int | None = None, pdl: bool = True, stream=None) -> None:
        """The chain with the synthetic producer before every step (d_dv(ti) = +-S(ti))."""
        if not (S.is_cuda and S.dtype == torch.float32 and S.is_contiguous() and S.numel() == self.N * self.C * self.hd):
            raise ValueError("run_producer: S is a contiguous float32 CUDA tensor shaped like d_dv")
        ti_end = self.T if ti_end is None else int(ti_end)
        self._keep_s = S
        _check(_lib.sdm_gx_gemm_plan_run_producer(self._h, S.data_ptr(), int(ti_begin), ti_end, _stream(stream),
                                                  int(bool(pdl))), "sdm_gx_gemm_plan_run_producer")

    def set_trace(self, buf, launches: int) -> int:
        """sdm_gx_gemm_plan_set_trace: record a timeline of the launches of steps ti < launches into buf (an int64 CUDA
        tensor of launches * ctas * 4 entries; None turns it off). Returns the CTAs per launch."""
        n = ctypes.c_int32(0)
        if buf is not None:
            if not (buf.is_cuda and buf.dtype == torch.int64 and buf.is_contiguous()):
                raise ValueError("set_trace: a contiguous int64 CUDA tensor")
            self._trace = buf
        _check(_lib.sdm_gx_gemm_plan_set_trace(self._h, buf.data_ptr() if buf is not None else None,
                                               int(launches) if buf is not None else 0, ctypes.byref(n)),
               "sdm_gx_gemm_plan_set_trace")
        return int(n.value)

    def geometry(self) -> dict:
        g = Geom()
        _check(_lib.sdm_gx_gemm_plan_geometry(self._h, ctypes.byref(g)), "sdm_gx_gemm_plan_geometry")
        return g.as_dict()

    def run_host(self, d_u_host, x_host, d_dv_host, ti_begin: int = 0, ti_end: int | None = None,
                 compute=None, h2d=None, d2h=None) -> None:
        """sdm_gx_gemm_plan_run_host: the chain fed from host tensors (pinned for overlap), copies overlapped with
        compute; d_u_host is updated when `d2h` (default: the plan's own copy-out stream) has finished."""
        for t, shape in ((x_host, (self.N, self.C, self.C)), (d_dv_host, (self.N, self.C, self.hd)),
                         (d_u_host, (self.N, self.C, self.hd))):
            if t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != shape:
                raise ValueError(f"run_host: contiguous float32 host tensors of shape {shape}")
        if not hasattr(self, "_streams"):
            self._streams = (torch.cuda.Stream(), torch.cuda.Stream())
        compute = torch.cuda.current_stream() if compute is None else compute
        h2d = self._streams[0] if h2d is None else h2d
        d2h = self._streams[1] if d2h is None else d2h
        ti_end = self.T if ti_end is None else int(ti_end)
        _check(_lib.sdm_gx_gemm_plan_run_host(self._h, d_u_host.data_ptr(), x_host.data_ptr(), d_dv_host.data_ptr(),
                                              int(ti_begin), ti_end, _stream(compute), _stream(h2d), _stream(d2h)),
               "sdm_gx_gemm_plan_run_host")
        return d2h

    def graph(self, ti_begin: int = 0, ti_end: int | None = None, pdl: bool = True, S=None,
              succ_out=None) -> "Graph":
        """sdm_gx_gemm_plan_graph_create: the chain captured once into a CUDA graph (with the producer if S given, or
        the synthetic successor if succ_out given)."""
        ti_end = self.T if ti_end is None else int(ti_end)
        if S is not None and not (S.is_cuda and S.dtype == torch.float32 and S.is_contiguous()
                                  and S.numel() == self.N * self.C * self.hd):
            raise ValueError("graph: S is a contiguous float32 CUDA tensor shaped like d_dv")
        if succ_out is not None:
            self._check_succ(succ_out)
        h = ctypes.c_void_p()
        _check(_lib.sdm_gx_gemm_plan_graph_create(ctypes.byref(h), self._h, S.data_ptr() if S is not None else None,
                                                  succ_out.data_ptr() if succ_out is not None else None,
                                                  int(ti_begin), ti_end, int(bool(pdl))),
               "sdm_gx_gemm_plan_graph_create")
        return Graph(h, (self, S, succ_out))

    def _check_succ(self, out) -> None:
        if not (out.is_cuda and out.dtype == torch.float32 and out.is_contiguous() and out.numel() == self.N):
            raise ValueError("successor: out is a contiguous float32 CUDA tensor of N elements")

    def run_successor(self, out, ti_begin: int = 0, ti_end: int | None = None, pdl: bool = True,
                      stream=None) -> None:
        """The chain with the synthetic successor (a consumer of d_u(ti): each chunk's leading-row sum into out[n])
        after every step."""
        self._check_succ(out)
        ti_end = self.T if ti_end is None else int(ti_end)
        self._keep_o = out
        _check(_lib.sdm_gx_gemm_plan_run_successor(self._h, out.data_ptr(), int(ti_begin), ti_end, _stream(stream),
                                                   int(bool(pdl))), "sdm_gx_gemm_plan_run_successor")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.sdm_gx_gemm_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001
            pass


class Graph:
    """An instantiated CUDA graph of a step chain (sdm_gx_graph_*). Keeps the plan and S alive."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep

    def launch(self, stream=None) -> None:
        _check(_lib.sdm_gx_graph_launch(self._h, _stream(stream)), "sdm_gx_graph_launch")

    def close(self) -> None:
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib.sdm_gx_graph_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001
            pass


def producer_step(d_dv, S, ti: int, P: int, pdl: bool = False, stream=None) -> None:
    """sdm_gx_producer_step: d_dv(ti) = S(ti), negated for odd ti (contiguous [N, C, hd])."""
    if not (d_dv.is_contiguous() and S.is_contiguous() and d_dv.shape == S.shape):
        raise ValueError("producer_step: contiguous d_dv and S of one shape")
    C, hd = int(d_dv.shape[-2]), int(d_dv.shape[-1])
    _check(_lib.sdm_gx_producer_step(d_dv.data_ptr(), S.data_ptr(), int(ti), int(P), C, hd, _stream(stream),
                                     int(bool(pdl))), "sdm_gx_producer_step")


def kernel_attrs(path: int, config: int) -> dict:
    out = (ctypes.c_int64 * 4)()
    _check(_lib.sdm_gx_gemm_kernel_attrs(int(path), int(config), out), "sdm_gx_gemm_kernel_attrs")
    return {"regs": out[0], "local_bytes": out[1], "static_smem": out[2], "max_threads": out[3]}


CONFIG_KINDS = {0: "tile", 1: "slab", 2: "stream", 3: "offset", 4: "offset_shifted"}


def config_info(path: int, config: int) -> dict:
    """sdm_gx_gemm_config_info: the static description of a configuration (kind: tile / slab / stream / offset /
    offset_shifted)."""
    out = (ctypes.c_int32 * 8)()
    _check(_lib.sdm_gx_gemm_config_info(int(path), int(config), out), "sdm_gx_gemm_config_info")
    return {"TI": out[0], "TC": out[1], "KB": out[2], "stages": out[3], "threads": out[4], "smem": out[5],
            "kind": CONFIG_KINDS.get(out[6], str(out[6])), "consumer_warps": out[7]}


def choose_config(path: int, sms: int, occ, P: int, C: int, hd: int, ws_bytes: int = 0, slab_ok: bool = True) -> int:
    """sdm_gx_gemm_choose_config: the configuration a plan would choose on a described device (SM count, resident
    CTAs per SM of every configuration of the path, workspace bytes); no GPU needed."""
    arr = (ctypes.c_int32 * len(occ))(*[int(v) for v in occ])
    k = _lib.sdm_gx_gemm_choose_config(int(path), int(sms), arr, len(occ), int(bool(slab_ok)), int(P), int(C), int(hd),
                                       int(ws_bytes))
    if k < 0:
        raise GxGemmError(k, "sdm_gx_gemm_choose_config")
    return int(k)


def stream_pieces(ntiles: int, C: int, G: int, b: int) -> list[tuple[int, int, int, int]]:
    """sdm_gx_gemm_stream_piece: the pieces (tile, j0, j1, kind) CTA b of G runs, in order, under the stream
    kernel's split of a step of ntiles tiles (host code shared with the kernel; no GPU needed)."""
    out = (ctypes.c_int32 * 4)()
    n = _lib.sdm_gx_gemm_stream_piece(int(ntiles), int(C), int(G), int(b), -1, out)
    if n < 0:
        raise GxGemmError(n, "sdm_gx_gemm_stream_piece")
    res = []
    for q in range(n):
        _check(_lib.sdm_gx_gemm_stream_piece(int(ntiles), int(C), int(G), int(b), q, out), "sdm_gx_gemm_stream_piece")
        res.append((out[0], out[1], out[2], out[3]))
    return res


def num_configs(path: int) -> int:
    return int(_lib.sdm_gx_gemm_num_configs(int(path)))


def device_error(clear: bool = True) -> int:
    """The device error word (synchronizes the device); 0 means no kernel gave up a bounded wait."""
    w = ctypes.c_uint32(0)
    rc = _lib.sdm_gx_device_error(ctypes.byref(w), int(bool(clear)))
    if rc not in (0, CODE["SDM_GX_E_DEVICE_FAULT"]):
        raise GxGemmError(rc, "sdm_gx_device_error")
    return int(w.value)


def launch_counts() -> dict:
    out = (ctypes.c_int64 * 4)()
    _lib.sdm_gx_launch_counts(out)
    return {"step": out[0], "producer": out[1], "pdl": out[2], "successor": out[3]}


def strerror(status: int) -> str:
    return _lib.sdm_gx_strerror(int(status)).decode()


def abi_version() -> int:
    return int(_lib.sdm_gx_abi_version())
