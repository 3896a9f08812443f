"""The timeline build of the library (libsdm_gx_gemm_trace.so: sdm_gx_gemm_plan_set_trace; its kernels carry per-CTA
global-timer stamps). The default build refuses the call; the timeline build's tests run in a child process that loads
that build (SDM_GX_TRACE_BUILD=1), with the same bit-exactness requirement as every other kernel."""

import importlib.util
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TRACE_CHILD = os.environ.get("SDM_GX_TRACE_BUILD") == "1"
pytestmark = pytest.mark.gpu

gx = pytest.importorskip("fp32_gemm_gb300") if torch.cuda.is_available() else None


def _build_trace_library():
    spec = importlib.util.spec_from_file_location("_sdm_gx_gemm_build", os.path.join(ROOT, "fp32_gemm_gb300",
                                                                                     "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(trace=True)


if not TRACE_CHILD:
    def test_default_build_refuses_a_timeline():
        import synth
        w = synth.Workload("trace", 76, T=2, P=8, C=64, hd=64)
        d = {k: torch.from_numpy(v).cuda() for k, v in synth.make_inputs(w).items()}
        pl = gx.Plan(d["d_u"], d["x"], d["d_dv"], 8)
        with pytest.raises(gx.GxGemmError) as e:
            pl.set_trace(torch.zeros(64, dtype=torch.int64, device="cuda"), 1)
        assert e.value.name == "SDM_GX_E_UNSUPPORTED"

    def test_timeline_build_in_a_child_process():
        _build_trace_library()
        env = dict(os.environ, SDM_GX_TRACE_BUILD="1")
        r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", os.path.abspath(__file__)],
                           capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
        assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
        assert "passed" in r.stdout
else:
    import oracle
    import synth
    from tests.gpu_util import DevArray, assert_bitwise

    def test_the_timeline_build_is_loaded():
        assert gx.LIB_PATH.endswith("libsdm_gx_gemm_trace.so")

    @pytest.mark.parametrize("P,C,hd,T,kind", [(32, 64, 128, 3, "tile"), (160, 100, 76, 3, "stream")])
    def test_timeline_stamps_and_unchanged_results(P, C, hd, T, kind):
        """Every CTA of every traced step writes its stamps in order (start <= past the wait <= first data (stream
        kernel) <= done), steps at or past `launches` write nothing, step ti + 1's chains start only after every CTA of
        step ti is done (the dependency wait), and the results stay bit-exact with the timeline on."""
        w = synth.Workload("trace", 76, T=T, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
        inp = synth.make_inputs(w)
        want = inp["d_u"].copy()
        for ti in range(T):
            oracle.step(want, inp["x"], inp["d_dv"], ti, P)
        du, dx, dv = DevArray(inp["d_u"]), DevArray(inp["x"]), DevArray(inp["d_dv"])
        k = [j for j in range(gx.num_configs(1)) if gx.config_info(1, j)["kind"] == kind][0] if kind == "stream" else None
        pl = gx.Plan(du.t, dx.t, dv.t, P, flags=gx.config_flag(k) if k is not None else 0)
        assert gx.config_info(1, pl.geometry()["config"])["kind"] == kind
        ctas = pl.set_trace(None, 0)
        assert ctas == pl.geometry()["ctas"]
        buf = torch.zeros((T * ctas * 4,), dtype=torch.int64, device="cuda")
        pl.set_trace(buf, T - 1)   # the last step is not traced
        pl.run(pdl=True)
        torch.cuda.synchronize()
        assert_bitwise(du.host(), want, f"traced {kind}")
        a = buf.view(T, ctas, 4).cpu().numpy()
        assert (a[T - 1] == 0).all()
        s = a[:T - 1]
        assert (s[:, :, 0] > 0).all() and (s[:, :, 1] >= s[:, :, 0]).all() and (s[:, :, 3] >= s[:, :, 1]).all()
        if kind == "stream":
            assert (s[:, :, 2] >= s[:, :, 1]).all() and (s[:, :, 3] >= s[:, :, 2]).all()
        assert s[1, :, 1].min() >= s[0, :, 3].max()
        pl.set_trace(None, 0)
