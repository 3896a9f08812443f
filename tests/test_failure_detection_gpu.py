"""Failure detection without a GPU fault: the test hook makes the TMA kernels' producer withhold its first stage, so
every wait on it runs out after its short bound (~20 ms). The launch must complete, the device error word must report
the expired waits, and the context must stay usable: a normal launch right after gives oracle-exact results."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import DevArray, assert_bitwise

pytestmark = pytest.mark.gpu

gx = pytest.importorskip("fp32_gemm_gb300") if torch.cuda.is_available() else None


def test_expired_waits_are_reported_and_the_context_survives():
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w)
    du, dx, dv = (DevArray(inp[k]) for k in ("d_u", "x", "d_dv"))
    gx.device_error(clear=True)
    stalled = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.FLAG_TEST_STALL)
    assert stalled.geometry()["path"] == 1
    stalled.step(0)
    torch.cuda.synchronize()                       # returns: the waits were bounded
    word = gx.device_error(clear=True)
    assert word & 1, f"consumer wait not reported: {word:#x}"
    assert gx.device_error(clear=True) == 0        # cleared
    # the context is still usable: a normal plan on fresh buffers matches the oracle bit for bit
    du2, dx2, dv2 = (DevArray(inp[k]) for k in ("d_u", "x", "d_dv"))
    ok = gx.Plan(du2.t, dx2.t, dv2.t, w.P)
    ok.run(pdl=True)
    torch.cuda.synchronize()
    want = inp["d_u"].copy()
    oracle.run_steps(want, inp["x"], inp["d_dv"], w.P)
    assert_bitwise(du2.host(), want, "after the stall test")
    assert gx.device_error(clear=True) == 0
    assert np.isfinite(du2.host()).all()


def _stream_config(thread_tile):
    """The stream configuration with 128 x 128 tiles and one CTA per SM whose threads hold thread_tile outputs (8 x 4:
    16 consumer warps; 8 x 8: 8, the large step's)."""
    warps = {"8x4": 16, "8x8": 8}[thread_tile]
    ks = [c for c in range(gx.num_configs(1)) if gx.config_info(1, c)["kind"] == "stream"
          and gx.config_info(1, c)["TC"] == 128 and gx.config_info(1, c)["consumer_warps"] == warps]
    assert len(ks) == 1, ks
    return ks[0]


@pytest.mark.parametrize("thread_tile", ["8x4", "8x8"])
def test_stream_kernel_expired_waits_are_reported(thread_tile):
    """The same hook on the stream kernel (one CTA per SM, chains handed between CTAs through the plan's workspace):
    both stalled launches complete with the error word set, the context stays usable, and a stream-kernel plan on
    fresh buffers then matches the oracle over two passes of its steps."""
    k = _stream_config(thread_tile)
    w = synth.Workload("stall_stream", 71, T=2, P=160, C=64, hd=64, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    du, dx, dv = (DevArray(inp[k_]) for k_ in ("d_u", "x", "d_dv"))
    gx.device_error(clear=True)
    stalled = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.FLAG_TEST_STALL | gx.config_flag(k))
    assert stalled.geometry()["config"] == k
    stalled.step(0)
    stalled.step(1)
    torch.cuda.synchronize()
    word = gx.device_error(clear=True)
    assert word & 1, f"consumer wait not reported: {word:#x}"
    du2, dx2, dv2 = (DevArray(inp[k_]) for k_ in ("d_u", "x", "d_dv"))
    ok = gx.Plan(du2.t, dx2.t, dv2.t, w.P, flags=gx.config_flag(k))
    ok.run(pdl=True)
    ok.run(pdl=True)
    torch.cuda.synchronize()
    want = inp["d_u"].copy()
    oracle.run_steps(want, inp["x"], inp["d_dv"], w.P)
    oracle.run_steps(want, inp["x"], inp["d_dv"], w.P)
    assert_bitwise(du2.host(), want, "stream kernel after the stall test")
    assert gx.device_error(clear=True) == 0


@pytest.mark.parametrize("thread_tile", ["8x4", "8x8"])
def test_stream_kernel_late_handoff_recomputes_exactly(thread_tile):
    """A hand-off that never comes (the test hook makes every CTA store but never flag its head's partial sums): each
    tail's wait runs out after its 1 ms bound and the CTA computes that tile's whole chain itself. The steps' results
    are still oracle-exact, the device error word carries only the informational bit 3 (device_error returns it without
    a fault status), and a normal launch on the same workspace afterwards is exact too (the flags it finds are stale,
    and the launch epochs tell)."""
    k = _stream_config(thread_tile)
    w = synth.Workload("late_handoff", 78, T=2, P=160, C=64, hd=64, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    du, dx, dv = (DevArray(inp[k_]) for k_ in ("d_u", "x", "d_dv"))
    gx.device_error(clear=True)
    late = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.FLAG_TEST_NO_HANDOFF | gx.config_flag(k))
    assert late.geometry()["config"] == k
    late.run(pdl=True)
    torch.cuda.synchronize()
    word = gx.device_error(clear=True)
    assert word == 8, f"expected only the informational hand-off bit: {word:#x}"
    want = inp["d_u"].copy()
    oracle.run_steps(want, inp["x"], inp["d_dv"], w.P)
    assert_bitwise(du.host(), want, "late hand-off, recomputed")
    assert du.guards_intact()
    rc = gx.lib().sdm_gx_device_error(__import__("ctypes").byref(__import__("ctypes").c_uint32(0)), 1)
    assert rc == 0
    # the same buffers again with a normal plan of the same configuration
    ok = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(k))
    ok.run(pdl=True)
    torch.cuda.synchronize()
    oracle.run_steps(want, inp["x"], inp["d_dv"], w.P)
    assert_bitwise(du.host(), want, "normal launch after the late hand-offs")
    assert gx.device_error(clear=True) == 0


@pytest.mark.parametrize("kind", ["offset", "offset_shifted"])
def test_offset_configurations_expired_waits_are_reported(kind):
    """The stall hook on the offset configurations (bases 4 bytes past a 16-byte boundary; the realigning 128 x 128
    one waits on its aligned buffers too): every forced configuration of the kind completes its stalled launch with
    the error word set, and a normal launch after it is oracle-exact."""
    w = synth.Workload("stall_offset", 79, T=2, P=3, C=64, hd=128, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    cfgs = [k for k in range(gx.num_configs(1)) if gx.config_info(1, k)["kind"] == kind]
    assert cfgs
    for k in cfgs:
        du, dx, dv = (DevArray(inp[n], 1) for n in ("d_u", "x", "d_dv"))
        gx.device_error(clear=True)
        stalled = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.FLAG_TEST_STALL | gx.config_flag(k))
        stalled.step(0)
        torch.cuda.synchronize()
        word = gx.device_error(clear=True)
        assert word & 1, f"config {k}: consumer wait not reported: {word:#x}"
        du2, dx2, dv2 = (DevArray(inp[n], 1) for n in ("d_u", "x", "d_dv"))
        ok = gx.Plan(du2.t, dx2.t, dv2.t, w.P, flags=gx.config_flag(k))
        ok.run(pdl=True)
        torch.cuda.synchronize()
        want = inp["d_u"].copy()
        oracle.run_steps(want, inp["x"], inp["d_dv"], w.P)
        assert_bitwise(du2.host(), want, f"config {k} after the stall test")
        assert gx.device_error(clear=True) == 0
