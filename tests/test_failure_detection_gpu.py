"""Failure detection without a GPU fault: the test hook makes the TMA kernel's producer withhold its first stage, so
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
