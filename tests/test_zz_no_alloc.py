"""sdm_gx_gemm_step_noalloc (the entry point whose scratch is a static device array, so that it allocates nothing)
against the existing stateless entry point sdm_gx_gemm_step, bit for bit, over two calls in a row: two consecutive
steps, then the same step applied twice (each call advances the launch counters inside the shared array)."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bitwise

pytestmark = pytest.mark.gpu

gx = pytest.importorskip("fp32_gemm_gb300") if torch.cuda.is_available() else None


@pytest.mark.parametrize("P,C,hd", [(200, 128, 128), (160, 100, 76), (8, 64, 64)])
def test_noalloc_matches_existing_entry_point(P, C, hd):
    w = synth.Workload("noalloc", 72, T=2, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    x = torch.from_numpy(inp["x"]).cuda()
    dv = torch.from_numpy(inp["d_dv"]).cuda()
    du_ref = torch.from_numpy(inp["d_u"]).cuda()
    du_new = du_ref.clone()
    gx.device_error(clear=True)
    for ti in (0, 1, 1):   # two consecutive steps, then step 1 again: three calls, two in a row on each pair
        gx.step(du_ref, x, dv, ti, P, pdl=True)
        gx.step_noalloc(du_new, x, dv, ti, P, pdl=True)
    torch.cuda.synchronize()
    assert gx.device_error(clear=True) == 0
    assert_bitwise(du_new.cpu().numpy(), du_ref.cpu().numpy(), f"noalloc vs step P={P} C={C} hd={hd}")
    # and both against the oracle on one chunk of each step
    want = inp["d_u"].copy()
    oracle.run_steps(want, inp["x"], inp["d_dv"], P, order=[0, 1, 1])
    got = du_new.cpu().numpy()
    for n in (0, P - 1, P, 2 * P - 1):
        assert_bitwise(got[n], want[n], f"noalloc chunk {n}")
    assert np.isfinite(got).all()


def test_noalloc_rejects_what_step_rejects():
    t = torch.zeros(4, 8, 8, device="cuda")
    with pytest.raises(gx.GxGemmError) as e:
        gx.step_noalloc(t, t, torch.zeros(4, 8, 8, device="cuda"), 0, 2)
    assert e.value.name == "SDM_GX_E_OVERLAP"
