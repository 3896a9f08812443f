"""sdm_gx_gemm_step_noalloc (the entry point whose scratch is a static device array, so that it allocates nothing)
against the existing stateless entry point sdm_gx_gemm_step, bit for bit, over calls in a row. The large shapes are
checked to run the stream kernel (the only kernel that uses the array: partial sums handed between CTAs, flags, launch
counters), and one test interleaves two shapes on the array, each result against the oracle."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import assert_bitwise

pytestmark = pytest.mark.gpu

gx = pytest.importorskip("fp32_gemm_gb300") if torch.cuda.is_available() else None


def _inputs(P, C, hd, seed_id=72, T=2):
    w = synth.Workload("noalloc", seed_id, T=T, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    dev = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    return inp, dev


def _uses_stream_kernel(dev, P):
    g = gx.noalloc_geometry(dev["d_u"], dev["x"], dev["d_dv"], P)
    return g["path"] == 1 and gx.config_info(1, g["config"])["kind"] == "stream", g


@pytest.mark.parametrize("P,C,hd", [(200, 128, 128), (200, 120, 100), (8, 64, 64)])
def test_noalloc_matches_existing_entry_point(P, C, hd):
    inp, dev = _inputs(P, C, hd)
    stream, g = _uses_stream_kernel(dev, P)
    if P >= 200:   # more tiles than SMs: the split over one CTA per SM, through the static array
        assert stream and g["ctas"] == g["sms"], g
    du_ref = dev["d_u"].clone()
    du_new = dev["d_u"].clone()
    gx.device_error(clear=True)
    for ti in (0, 1, 1):   # two consecutive steps, then step 1 again: three calls, two in a row on each pair
        gx.step(du_ref, dev["x"], dev["d_dv"], ti, P, pdl=True)
        gx.step_noalloc(du_new, dev["x"], dev["d_dv"], ti, P, pdl=True)
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


def test_noalloc_interleaved_shapes():
    """Two shapes alternating on the one array (each call's split runs one CTA per SM, so the per-CTA launch counters
    stay equal whatever the shape): large, ragged, large again, each step against the oracle."""
    a_inp, a = _inputs(200, 128, 128, seed_id=73)
    b_inp, b = _inputs(200, 120, 100, seed_id=74)
    assert _uses_stream_kernel(a, 200)[0] and _uses_stream_kernel(b, 200)[0]
    gx.device_error(clear=True)
    gx.step_noalloc(a["d_u"], a["x"], a["d_dv"], 0, 200, pdl=True)
    gx.step_noalloc(b["d_u"], b["x"], b["d_dv"], 1, 200, pdl=True)
    gx.step_noalloc(a["d_u"], a["x"], a["d_dv"], 1, 200, pdl=True)
    gx.step_noalloc(b["d_u"], b["x"], b["d_dv"], 0, 200, pdl=True)
    torch.cuda.synchronize()
    assert gx.device_error(clear=True) == 0
    for inp, dev, P, order in ((a_inp, a, 200, [0, 1]), (b_inp, b, 200, [1, 0])):
        want = inp["d_u"].copy()
        oracle.run_steps(want, inp["x"], inp["d_dv"], P, order=order)
        got = dev["d_u"].cpu().numpy()
        for n in (0, P // 2, P - 1, P, 2 * P - 1):
            assert_bitwise(got[n], want[n], f"interleaved P={P} chunk {n}")


def test_noalloc_offset_bases():
    """Operands 4 bytes past a 16-byte boundary (contiguous views at a storage offset of one float): the allocation-free
    call takes the TMA path's offset configurations like the stateless call, with the same bits."""
    from tests.gpu_util import DevArray
    inp, _ = _inputs(32, 64, 128)
    ref = [DevArray(inp[k], 1) for k in ("d_u", "x", "d_dv")]
    new = [DevArray(inp[k], 1) for k in ("d_u", "x", "d_dv")]
    g = gx.noalloc_geometry(new[0].t, new[1].t, new[2].t, 32)
    assert g["path"] == 1 and gx.config_info(1, g["config"])["kind"].startswith("offset"), g
    gx.device_error(clear=True)
    for ti in (1, 0):
        gx.step(ref[0].t, ref[1].t, ref[2].t, ti, 32, pdl=True)
        gx.step_noalloc(new[0].t, new[1].t, new[2].t, ti, 32, pdl=True)
    torch.cuda.synchronize()
    assert gx.device_error(clear=True) == 0
    assert_bitwise(new[0].host(), ref[0].host(), "noalloc vs step, offset bases")
    want = inp["d_u"].copy()
    oracle.run_steps(want, inp["x"], inp["d_dv"], 32, order=[1, 0])
    assert_bitwise(new[0].host(), want, "noalloc offset bases vs oracle")
    assert all(a.guards_intact() for a in new)


def test_noalloc_rejects_what_step_rejects():
    t = torch.zeros(4, 8, 8, device="cuda")
    with pytest.raises(gx.GxGemmError) as e:
        gx.step_noalloc(t, t, torch.zeros(4, 8, 8, device="cuda"), 0, 2)
    assert e.value.name == "SDM_GX_E_OVERLAP"


def test_noalloc_geometry_flag_alone():
    _, dev = _inputs(8, 64, 64)
    with pytest.raises(gx.GxGemmError) as e:
        gx.geometry(dev["d_u"], dev["x"], dev["d_dv"], 8, flags=gx.FLAG_NOALLOC | gx.FLAG_GENERIC)
    assert e.value.name == "SDM_GX_E_FLAGS"


_CAPTURE_CHILD = r"""
import json, torch
import fp32_gemm_gb300 as gx
P, C, hd = 8, 64, 64
x = torch.randn(2 * P, C, C, device="cuda") * 0.1
dv = torch.randn(2 * P, C, hd, device="cuda")
du = torch.randn(2 * P, C, hd, device="cuda")
gx.geometry(du, x, dv, P)   # the library's per-device set-up happens outside the capture
g = torch.cuda.CUDAGraph()
name = None
with torch.cuda.graph(g):
    try:
        gx.step_noalloc(du, x, dv, 0, P)
    except gx.GxGemmError as e:
        name = e.name
ref = du.clone()
gx.step(ref, x, dv, 0, P)
gx.step_noalloc(du, x, dv, 0, P)   # outside the capture the first call sets the array up and runs
torch.cuda.synchronize()
print(json.dumps({"in_capture": name, "same": bool(torch.equal(du, ref)), "err": gx.device_error(clear=True)}))
"""


def test_noalloc_first_call_in_capture_is_refused():
    """A process whose first allocation-free call comes during stream capture gets SDM_GX_E_CAPTURE (the one-time set-up
    would break the capture) and nothing else happens; the next call outside the capture sets the array up and gives
    the stateless call's bits. Run in a child process, whose array is not set up yet."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CAPTURE_CHILD], capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out == {"in_capture": "SDM_GX_E_CAPTURE", "same": True, "err": 0}, out
