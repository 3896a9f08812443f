"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle, bit for bit (NaN as a class), on the
seeded workloads of the gx_gemm page's step update (sparse_delta_memory/cuda/gx_gemm_cuda.py, module docstring
formula), at sizes the oracle finishes in seconds, with ragged tails, every tile configuration, misaligned and
strided layouts, the producer chain and the programmatic-dependent-launch chain."""

import numpy as np
import pytest
import torch

import oracle
import synth
from tests.gpu_util import DevArray, assert_bitwise

pytestmark = pytest.mark.gpu

gx = pytest.importorskip("fp32_gemm_gb300") if torch.cuda.is_available() else None


def _oracle_steps(inp, P, steps, S=None):
    du = inp["d_u"].copy()
    dv = inp["d_dv"].copy()
    for ti in steps:
        if S is not None:
            oracle.producer_step(dv, S, ti, P)
        oracle.step(du, inp["x"], dv, ti, P)
    return du, dv


def _dev(inp, offset=0, row_pad=0):
    return (DevArray(inp["d_u"], offset, row_pad), DevArray(inp["x"], offset, 0),
            DevArray(inp["d_dv"], offset, row_pad))


def _check_untouched(dx, dv, inp, what):
    assert_bitwise(dx.host(), inp["x"], what + " x modified")
    assert_bitwise(dv.host(), inp["d_dv"], what + " d_dv modified")


@pytest.fixture(autouse=True)
def _no_device_errors():
    gx.device_error(clear=True)
    yield
    assert gx.device_error(clear=True) == 0, "a kernel gave up a bounded wait"


@pytest.mark.parametrize("pdl", [False, True])
@pytest.mark.parametrize("mode", ["plan_run", "plan_step", "step", "step_ex"])
def test_tiny_all_steps(mode, pdl):
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    du, dx, dv = _dev(inp)
    if mode == "plan_run":
        pl = gx.Plan(du.t, dx.t, dv.t, w.P)
        pl.run(pdl=pdl)
    elif mode == "plan_step":
        pl = gx.Plan(du.t, dx.t, dv.t, w.P)
        for ti in reversed(range(w.T)):
            pl.step(ti, pdl=pdl)
    elif mode == "step":
        for ti in range(w.T):
            gx.step(du.t, dx.t, dv.t, ti, w.P, pdl=pdl)
    else:
        for ti in range(w.T):
            gx.step_ex(du.t, dx.t, dv.t, ti, w.P, pdl=pdl)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"tiny {mode}")
    assert du.guards_intact() and dx.guards_intact() and dv.guards_intact()
    _check_untouched(dx, dv, inp, "tiny")


def _ragged_workload():
    # C and hd not multiples of any tile; C % 4 == 0 and hd % 4 == 0 so the TMA path is eligible
    return synth.Workload("ragged", 60, T=2, P=3, C=100, hd=76, x_scale="inv_sqrt_c")


MAX_TMA_CONFIGS = 24   # the parametrisation below covers every configuration while the menu stays within this


def test_config_menu_covered():
    assert gx.num_configs(1) <= MAX_TMA_CONFIGS, "extend MAX_TMA_CONFIGS so that every configuration is tested"


@pytest.mark.parametrize("config", list(range(MAX_TMA_CONFIGS)))
def test_every_tma_config_ragged(config):
    if config >= gx.num_configs(1):
        pytest.skip("no such configuration")
    w = _ragged_workload()
    kind = gx.config_info(1, config)["kind"]
    if kind == "slab":
        # the slab kernel needs whole 32-row slabs: ragged in columns and P only
        w = synth.Workload("ragged_slab", 65, T=2, P=5, C=96, hd=76, x_scale="inv_sqrt_c")
    elif kind == "stream":
        # the stream kernel needs at least one tile per SM: 160 one-tile chunks, ragged in rows and columns
        w = synth.Workload("ragged_stream", 67, T=2, P=160, C=100, hd=76, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, [1, 0])
    du, dx, dv = _dev(inp)
    flags = gx.config_flag(config)
    if kind == "stream":   # stateless calls have no workspace: the stream kernel exists for plans only
        with pytest.raises(gx.GxGemmError) as e:
            gx.geometry(du.t, dx.t, dv.t, w.P, flags=flags)
        assert e.value.name == "SDM_GX_E_FLAGS"
    else:
        g = gx.geometry(du.t, dx.t, dv.t, w.P, flags=flags)
        assert g["path"] == 1 and g["config"] == config
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=flags)
    assert pl.geometry()["config"] == config
    pl.run(1, -1, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"tma config {config}")
    assert du.guards_intact()
    _check_untouched(dx, dv, inp, f"tma config {config}")


GENERIC_CONFIGS = [0, 1, 2, 3]


@pytest.mark.parametrize("config", list(range(MAX_TMA_CONFIGS)))
def test_every_tile_config_multi_round(config):
    """Every tile configuration forced on a step with more tiles than resident CTAs (400 chunks of 100 x 76: a CTA
    runs two or more tiles, so the configurations that store the tiles before a CTA's last by TMA do so), ragged in rows
    and columns, two chained steps, bit-exact against the oracle with the guard bands intact."""
    if config >= gx.num_configs(1) or gx.config_info(1, config)["kind"] != "tile":
        pytest.skip("not a tile configuration")
    w = synth.Workload("multi_round", 66, T=2, P=400, C=100, hd=76, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, [1, 0])
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(config))
    g = pl.geometry()
    assert g["config"] == config and g["tiles"] > g["ctas"]
    pl.run(1, -1, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"tile config {config}, {g['tiles']} tiles on {g['ctas']} CTAs")
    assert du.guards_intact()
    _check_untouched(dx, dv, inp, f"tile config {config}")


def test_generic_menu_covered():
    assert gx.num_configs(0) == len(GENERIC_CONFIGS), "every generic configuration must be in GENERIC_CONFIGS"


@pytest.mark.parametrize("config", GENERIC_CONFIGS)
@pytest.mark.parametrize("shape", [(100, 76), (48, 99), (256, 3), (1, 1), (7, 130)])
def test_every_generic_config(config, shape):
    C, hd = shape
    w = synth.Workload("gen", 61, T=2, P=2, C=C, hd=hd, x_scale="unit")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, [0, 1])
    du, dx, dv = _dev(inp)
    flags = gx.FLAG_GENERIC | gx.config_flag(config)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=flags)
    assert pl.geometry()["path"] == 0
    pl.run(pdl=False)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"generic {config} {shape}")
    assert du.guards_intact()


EDGE_VARIANTS = {
    "hd100": dict(hd=100, offset=0, row_pad=0, path=1),
    "hd99": dict(hd=99, offset=0, row_pad=0, path=0),
    "hd128_misaligned": dict(hd=128, offset=1, row_pad=0, path=1),   # an offset configuration (aligned-down maps)
    "hd128_ld129": dict(hd=128, offset=0, row_pad=1, path=0),
    "hd128_ld132": dict(hd=128, offset=0, row_pad=4, path=1),
}


@pytest.mark.parametrize("variant", sorted(EDGE_VARIANTS))
@pytest.mark.parametrize("vset", synth.VALUE_SETS)
def test_edge_patterns(vset, variant):
    v = EDGE_VARIANTS[variant]
    w = synth.WORKLOADS["edge"]
    inp = synth.make_inputs(w, value_set=vset, hd=v["hd"])
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    du, dx, dv = _dev(inp, offset=v["offset"], row_pad=v["row_pad"])
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    assert pl.geometry()["path"] == v["path"], pl.geometry()
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"edge {vset} {variant}")
    assert du.guards_intact() and dx.guards_intact() and dv.guards_intact()
    _check_untouched(dx, dv, inp, f"edge {vset} {variant}")
    got = du.host()
    zero = (got == 0) & ~np.isnan(got)
    assert not np.any(np.signbit(got[zero])), "a -0 output"


def _offset_configs():
    return [k for k in range(gx.num_configs(1)) if gx.config_info(1, k)["kind"].startswith("offset")]


OFFSET_PATTERNS = [(1, 1, 1), (2, 0, 3), (3, 2, 1), (0, 1, 0), (0, 0, 2)]   # floats past 16 bytes: d_u, x, d_dv


@pytest.mark.parametrize("offs", OFFSET_PATTERNS)
@pytest.mark.parametrize("shape", [(3, 100, 76), (2, 48, 128), (5, 12, 4)])
def test_offset_bases_every_offset_config(shape, offs):
    """Operand bases 4, 8 or 12 bytes past a 16-byte boundary, each operand its own offset: the plan takes an offset
    configuration (TMA from aligned-down maps; element loads of wider boxes, or tiles on the shifted grid), and every
    offset configuration, forced, gives the oracle's bits, ragged in rows, columns and j, without touching the floats
    around the operands. A configuration of the aligned kernels, forced on such bases, is refused, and so is a
    shifted-grid one where d_u and d_dv lie differently far off."""
    P, C, hd = shape
    w = synth.Workload("offset", 69, T=2, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, [1, 0])
    cfgs = _offset_configs()
    assert cfgs
    auto = None
    for k in [None] + cfgs:
        du = DevArray(inp["d_u"], offs[0])
        dx, dv = DevArray(inp["x"], offs[1]), DevArray(inp["d_dv"], offs[2])
        if k is not None and gx.config_info(1, k)["kind"] == "offset_shifted" and offs[0] != offs[2]:
            with pytest.raises(gx.GxGemmError) as e:   # the shifted grid needs d_u and d_dv equally far off
                gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(k))
            assert e.value.name == "SDM_GX_E_FLAGS"
            continue
        pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=0 if k is None else gx.config_flag(k))
        g = pl.geometry()
        assert g["path"] == 1 and gx.config_info(1, g["config"])["kind"].startswith("offset"), g
        if k is None:
            auto = g["config"]
        pl.run(1, -1, pdl=True)
        torch.cuda.synchronize()
        assert_bitwise(du.host(), want, f"offset config {k if k is not None else auto} {shape} {offs}")
        assert du.guards_intact() and dx.guards_intact() and dv.guards_intact()
        _check_untouched(dx, dv, inp, f"offset config {k}")
    # a configuration of the aligned kernels, forced on offset bases, is refused
    du = DevArray(inp["d_u"], offs[0])
    dx, dv = DevArray(inp["x"], offs[1]), DevArray(inp["d_dv"], offs[2])
    with pytest.raises(gx.GxGemmError) as e:
        gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(0))
    assert e.value.name == "SDM_GX_E_FLAGS"


@pytest.mark.parametrize("vset", synth.VALUE_SETS)
def test_offset_configs_value_sets(vset):
    """Every offset configuration, forced, on every value set (zeros and signed zeros, 1e30 magnitudes, wide exponents,
    denormals, +-Inf and NaN sprinkled in): bases 4 bytes past a 16-byte boundary, a shape with several row and column
    tiles and a ragged last stage, compared with the oracle bit for bit (NaN as a class)."""
    w = synth.Workload("offset_vsets", 80, T=2, P=2, C=100, hd=136, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w, value_set=vset)
    want, _ = _oracle_steps(inp, w.P, [1, 0])
    for k in _offset_configs():
        du, dx, dv = _dev(inp, offset=1)
        pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(k))
        pl.run(1, -1, pdl=True)
        torch.cuda.synchronize()
        assert_bitwise(du.host(), want, f"offset config {k} on {vset}")
        assert du.guards_intact()


def test_offset_bases_large_shape():
    """The large shape (P = 256, C = hd = 128) with every base 4 bytes past a 16-byte boundary: two full steps through
    the plan's offset configuration, compared everywhere."""
    w = synth.WORKLOADS["large"]
    inp = synth.make_inputs(w, N=2 * w.P)
    want, _ = _oracle_steps(inp, w.P, [0, 1])
    du, dx, dv = _dev(inp, offset=1)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    g = pl.geometry()
    assert g["path"] == 1 and gx.config_info(1, g["config"])["kind"].startswith("offset"), g
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, "large 2 steps, offset bases")
    assert du.guards_intact() and dx.guards_intact() and dv.guards_intact()


def test_producer_chain_full():
    """T=64, P=8, C=64, hd=64; d_dv rewritten before every step by the synthetic producer; PDL chain."""
    w = synth.WORKLOADS["producer_chain"]
    inp = synth.make_inputs(w)
    S = synth.make_source(w)
    want_du, want_dv = _oracle_steps(inp, w.P, range(w.T), S=S)
    du, dx, dv = _dev(inp)
    Sd = torch.from_numpy(S).cuda()
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    pl.run_producer(Sd, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want_du, "producer chain d_u")
    assert_bitwise(dv.host(), want_dv, "producer chain d_dv")
    assert du.guards_intact() and dv.guards_intact()


def test_pdl_chain_full():
    """T=128, P=32, C=64, hd=128, all steps chained with PDL, reverse order."""
    w = synth.WORKLOADS["pdl_chain"]
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    pl.run(w.T - 1, -1, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, "pdl chain")
    assert du.guards_intact()


def test_large_two_steps():
    """The large shape (P=256, C=128, hd=128) over two full steps, compared everywhere."""
    w = synth.WORKLOADS["large"]
    inp = synth.make_inputs(w, N=2 * w.P)
    want, _ = _oracle_steps(inp, w.P, [0, 1])
    for workspace in (True, False):   # the plan's choice with a workspace (stream kernel) and without (tile kernel)
        du, dx, dv = _dev(inp)
        pl = gx.Plan(du.t, dx.t, dv.t, w.P, workspace=workspace)
        kind = gx.config_info(1, pl.geometry()["config"])["kind"]
        assert (kind == "stream") == workspace, kind
        pl.run(pdl=True)
        torch.cuda.synchronize()
        assert_bitwise(du.host(), want, f"large 2 steps ({kind} kernel)")
        assert du.guards_intact()


def test_kernel_attrs_no_spills():
    for path in (0, 1):
        for k in range(gx.num_configs(path)):
            a = gx.kernel_attrs(path, k)
            assert a["local_bytes"] == 0, (path, k, a)
            assert a["regs"] <= 255


def test_errors_on_device():
    """Errors that need the device: host memory is not device memory; a plan used for a ti beyond ti_max."""
    w = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(w)
    du, dx, dv = _dev(inp)
    host = torch.from_numpy(inp["d_u"].copy())
    rc = gx.lib().sdm_gx_gemm_step(host.data_ptr(), dx.t.data_ptr(), dv.t.data_ptr(), 0, w.P, w.C, w.hd, None, 0)
    assert gx.GxGemmError(rc, "step").name == "SDM_GX_E_DEVICE"
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, ti_max=1)
    with pytest.raises(gx.GxGemmError) as e2:
        pl.step(2)
    assert e2.value.name == "SDM_GX_E_PLAN_TI"


def test_graph_chain_replayed_twice():
    """The chain captured into a CUDA graph, replayed twice: every step applied twice (oracle applied twice)."""
    w = synth.WORKLOADS["pdl_chain"]
    inp = synth.make_inputs(w, N=8 * w.P)
    want, _ = _oracle_steps(inp, w.P, list(range(8)) * 2)
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    g = pl.graph(7, -1, pdl=True)
    c0 = gx.launch_counts()
    g.launch()
    g.launch()
    torch.cuda.synchronize()
    c1 = gx.launch_counts()
    assert c1["step"] - c0["step"] == 16
    assert_bitwise(du.host(), want, "graph chain x2")
    assert du.guards_intact()
    g.close()


def test_graph_producer_chain():
    w = synth.WORKLOADS["producer_chain"]
    inp = synth.make_inputs(w, N=16 * w.P)
    S = synth.make_source(w, N=16 * w.P)
    want_du, want_dv = _oracle_steps(inp, w.P, range(16), S=S)
    du, dx, dv = _dev(inp)
    Sd = torch.from_numpy(S).cuda()
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    g = pl.graph(0, 16, pdl=True, S=Sd)
    g.launch()
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want_du, "graph producer chain d_u")
    assert_bitwise(dv.host(), want_dv, "graph producer chain d_dv")


def test_large_full_size_bench_configuration_sampled():
    """The large workload at full size (N = 8192, 1.6 GB), run exactly as bench.py times it (the library's CUDA graph
    of the 32-step PDL chain); checked against the oracle on whole chunks of two steps and on 4000 random outputs."""
    w = synth.WORKLOADS["large"]
    inp = synth.make_inputs(w)
    d = {k: torch.from_numpy(v).cuda() for k, v in inp.items()}
    pl = gx.Plan(d["d_u"], d["x"], d["d_dv"], w.P)
    assert pl.geometry() == gx.Plan(d["d_u"], d["x"], d["d_dv"], w.P).geometry()
    assert gx.config_info(1, pl.geometry()["config"])["kind"] == "stream"   # the kernel bench.py times
    g = pl.graph(0, w.T, pdl=True)
    g.launch()
    torch.cuda.synchronize()
    got = d["d_u"].cpu().numpy()
    # whole chunks: the first chunk of step 0 and the last chunk of step T-1
    for n in (0, w.N - 1):
        want = inp["d_u"].copy()
        oracle.step(want, inp["x"], inp["d_dv"], n, 1)
        assert_bitwise(got[n], want[n], f"large chunk {n}")
    rng = np.random.default_rng(8)
    n = rng.integers(0, w.N, 4000)
    i = rng.integers(0, w.C, 4000)
    c = rng.integers(0, w.hd, 4000)
    pts = oracle.points(inp["d_u"], inp["x"], inp["d_dv"], n, i, c)
    assert_bitwise(got[n, i, c], pts, "large sampled outputs")


def _cross_pattern(P, C, hd, pattern, seed):
    """One step's operands in one of the six value patterns of the gx_gemm page's qualification probe (its
    `_probe_inputs`: normal values with signed zeros, half zeros, magnitudes spread over 2^-60..2^60 with values near
    the float32 maximum, denormal-scale products, rows that nearly cancel, and sprinkled NaN / infinities / -0 /
    subnormals / near-maximum values). Our own generator (numpy, seeded); x [P, C, C], d_dv and d_u [P, C, hd]."""
    g = np.random.default_rng(seed)
    x = (g.standard_normal((P, C, C)) * 0.25).astype(np.float32)
    dv = g.standard_normal((P, C, hd)).astype(np.float32)
    du = g.standard_normal((P, C, hd)).astype(np.float32)
    if pattern == "normal":
        x.reshape(-1)[::7] = -0.0
        dv.reshape(-1)[::11] = 0.0
        du.reshape(-1)[::13] = -0.0
    elif pattern == "zeros":
        x[g.random(x.shape) < 0.5] = -0.0
        dv[g.random(dv.shape) < 0.5] = 0.0
        du[g.random(du.shape) < 0.5] = -0.0
    elif pattern == "large":
        for t in (x, dv, du):
            t *= np.exp2(g.integers(-60, 61, t.shape)).astype(np.float32)
        x.reshape(-1)[::17] = 3.0e38
        dv.reshape(-1)[::19] = -3.0e38
    elif pattern == "denormal":
        x *= np.float32(1e-20)
        dv *= np.float32(1e-19)
        du *= np.float32(1e-38)
        du.reshape(-1)[::5] = np.float32(1e-41)
    elif pattern == "cancel":
        x = (np.sign(g.standard_normal((P, C, C))) * (1.0 + g.random((P, C, C)))).astype(np.float32)
        dv *= np.float32(1e4)
        h = C // 2
        dv[:, 1:2 * h:2, :] = (-dv[:, 0:2 * h:2, :] * (1.0 + 1e-3 * g.standard_normal((P, h, hd)))).astype(np.float32)
        du *= np.float32(1e-3)
    elif pattern == "special":
        vals = np.array([np.nan, np.inf, -np.inf, -0.0, 1e-41, 3.4e38, -3.4e38], np.float32)
        for t, k in ((dv, 64), (x, 16), (du, 32)):
            fl = t.reshape(-1)
            pos = g.permutation(fl.size)[:k]
            fl[pos] = vals[np.arange(k) % vals.size]
    return x, dv, du


def _forced_nan(x, dv, du):
    """Outputs that IEEE arithmetic makes NaN in ANY summation order: a NaN operand in the output's chain or its d_u,
    a zero times an infinity, or exact infinite products (or d_u) of both signs. (Infinities reached by overflow are
    order-dependent and left out.)"""
    x64, v64, u64 = x.astype(np.float64), dv.astype(np.float64), du.astype(np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        prod = x64[:, :, :, None] * v64[:, :, None, :]          # [P, j, i, c]
    nan = np.isnan(prod).any(axis=1) | np.isnan(u64)
    xinf, vinf = np.isinf(x64), np.isinf(v64)
    pos = ((xinf[:, :, :, None] | vinf[:, :, None, :]) & (prod > 0)).any(axis=1) | (np.isposinf(u64))
    neg = ((xinf[:, :, :, None] | vinf[:, :, None, :]) & (prod < 0)).any(axis=1) | (np.isneginf(u64))
    return nan | (pos & neg)


def test_informative_cublas_cross_check():
    """The pages' second reference: cuBLAS FP32 batched GEMM (torch.baddbmm on the x.transpose(1, 2) view, TF32 off)
    computed the same chain on the configurations the page tested, but that is not a cuBLAS guarantee. Informative,
    as the page's qualification probe is set up: the six value patterns against every 4-byte base offset mod 256 of
    each operand (the others 256-byte aligned; 16-byte-aligned offsets take the aligned TMA configurations, the others
    the offset ones), and the bitwise agreement printed per pattern and operand. Required: finite results of both within the
    recursive-summation error bound of each other, and NaN from both wherever IEEE forces it in every order."""
    P, C, hd = 3, 64, 96
    bound_k = 2 * (C + 1) * 2.0 ** -24
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    rows = []
    try:
        for pi, pattern in enumerate(("normal", "zeros", "large", "denormal", "cancel", "special")):
            x, dv, du = _cross_pattern(P, C, hd, pattern, 20261203 + 7919 * pi)
            with np.errstate(invalid="ignore", over="ignore"):
                scale = np.abs(du).astype(np.float64) + np.einsum("nji,njc->nic", np.abs(x).astype(np.float64),
                                                                   np.abs(dv).astype(np.float64))
            forced = _forced_nan(x, dv, du)
            for operand in ("d_u", "x", "d_dv"):
                agree = []
                for res in range(0, 256, 4):
                    off = {"d_u": 0, "x": 0, "d_dv": 0}
                    off[operand] = res // 4
                    u_d = DevArray(du, offset_floats=off["d_u"])
                    x_d = DevArray(x, offset_floats=off["x"])
                    v_d = DevArray(dv, offset_floats=off["d_dv"])
                    ref = torch.baddbmm(u_d.t, x_d.t.transpose(1, 2), v_d.t)
                    gx.step_ex(u_d.t, x_d.t, v_d.t, 0, P)
                    torch.cuda.synchronize()
                    a, b = u_d.host(), ref.cpu().numpy()
                    assert u_d.guards_intact()
                    agree.append(float(np.mean(a.view(np.uint32) == b.view(np.uint32))))
                    both = np.isfinite(a) & np.isfinite(b)
                    with np.errstate(invalid="ignore"):
                        err = np.abs(a.astype(np.float64) - b.astype(np.float64))
                    assert np.all(err[both] <= bound_k * scale[both] * 1.0001 + 1e-44), (pattern, operand, res)
                    assert np.isnan(a[forced]).all() and np.isnan(b[forced]).all(), (pattern, operand, res)
                rows.append((pattern, operand, min(agree), float(np.mean(agree)), max(agree)))
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    print("\nbitwise agreement with cuBLAS baddbmm over 64 base offsets mod 256 (min / mean / max):")
    for pattern, operand, lo, mean, hi in rows:
        print(f"  {pattern:8s} offset on {operand:5s}: {lo:.4f} / {mean:.4f} / {hi:.4f}")


@pytest.mark.parametrize("graph", [False, True])
def test_successor_chain(graph):
    """Each step followed by the synthetic successor under PDL: the successor of step ti sees exactly d_u after step
    ti (each chunk's leading-row sum in the fixed order), and d_u itself matches the oracle."""
    w = synth.WORKLOADS["pdl_chain"]
    T = 6
    inp = synth.make_inputs(w, N=T * w.P)
    du, dx, dv = _dev(inp)
    out = torch.full((T * w.P,), float("nan"), device="cuda")
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    if graph:
        pl.graph(0, T, pdl=True, succ_out=out).launch()
    else:
        pl.run_successor(out, pdl=True)
    torch.cuda.synchronize()
    ref = inp["d_u"].copy()
    want_out = np.empty((T * w.P,), np.float32)
    for ti in range(T):
        oracle.step(ref, inp["x"], inp["d_dv"], ti, w.P)
        want_out[ti * w.P:(ti + 1) * w.P] = oracle.successor_rows(ref, ti, w.P)
    assert_bitwise(du.host(), ref, "d_u under the successor chain")
    assert_bitwise(out.cpu().numpy(), want_out, "successor row sums")


@pytest.mark.parametrize("C,hd,P,N,path", [
    (256, 256, 2, 4, None),      # the largest C
    (256, 36, 1, 2, None),
    (64, 1000, 2, 4, None),      # many column tiles
    (12, 8, 3, 7, None),         # P does not divide N: chunk 6 is never touched
    (96, 68, 2, 4, "generic"),
])
def test_corner_shapes(C, hd, P, N, path):
    w = synth.Workload("corner", 62, T=N // P, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w, N=N)
    T = N // P
    want, _ = _oracle_steps(inp, P, range(T))
    du, dx, dv = _dev(inp)
    flags = gx.FLAG_GENERIC if path == "generic" else 0
    pl = gx.Plan(du.t, dx.t, dv.t, P, flags=flags)
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"corner C={C} hd={hd} P={P} N={N}")
    assert du.guards_intact()


@pytest.mark.parametrize("x_pad,expect_path", [(4, 1), (1, 0)])
def test_strided_x(x_pad, expect_path):
    """x rows padded (x_sj = C + pad): a multiple-of-4 pad keeps the TMA path, an odd pad falls back to generic."""
    w = synth.Workload("sx", 63, T=2, P=3, C=64, hd=64)
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    du = DevArray(inp["d_u"])
    dv = DevArray(inp["d_dv"])
    dx = DevArray(inp["x"], 0, x_pad)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    assert pl.geometry()["path"] == expect_path
    pl.run(pdl=False)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"strided x pad {x_pad}")
    assert dx.guards_intact()


def test_x_and_d_dv_may_alias():
    """x and d_dv may be the same memory (both only read); d_u may not overlap either."""
    w = synth.Workload("alias", 64, T=2, P=2, C=32, hd=32)
    inp = synth.make_inputs(w)
    inp["d_dv"] = inp["x"].copy()
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    du = DevArray(inp["d_u"])
    dx = DevArray(inp["x"])
    pl = gx.Plan(du.t, dx.t, dx.t, w.P)
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, "x aliased with d_dv")
    with pytest.raises(gx.GxGemmError) as e:
        gx.Plan(dx.t, dx.t, du.t, w.P)
    assert e.value.name == "SDM_GX_E_OVERLAP"


@pytest.mark.parametrize("P,C,hd,T", [(256, 128, 128, 2), (37, 128, 128, 2), (7, 96, 200, 3), (160, 128, 64, 2),
                                      (3, 128, 128, 2)])
def test_slab_kernel_shapes(P, C, hd, T):
    """The balanced slab kernel: full rounds (four slabs of one chunk), rounds across chunks, partial rounds, several
    column blocks, fewer slabs than SMs."""
    slab = [k for k in range(gx.num_configs(1)) if gx.config_info(1, k)["kind"] == "slab"][0]
    w = synth.Workload("slab", 66, T=T, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, P, range(T))
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, P, flags=gx.config_flag(slab))
    assert pl.geometry()["config"] == slab
    g = pl.graph(0, T, pdl=True)
    g.launch()
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"slab P={P} C={C} hd={hd}")
    assert du.guards_intact()


def test_run_host_overlapped_copies():
    """sdm_gx_gemm_plan_run_host: the chain fed from pinned host memory with copies overlapped; d_u comes back to the
    host array. Two calls in a row (the second starts from the first's result) match the oracle applied twice."""
    w = synth.WORKLOADS["pdl_chain"]
    T = 6
    inp = synth.make_inputs(w, N=T * w.P)
    want, _ = _oracle_steps(inp, w.P, list(range(T)) * 2)
    host = {k: torch.from_numpy(v.copy()).pin_memory() for k, v in inp.items()}
    dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}
    pl = gx.Plan(dev["d_u"], dev["x"], dev["d_dv"], w.P)
    d2h = pl.run_host(host["d_u"], host["x"], host["d_dv"])
    d2h = pl.run_host(host["d_u"], host["x"], host["d_dv"])
    d2h.synchronize()
    torch.cuda.synchronize()
    assert_bitwise(host["d_u"].numpy(), want, "run_host x2")
    assert_bitwise(host["x"].numpy(), inp["x"], "x host unchanged")


def _stream_config(thread_tile="8x8"):
    """The stream configuration with 128 x 128 tiles and one CTA per SM whose threads hold thread_tile outputs: 8 x 8
    (8 consumer warps, the large step's) or 8 x 4 (16 consumer warps)."""
    warps = {"8x4": 16, "8x8": 8}[thread_tile]
    ks = [k for k in range(gx.num_configs(1)) if gx.config_info(1, k)["kind"] == "stream"
          and gx.config_info(1, k)["TC"] == 128 and gx.config_info(1, k)["consumer_warps"] == warps]
    assert len(ks) == 1, ks
    return ks[0]


@pytest.mark.parametrize("thread_tile", ["8x4", "8x8"])
@pytest.mark.parametrize("P,C,hd,T", [(160, 100, 76, 2), (153, 64, 64, 2), (100, 128, 200, 2), (304, 128, 128, 2),
                                      (200, 32, 500, 2), (256, 128, 128, 2), (1000, 32, 64, 2), (160, 256, 128, 2)])
def test_stream_kernel_shapes(P, C, hd, T, thread_tile):
    """The stream kernel (a step's (tile, j) work split evenly over one CTA per SM; chains continued across CTAs from
    the accumulators left in the plan's workspace): ragged rows and columns, one tile more than SMs (hand-offs with
    almost no slack), several column blocks, exactly two tiles per CTA (no split), the large step, many whole tiles
    per CTA (1000 tiles), and C = 256 (two row blocks per chunk). The chain is captured into a graph and replayed
    twice, so the workspace's launch epoch advances over 2T launches. Both 128 x 128 thread tilings."""
    k = _stream_config(thread_tile)
    w = synth.Workload("stream", 68, T=T, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, P, list(range(T - 1, -1, -1)) * 2)
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, P, flags=gx.config_flag(k))
    g = pl.geometry()
    assert g["config"] == k and g["ctas"] == g["sms"]
    assert pl.workspace_bytes > 0
    gr = pl.graph(T - 1, -1, pdl=True)
    gr.launch()
    gr.launch()
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"stream P={P} C={C} hd={hd}")
    assert du.guards_intact()
    _check_untouched(dx, dv, inp, "stream")
    gr.close()


def test_stream_kernel_direct_launches_then_graph():
    """Plan launches outside a graph (plain and PDL) and a graph on the same workspace, interleaved: every launch
    reads the epoch its predecessor left."""
    k = _stream_config()
    w = synth.Workload("stream2", 69, T=3, P=160, C=96, hd=96, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, [0, 1, 2, 2, 1, 0, 1])
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(k))
    pl.step(0, pdl=False)
    pl.run(1, 3, pdl=True)
    gr = pl.graph(2, -1, pdl=True)
    gr.launch()
    pl.step(1, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, "stream interleaved launches")
    gr.close()


def test_stream_workspace_rules():
    """Without a workspace the stream kernel is not available (forcing it is an error); the workspace size is 0 for
    shapes with fewer tiles than SMs; a misaligned or overlapping workspace is refused."""
    k = _stream_config()
    small = synth.WORKLOADS["tiny"]
    inp = synth.make_inputs(small)
    du, dx, dv = _dev(inp)
    assert gx.workspace_size(du.t, dx.t, dv.t, small.P) == 0
    w = synth.Workload("stream3", 70, T=1, P=160, C=64, hd=64, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    du, dx, dv = _dev(inp)
    n = gx.workspace_size(du.t, dx.t, dv.t, w.P)
    assert n > 0
    with pytest.raises(gx.GxGemmError) as e:
        gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(k), workspace=False)
    assert e.value.name == "SDM_GX_E_FLAGS"
    L = gx.lib()
    import ctypes
    uv, xv, vv = du.t, dx.t, dv.t
    s = gx.Strides(xv.stride(0), xv.stride(1), vv.stride(0), vv.stride(1), uv.stride(0), uv.stride(1))
    buf = torch.empty(n + 512, dtype=torch.uint8, device="cuda")
    base = (buf.data_ptr() + 255) // 256 * 256
    h = ctypes.c_void_p()
    rc = L.sdm_gx_gemm_plan_create_ws(ctypes.byref(h), uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), w.N, w.P, w.C,
                                      w.hd, ctypes.byref(s), 0, 0, base + 16, n)
    assert gx.strerror(rc) and rc == -4          # SDM_GX_E_ALIGN
    rc = L.sdm_gx_gemm_plan_create_ws(ctypes.byref(h), uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), w.N, w.P, w.C,
                                      w.hd, ctypes.byref(s), 0, 0, (uv.data_ptr() + 255) // 256 * 256, n)
    assert rc == -5                              # SDM_GX_E_OVERLAP
    rc = L.sdm_gx_gemm_plan_create_ws(ctypes.byref(h), uv.data_ptr(), xv.data_ptr(), vv.data_ptr(), w.N, w.P, w.C,
                                      w.hd, ctypes.byref(s), 0, 0, base, n)
    assert rc == 0
    L.sdm_gx_gemm_plan_destroy(h)


def test_stream_kernel_strided_rows():
    """The stream kernel on row-padded views (leading dimension hd + 4 for d_u and d_dv, C + 4 for x: strided, still
    TMA-eligible): the tensor maps carry the strides, the hand-off does not depend on them."""
    k = _stream_config()
    w = synth.Workload("stream_ld", 73, T=2, P=160, C=64, hd=64, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, [1, 0])
    du, dx, dv = _dev(inp, row_pad=4)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(k))
    assert pl.geometry()["config"] == k
    pl.run(1, -1, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, "stream kernel, padded rows")
    assert du.guards_intact()
    _check_untouched(dx, dv, inp, "stream kernel, padded rows")


def test_run_host_stream_kernel():
    """The host-buffer driver on a shape the plan runs with the stream kernel (its workspace held by the plan), as the
    bench's end-to-end leg does on the large workload: two calls in a row match the oracle applied twice."""
    w = synth.Workload("host_stream", 74, T=4, P=200, C=64, hd=64, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, list(range(w.T)) * 2)
    host = {k: torch.from_numpy(v.copy()).pin_memory() for k, v in inp.items()}
    dev = {k: torch.empty_like(v, device="cuda") for k, v in host.items()}
    pl = gx.Plan(dev["d_u"], dev["x"], dev["d_dv"], w.P, flags=gx.config_flag(_stream_config()))
    d2h = pl.run_host(host["d_u"], host["x"], host["d_dv"])
    d2h = pl.run_host(host["d_u"], host["x"], host["d_dv"])
    d2h.synchronize()
    torch.cuda.synchronize()
    assert_bitwise(host["d_u"].numpy(), want, "run_host stream kernel x2")


@pytest.mark.parametrize("P,C,hd", [(2600, 32, 64), (3100, 48, 36)])
def test_stream_kernel_many_tiles_per_cta(P, C, hd):
    """The 8 x 8 stream configuration past 16 tiles a CTA (17 and 20 tiles an SM; no bound for the configuration that
    stores mid-CTA tiles by TMA): two chained steps and the reverse, bit-exact; the 8 x 4 configuration, bounded at 16
    tiles a CTA, is refused when forced on the same shape."""
    k = _stream_config("8x8")
    w = synth.Workload("stream_many", 86, T=2, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, P, [0, 1, 1, 0])
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, P, flags=gx.config_flag(k))
    g = pl.geometry()
    assert g["config"] == k and g["tiles"] > 16 * g["ctas"]
    pl.run(0, 2, pdl=True)
    pl.step(1, pdl=False)   # not a dependent launch of the step 1 before it (it writes this step's d_u)
    pl.step(0, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"stream 8x8, {g['tiles']} tiles on {g['ctas']} CTAs")
    assert du.guards_intact()
    _check_untouched(dx, dv, inp, "stream many tiles")
    with pytest.raises(gx.GxGemmError) as e:
        gx.Plan(du.t, dx.t, dv.t, P, flags=gx.config_flag(_stream_config("8x4")))
    assert e.value.name == "SDM_GX_E_FLAGS"


def _random_stream_shapes(n, seed, sms=152):
    """n step shapes (P, C, hd) on which a 128 x 128 stream configuration with one CTA per SM is admitted: C and hd
    multiples of 4 (TMA rows), 1 or 2 row blocks and 1 to 3 column blocks per chunk, between one and four tiles a CTA."""
    import random
    rng = random.Random(seed)
    out = []
    while len(out) < n:
        C = 4 * rng.randint(1, 64)
        hd = 4 * rng.randint(1, 96)
        per_chunk = -(-C // 128) * -(-hd // 128)
        P = -(-rng.randint(sms, 4 * sms) // per_chunk)
        if sms <= P * per_chunk <= 16 * sms:
            out.append((P, C, hd))
    return out


@pytest.mark.parametrize("thread_tile", ["8x4", "8x8"])
@pytest.mark.parametrize("shape", _random_stream_shapes(6, 2026))
def test_stream_kernel_random_shapes(shape, thread_tile):
    """Seeded random shapes through the stream kernel (any split point, ragged rows and columns in any tile, one to
    three column blocks, tight and loose hand-offs), steps 0, 1, 1, 0, bit-exact against the oracle; the guard bands
    around d_u stay intact and x and d_dv are not written."""
    P, C, hd = shape
    k = _stream_config(thread_tile)
    w = synth.Workload("stream_rand", 80 + P % 7, T=2, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, P, [0, 1, 1, 0])
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, P, flags=gx.config_flag(k))
    assert pl.geometry()["config"] == k
    pl.run(0, 2, pdl=True)
    # step 1 again: not a dependent launch of the step 1 before it, which writes its d_u (the PDL contract: the
    # predecessor writes neither x nor this step's d_u)
    pl.step(1, pdl=False)
    pl.step(0, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"stream {thread_tile} P={P} C={C} hd={hd}")
    assert du.guards_intact()
    _check_untouched(dx, dv, inp, "stream random")


@pytest.mark.parametrize("thread_tile", ["8x4", "8x8"])
@pytest.mark.parametrize("vset", synth.VALUE_SETS)
def test_stream_kernel_value_sets(vset, thread_tile):
    """The stream kernel on every value set (zeros and signed zeros, 1e30-scale overflow, the wide range, subnormals,
    +-Inf, NaN): the FP32 accumulators handed between CTAs through shared memory, bulk copies and the workspace keep
    their bits (NaN as a class), and no output is -0. 160 chunks of 48 x 100: every hand-off is tight."""
    k = _stream_config(thread_tile)
    w = synth.Workload("stream_vs", 75, T=2, P=160, C=48, hd=100, x_scale="unit")
    inp = synth.make_inputs(w, value_set=vset)
    want, _ = _oracle_steps(inp, w.P, [0, 1])
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(k))
    assert pl.geometry()["config"] == k
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"stream kernel, {vset}")
    assert du.guards_intact()
    got = du.host()
    zero = (got == 0) & ~np.isnan(got)
    assert not np.any(np.signbit(got[zero])), "a -0 output"


def _stream_configs():
    return [k for k in range(gx.num_configs(1)) if gx.config_info(1, k)["kind"] == "stream"]


@pytest.mark.parametrize("P,C,hd", [(400, 128, 64), (320, 96, 60), (600, 64, 128)])
def test_stream_kernel_all_tile_shapes(P, C, hd):
    """Every stream configuration (128 x 128 tiles with one CTA per SM; 128 x 64 tiles with two per SM, 304 CTAs and
    a workspace sized for them) on shapes it splits: column blocks of 64, ragged rows and columns, many tiles per CTA.
    A graph of the two steps, replayed twice."""
    w = synth.Workload("stream_ts", 76, T=2, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, P, [1, 0] * 2)
    for k in _stream_configs():
        du, dx, dv = _dev(inp)
        pl = gx.Plan(du.t, dx.t, dv.t, P, flags=gx.config_flag(k))
        g = pl.geometry()
        info = gx.config_info(1, k)
        assert g["config"] == k and g["ctas"] == g["sms"] * g["ctas_per_sm"], (g, info)
        gr = pl.graph(1, -1, pdl=True)
        gr.launch()
        gr.launch()
        torch.cuda.synchronize()
        assert_bitwise(du.host(), want, f"stream config {k} ({info['TI']} x {info['TC']}) P={P} C={C} hd={hd}")
        assert du.guards_intact()
        gr.close()


@pytest.mark.parametrize("case", ["ws", "no_ws", "generic"])
def test_autotune_then_plan_is_bit_exact(case):
    """sdm_gx_gemm_autotune times the admitted configurations on a scratch copy of d_u; a plan forced to its pick
    gives the oracle's bits, and the tuning leaves x, d_dv and the real d_u alone. 160 x 64 x 128 is a shape where
    the plan's estimate is not the fastest; the generic case (rows padded to 129 floats) tunes the generic path."""
    P, C, hd = (160, 64, 128) if case != "generic" else (16, 48, 100)
    w = synth.Workload("autotune", 61, T=2, P=P, C=C, hd=hd)
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    row_pad = 29 if case == "generic" else 0
    du, dx, dv = _dev(inp, row_pad=row_pad)
    scratch = DevArray(inp["d_u"], 0, row_pad)
    res = gx.autotune(scratch.t, dx.t, dv.t, w.P, steps=10, workspace=(case == "ws"))
    torch.cuda.synchronize()
    path = 0 if case == "generic" else 1
    assert 0 <= res["config"] < gx.num_configs(path) and res["us"] > 0.0
    assert res["flags"] == gx.config_flag(res["config"])
    if case == "no_ws":
        assert gx.config_info(1, res["config"])["kind"] != "stream"
    assert_bitwise(du.host(), inp["d_u"], "autotune touched d_u")
    _check_untouched(dx, dv, inp, "autotune")
    assert scratch.guards_intact() and dx.guards_intact() and dv.guards_intact()
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=res["flags"], workspace=(case == "ws"))
    g = pl.geometry()
    assert (g["path"], g["config"]) == (path, res["config"])
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"autotuned plan ({case})")
    assert du.guards_intact()


@pytest.mark.parametrize("shape", [(64, 64, 128), (48, 64, 128), (100, 32, 64), (32, 64, 128)])
def test_latency_rule_prefers_small_tiles(shape):
    """Small steps take the configuration with the most tiles that fit one wave, and among equally many tiles the
    smallest tile (rows and columns past C and hd cost time too): 64 x 64 or 32 x 128 on C = 64 rather than 128 x 64,
    32 x 64 on C = 32 rather than 128 x 128 (measured 4.2 against 5.8 and 2.7 against 5.4 us a step). The pick is
    bit-exact like every configuration."""
    P, C, hd = shape
    w = synth.Workload("latency_rule", 62, T=2, P=P, C=C, hd=hd)
    inp = synth.make_inputs(w)
    du, dx, dv = _dev(inp)
    pl = gx.Plan(du.t, dx.t, dv.t, w.P)
    g = pl.geometry()
    sms = g["sms"]
    tiles = lambda k: P * -(-C // gx.config_info(1, k)["TI"]) * -(-hd // gx.config_info(1, k)["TC"])
    assert g["path"] == 1 and tiles(g["config"]) <= sms
    for k in range(gx.num_configs(1)):
        info = gx.config_info(1, k)
        if info["kind"] != "tile" or tiles(k) > sms:
            continue
        assert tiles(k) <= tiles(g["config"]), (k, g)
        if tiles(k) == tiles(g["config"]):
            assert info["TI"] * info["TC"] >= g["TI"] * g["TC"], (k, g)
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"latency rule {shape}")


@pytest.mark.parametrize("layout", ["ld129", "offset4"])
def test_generic_large_tile_kernel(layout):
    """The generic path's large-tile kernel (128 x 64 tiles, packed FMAs, double-buffered cp.async staging) on layouts
    TMA cannot describe: rows of 129 floats, and bases 4 bytes past a 16-byte boundary with x rows of 130 floats.
    80 chunks of C = 130, hd = 100 span several tiles per CTA with ragged rows, columns and j; the plan picks the
    kernel itself once its tiles fill the SMs (here forced, then checked on a filling step)."""
    w = synth.Workload("generic_big", 63, T=2, P=80, C=130, hd=100, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    offset, row_pad = (0, 29) if layout == "ld129" else (1, 0)
    du, dx, dv = _dev(inp, offset=offset, row_pad=row_pad)
    big = gx.num_configs(0) - 1
    pl = gx.Plan(du.t, dx.t, dv.t, w.P, flags=gx.config_flag(big))
    g = pl.geometry()
    assert (g["path"], g["config"], g["TI"], g["TC"]) == (0, big, 128, 64)
    pl.run(w.T - 1, -1, pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"generic large-tile kernel ({layout})")
    assert du.guards_intact() and dx.guards_intact() and dv.guards_intact()
    _check_untouched(dx, dv, inp, f"generic large-tile kernel ({layout})")
    # a step whose 128 x 64 tiles fill the SMs takes it without being asked
    assert 2 * w.P * 2 >= g["sms"]
    auto = gx.Plan(du.t, dx.t, dv.t, w.P).geometry()
    assert (auto["path"], auto["config"]) == (0, big)



@pytest.mark.parametrize("vset", synth.VALUE_SETS)
def test_transposed_x_view_edge(vset):
    """x given as the page's baddbmm call sees it: stored as [n][i][j] (x.transpose(1, 2) of the stored tensor is the
    logical x[n, j, i]). The edge workload's ragged shape (C = 48, hd = 99), every value set, a PDL chain of its T
    steps; bit-exact against the oracle on the logical x, guards and x untouched."""
    w = synth.WORKLOADS["edge"]
    inp = synth.make_inputs(w, value_set=vset, hd=99)
    want, _ = _oracle_steps(inp, w.P, range(w.T))
    stored = np.ascontiguousarray(inp["x"].transpose(0, 2, 1))   # [n][i][j]
    dxs = DevArray(stored)
    du, dv = DevArray(inp["d_u"]), DevArray(inp["d_dv"])
    xview = dxs.t.transpose(1, 2)
    pl = gx.Plan(du.t, xview, dv.t, w.P)
    g = pl.geometry()
    assert g["path"] == 0 and g["config"] < gx.num_configs(0) - 1, g
    pl.run(pdl=True)
    torch.cuda.synchronize()
    assert_bitwise(du.host(), want, f"transposed x {vset}")
    assert du.guards_intact() and dxs.guards_intact() and dv.guards_intact()
    assert np.array_equal(dxs.host().view(np.uint32), stored.view(np.uint32))


@pytest.mark.parametrize("P,C,hd", [(160, 100, 76), (200, 128, 128), (3, 256, 40)])
def test_transposed_x_view_shapes(P, C, hd):
    """The transposed x on filling steps (the 64-row generic kernel), the large step's chunk shape, and C = 256 with a
    narrow hd; through step_ex (one step), a plan graph replayed twice in reverse, and against the row-major x."""
    T = 2
    w = synth.Workload("xt", 77, T=T, P=P, C=C, hd=hd, x_scale="inv_sqrt_c")
    inp = synth.make_inputs(w)
    want, _ = _oracle_steps(inp, P, [1, 0] * 2)
    stored = np.ascontiguousarray(inp["x"].transpose(0, 2, 1))
    xs = torch.from_numpy(stored).cuda()
    du = torch.from_numpy(inp["d_u"]).cuda()
    dv = torch.from_numpy(inp["d_dv"]).cuda()
    pl = gx.Plan(du, xs.transpose(1, 2), dv, P)
    assert pl.geometry()["path"] == 0
    gr = pl.graph(T - 1, -1, pdl=True)
    gr.launch()
    gr.launch()
    torch.cuda.synchronize()
    assert_bitwise(du.cpu().numpy(), want, f"transposed x P={P} C={C} hd={hd}")
    # one step through step_ex equals the same step on the row-major x
    du1 = torch.from_numpy(inp["d_u"]).cuda()
    du2 = du1.clone()
    gx.step_ex(du1, xs.transpose(1, 2), dv, 1, P, pdl=False)
    gx.step_ex(du2, torch.from_numpy(inp["x"]).cuda(), dv, 1, P, pdl=False)
    torch.cuda.synchronize()
    assert_bitwise(du1.cpu().numpy(), du2.cpu().numpy(), "transposed vs row-major x")
