"""The plan's configuration choice on a described GB300-like device, without a GPU (sdm_gx_gemm_choose_config runs the
same host rule as plan creation). The device: 152 SMs and the resident CTAs per SM of every configuration, both as a
GB300 reports them through plan geometry (1 for the 128 x 128 tiles, their offset variant and the one-CTA stream
configuration, 2 for the 64-128-row tiles, 4 for 32 x 64 and 16 x 64 and both offset 32 x 64 variants, 10 for the
one-warp tiles and the offset 8 x 32; generic 6, 4, 2, 2). The expected picks are the configurations measured fastest on a
GB300 for these shapes."""

import pytest

gx = pytest.importorskip("fp32_gemm_gb300")

SMS = 152
TMA_OCC = [1, 1, 2, 2, 2, 2, 2, 4, 4, 10, 10, 1, 1, 2, 1, 1, 4, 4, 10]
GEN_OCC = [6, 4, 2, 2]
WS = 64 << 20   # a plan workspace large enough for every stream configuration


def pick(P, C, hd, ws=WS, path=1):
    occ = TMA_OCC if path == 1 else GEN_OCC
    return gx.choose_config(path, SMS, occ, P, C, hd, ws_bytes=ws)


def info(k):
    return gx.config_info(1, k)


def test_description_matches_the_menu():
    assert gx.num_configs(1) == len(TMA_OCC) and gx.num_configs(0) == len(GEN_OCC)


def test_large_step_takes_the_stream_kernel_with_a_workspace():
    k = pick(256, 128, 128)
    assert info(k)["kind"] == "stream" and (info(k)["TI"], info(k)["TC"]) == (128, 128)
    assert info(k)["consumer_warps"] == 8   # 8 x 8 outputs a thread: measured 21.8-21.9 us against 22.3 for 8 x 4
    k0 = pick(256, 128, 128, ws=0)   # without a workspace: a tile kernel on 128 x 64 or larger tiles
    assert info(k0)["kind"] == "tile" and info(k0)["TI"] * info(k0)["TC"] >= 128 * 64


def test_many_tiles_per_sm():
    """The 8 x 8 stream configuration, whose CTAs store the tiles they finish before their last piece by TMA, is offered
    at any number of tiles a CTA (8192 chunks of the large shape, 54 tiles an SM: 531 us a step against 568 on whole
    tiles). A stream configuration whose consumers store every tile is offered only up to 16 tiles a CTA (with 8 x 4
    tiles: 584 us against 568); without the 8 x 8 one (no slot for it on the described device) the rule then takes
    whole tiles."""
    for P in (2048, 8192):
        k = pick(P, 128, 128)
        assert info(k)["kind"] == "stream" and info(k)["consumer_warps"] == 8, (P, k)
    k14 = pick(256, 128, 128)
    occ = list(TMA_OCC)
    occ[k14] = 0
    k = gx.choose_config(1, SMS, occ, 8192, 128, 128, ws_bytes=WS)
    assert info(k)["kind"] == "tile"
    k = gx.choose_config(1, SMS, occ, 2048, 128, 128, ws_bytes=WS)   # 13.5 tiles an SM
    assert info(k)["kind"] == "stream" and info(k)["consumer_warps"] == 16


@pytest.mark.parametrize("shape,tile", [((32, 64, 128), (32, 64)),    # pdl_chain: 128 tiles of 32 x 64
                                        ((8, 64, 64), (8, 32)),       # producer_chain: 128 tiles of 8 x 32
                                        ((2, 16, 32), (8, 32)),       # tiny
                                        ((4, 48, 100), (8, 32))])     # edge, hd = 100
def test_latency_bound_steps_fill_one_wave_with_the_most_tiles(shape, tile):
    k = pick(*shape)
    assert (info(k)["TI"], info(k)["TC"]) == tile


@pytest.mark.parametrize("shape", [(64, 64, 128), (48, 64, 128), (72, 64, 96), (100, 32, 64)])
def test_ties_go_to_the_smallest_tile(shape):
    """Among configurations with equally many tiles in one wave the smallest tile wins (rows and columns past C and hd
    cost time): never 128 x 64 on C = 64 or 128 x 128 on C = 32."""
    P, C, hd = shape
    k = pick(*shape)
    tiles = lambda j: P * -(-C // info(j)["TI"]) * -(-hd // info(j)["TC"])
    same = [j for j in range(len(TMA_OCC)) if info(j)["kind"] == "tile" and tiles(j) == tiles(k)]
    assert tiles(k) <= SMS
    assert info(k)["TI"] * info(k)["TC"] == min(info(j)["TI"] * info(j)["TC"] for j in same)
    assert info(k)["TI"] <= max(C, 32)


def test_generic_path_large_tile_kernel_for_filling_steps():
    assert pick(256, 128, 128, path=0) == len(GEN_OCC) - 1   # 512 tiles of 128 x 64: the large-tile kernel
    assert pick(4, 48, 99, path=0) == 0                      # 4 chunks: 16-row tiles in one wave
    # 70 x 100 x 100: 140 tiles of 128 x 64 do not fill 152 SMs; 980 16-row tiles exceed one wave of 152 x 6 resident
    # CTAs, 560 32-row tiles fit one of 152 x 4
    assert pick(70, 100, 100, path=0) == 1
    assert pick(40, 100, 100, path=0) == 0                   # 560 16-row tiles fit one wave


def test_argument_errors():
    codes = gx._binding.CODE
    with pytest.raises(gx.GxGemmError) as e:
        gx.choose_config(1, 0, TMA_OCC, 8, 64, 64)
    assert e.value.status == codes["SDM_GX_E_RANGE"]
    with pytest.raises(gx.GxGemmError) as e:
        gx.choose_config(1, SMS, TMA_OCC[:-1], 8, 64, 64)
    assert e.value.status == codes["SDM_GX_E_RANGE"]
    with pytest.raises(gx.GxGemmError) as e:
        gx.choose_config(2, SMS, TMA_OCC, 8, 64, 64)
    assert e.value.status == codes["SDM_GX_E_FLAGS"]
    with pytest.raises(gx.GxGemmError) as e:
        gx.choose_config(1, SMS, TMA_OCC, 8, 0, 64)
    assert e.value.status == codes["SDM_GX_E_SHAPE"]
    with pytest.raises(gx.GxGemmError) as e:
        gx.choose_config(1, SMS, [0] * len(TMA_OCC), 8, 64, 64)   # nothing resident: nothing usable
    assert e.value.status == codes["SDM_GX_E_SMEM"]


def _sweep(name="config_sweep_gb300.jsonl"):
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "data", name)
    with open(path) as f:
        return [json.loads(line) for line in f if line.strip()]


def _excess(r, k):
    """The measured step time of pick k over the fastest configuration the rule may take for these contiguous operands
    (the sweep also times the offset configurations, forced, which serve only operand bases off a 16-byte boundary)."""
    aligned = [v for kk, v in r["us"].items() if info(int(kk))["kind"] in ("tile", "slab", "stream")]
    return r["us"][str(k)] / min(aligned) - 1.0


def test_rule_against_the_measured_sweep():
    """The rule's pick on each of 66 shapes (C 32 .. 128, hd 64 .. 128, P 48 .. 800), against every configuration
    timed on one GB300 (tests/data/config_sweep_gb300.jsonl, written by tests/data/sweep_configs.py): the pick is one
    the shape admits, and its measured step time is close to the fastest. The bounds hold the fitted model's result on
    this recording (mean 1.2 % and worst 7.8 % over the fastest at C = 64 and 96, 37 of 42 within 5 %; 2.4 % and
    12.5 % at C = 32, 48 and 128, where the close calls sit between configurations within a few tenths of a
    microsecond); the earlier whole-round estimate scored 7.1 % / 41.9 % on the first set. (Since the 8 x 8 and 4 x 8
    tiles store mid-CTA tiles by TMA they are faster, 6% and 2% at the median, and closer to their neighbours than the
    model's fixed costs can rank: the rule's picks ran 1.2% faster on average than on the menu before, 29 shapes by
    more than 2% and 3 slower by more than 2%, while the excess over the fastest grew.)"""
    rows = _sweep()
    assert len(rows) == 66
    excess = {True: [], False: []}
    for r in rows:
        k = pick(r["P"], r["C"], r["hd"])
        assert str(k) in r["us"], (r["P"], r["C"], r["hd"], k)
        excess[r["C"] in (64, 96)].append(_excess(r, k))
    small, wide = excess[True], excess[False]
    assert len(small) == 42 and len(wide) == 24
    assert sum(small) / len(small) <= 0.015 and max(small) <= 0.08
    assert sum(1 for e in small if e <= 0.05) >= 37
    assert sum(wide) / len(wide) <= 0.025 and max(wide) <= 0.125


def test_rule_against_the_large_c_sweep():
    """The same against 18 shapes with C = 192 and 256 (hd 64 .. 256, P 16 .. 200; the tile, slab and stream
    configurations timed on one GB300, tests/data/config_sweep_gb300_large_c.jsonl, the large_c set of
    tests/data/sweep_configs.py): mean 1.6% and worst 12.4% over the fastest (before the slab kernel was kept out of the
    latency-bound branch: 4.8% and 28%; the worst picks are tile kernels next to the 64 x 128 tile with its TMA
    stores)."""
    rows = _sweep("config_sweep_gb300_large_c.jsonl")
    assert len(rows) == 18
    excess = []
    for r in rows:
        k = pick(r["P"], r["C"], r["hd"])
        assert str(k) in r["us"], (r["P"], r["C"], r["hd"], k)
        excess.append(_excess(r, k))
    assert sum(excess) / len(excess) <= 0.025 and max(excess) <= 0.13


def test_rule_against_the_narrow_sweep():
    """The same against 18 narrow shapes (C 16 .. 64, hd 16 and 32, P 64 .. 1024;
    tests/data/config_sweep_gb300_narrow.jsonl, the narrow set of tests/data/sweep_configs.py): mean 0.9% and worst
    8.1% over the fastest (one wave of one-warp CTAs counts two an SM: 3.5% and 14% on an earlier recording)."""
    rows = _sweep("config_sweep_gb300_narrow.jsonl")
    assert len(rows) == 18
    excess = []
    for r in rows:
        k = pick(r["P"], r["C"], r["hd"])
        assert str(k) in r["us"], (r["P"], r["C"], r["hd"], k)
        excess.append(_excess(r, k))
    assert sum(excess) / len(excess) <= 0.015 and max(excess) <= 0.085
