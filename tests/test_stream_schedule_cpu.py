"""The stream kernel's split of a step's (tile, j) work over the CTAs, checked on the CPU through the library's own
host copy of the code the kernel runs (sdm_gx_gemm_stream_piece). For every shape: each tile's j range 0..C-1 is
covered exactly once, either whole by one CTA or as a head [0, s) on CTA b and a tail [s, C) on CTA b + 1; a CTA runs
at most one head (first) and one tail (last); the CTAs' work differs by at most one unit, or, where the split charges
each tile boundary inside a range KAPPA units of cost (steps of at least C + 2 KAPPA units per CTA), by at most
2 KAPPA + 1 with the ranges that hold more boundaries the shorter; and, at equal rates, CTA b reaches its tail no
earlier than CTA b - 1 has finished the matching head, so the hand-off never waits on work that has not started."""

import random

import pytest

gx = pytest.importorskip("fp32_gemm_gb300")

KAPPA = 12   # the library's charge per tile boundary of the split (applied when ntiles * C / G >= C + 2 KAPPA)

SHAPES = [(256, 128, 152), (160, 100, 152), (152, 128, 152), (153, 128, 152), (303, 128, 152), (1000, 7, 152),
          (200, 1, 152), (4096, 256, 152), (5, 3, 5), (7, 64, 3), (1, 1, 1), (300, 96, 148)]


def _check(ntiles, C, G):
    cover = {}
    per_cta = []
    heads, tails = {}, {}
    for b in range(G):
        pcs = gx.stream_pieces(ntiles, C, G, b)
        assert pcs, (b, "a CTA without work")
        kinds = [k for (_, _, _, k) in pcs]
        assert kinds.count(1) <= 1 and kinds.count(2) <= 1
        if 1 in kinds:
            assert kinds[0] == 1, "the head runs first"
        if 2 in kinds:
            assert kinds[-1] == 2, "the tail runs last"
        done = 0
        for (t, j0, j1, k) in pcs:
            assert 0 <= t < ntiles and 0 <= j0 < j1 <= C
            if k == 0:
                assert (j0, j1) == (0, C)
            elif k == 1:
                assert j0 == 0 and j1 < C
                heads[t] = (b, j1, done + (j1 - j0))      # CTA, split point, units done when the head ends
            else:
                assert 0 < j0 and j1 == C
                tails[t] = (b, j0, done)                   # CTA, split point, units done when the tail starts
            cover.setdefault(t, []).append((j0, j1))
            done += j1 - j0
        per_cta.append(done)
    assert sum(per_cta) == ntiles * C
    charged = ntiles * C // G >= C + 2 * KAPPA
    assert max(per_cta) - min(per_cta) <= (2 * KAPPA + 1 if charged else 1)
    for t in range(ntiles):
        spans = sorted(cover[t])
        assert spans[0][0] == 0 and spans[-1][1] == C
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 == b0, (t, spans)
        assert len(spans) in (1, 2)
    assert set(heads) == set(tails)
    for t, (bh, sh, end_h) in heads.items():
        bt, st, start_t = tails[t]
        assert bt == bh + 1 and st == sh, (t, heads[t], tails[t])
        assert start_t >= end_h, (t, "tail reached before the head is done")


@pytest.mark.parametrize("shape", SHAPES)
def test_stream_split_invariants(shape):
    _check(*shape)


def test_large_step_charges_the_extra_piece():
    """The large step (256 tiles of 128 x 128 on 152 CTAs, 215.6 units each): CTAs with three pieces (head, whole
    tile, tail) take fewer units than those with two, by about the charge."""
    units = {2: [], 3: []}
    for b in range(152):
        pcs = gx.stream_pieces(256, 128, 152, b)
        units.setdefault(len(pcs), []).append(sum(j1 - j0 for (_, j0, j1, _) in pcs))
    assert units[2] and units[3]
    assert max(units[3]) < min(units[2]) + KAPPA and sum(units[3]) / len(units[3]) < sum(units[2]) / len(units[2]) - 4


def test_stream_split_random_shapes():
    rng = random.Random(7)
    for _ in range(40):
        G = rng.randint(1, 160)
        ntiles = rng.randint(G, 4 * G + 3)
        C = rng.randint(1, 256)
        _check(ntiles, C, G)


def test_stream_split_rejects_short_ranges():
    with pytest.raises(gx.GxGemmError):
        gx.stream_pieces(100, 128, 152, 0)      # fewer tiles than CTAs: a range would be shorter than a tile
    with pytest.raises(gx.GxGemmError):
        gx.stream_pieces(256, 128, 152, 152)    # no such CTA


@pytest.mark.parametrize("ntiles", [100_900, 100_915, 100_916, 101_000, 2_000_000, 16_000_000])
def test_stream_split_on_both_sides_of_32_bit_arithmetic(ntiles):
    """The split is computed in 32-bit arithmetic while G x F fits in 31 bits (F = ntiles (C + KAPPA) - KAPPA, the
    step's cost) and in 64-bit beyond: both give the ranges of the cost formula, here in Python integers."""
    C, G = 128, 152
    F = ntiles * (C + KAPPA) - KAPPA

    def unit_at_cost(y):
        t, r = divmod(y, C + KAPPA)
        return t * C + min(r, C)

    for b in (0, 1, 75, 150, 151):
        pcs = gx.stream_pieces(ntiles, C, G, b)
        lo = min(t * C + j0 for (t, j0, _, _) in pcs)
        hi = max(t * C + j1 for (t, _, j1, _) in pcs)
        assert (lo, hi) == (unit_at_cost(b * F // G), unit_at_cost((b + 1) * F // G)), (ntiles, b)
