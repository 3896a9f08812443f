"""Time every TMA configuration, forced, against the plan's own pick on a set of step shapes (one GPU; run by hand,
not a test): each plan runs a CUDA graph of 8 PDL-chained steps of P chunks, 3 warm-up replays, then 30 timed replays
bracketed by CUDA events, in three passes of which the fastest is kept (a single pass now and then reads a few percent
high on a latency-bound step). One JSON line per shape: P, C, hd, the pick and its time, and the time of every configuration
the shape admits (microseconds per step). The inputs are N(0, 0.1) x, N(0, 1) d_dv and d_u, contiguous.

    python tests/data/sweep_configs.py [small_c|wide|large_c|narrow] > out.jsonl

small_c: C in {64, 96} x hd in {64, 96, 128} x P in {48 .. 600}; wide: C in {32, 48, 128} x hd in {64, 128} x
P in {100 .. 800}; large_c: C in {192, 256} x hd in {64, 128, 256} x P in {16, 64, 200}; narrow: C in {16, 32, 64} x
hd in {16, 32} x P in {64, 256, 1024}. config_sweep_gb300.jsonl holds
the first two sets, config_sweep_gb300_large_c.jsonl and config_sweep_gb300_narrow.jsonl the others (the tile, slab
and stream configurations), as measured on one GB300."""
import json
import os
import sys

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", ".."))

import torch  # noqa: E402

import fp32_gemm_gb300 as gx  # noqa: E402

T = 8
PASSES = 3


def timed(pl, reps=30):
    g = pl.graph(0, T, pdl=True)
    for _ in range(3):
        g.launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.launch()
    e1.record()
    torch.cuda.synchronize()
    g.close()
    return e0.elapsed_time(e1) * 1000 / (reps * T)


def shapes(which):
    if which == "wide":
        return [(P, C, hd) for C in (32, 48, 128) for hd in (64, 128) for P in (100, 200, 400, 800)]
    if which == "large_c":
        return [(P, C, hd) for C in (192, 256) for hd in (64, 128, 256) for P in (16, 64, 200)]
    if which == "narrow":
        return [(P, C, hd) for C in (16, 32, 64) for hd in (16, 32) for P in (64, 256, 1024)]
    return [(P, C, hd) for C in (64, 96) for hd in (64, 96, 128) for P in (48, 100, 160, 220, 300, 400, 600)]


def main():
    which = sys.argv[1] if len(sys.argv) > 1 else "small_c"
    torch.manual_seed(0)
    nk = gx.num_configs(1)
    for (P, C, hd) in shapes(which):
        N = T * P
        x = torch.randn(N, C, C, device="cuda") * 0.1
        dv = torch.randn(N, C, hd, device="cuda")
        du = torch.randn(N, C, hd, device="cuda")
        auto = gx.Plan(du, x, dv, P)
        pick = auto.geometry()["config"]
        pick_us = min(timed(auto) for _ in range(PASSES))
        auto.close()
        per = {}
        for k in range(nk):
            try:
                pl = gx.Plan(du, x, dv, P, flags=gx.config_flag(k))
            except gx.GxGemmError:
                continue   # not admitted for this shape
            per[k] = min(timed(pl) for _ in range(PASSES))
            pl.close()
        print(json.dumps({"P": P, "C": C, "hd": hd, "pick": pick, "pick_us": round(pick_us, 3),
                          "us": {str(k): round(v, 3) for k, v in per.items()}}), flush=True)
        del x, dv, du
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
