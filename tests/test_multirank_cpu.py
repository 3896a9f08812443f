"""The multi-rank bench logic on CPU with the gloo backend (world size 2): each rank runs its own replica with its own
seed, the only collectives are a barrier and the max-reduction of the timings, and rank 0 reports the summed work."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _child(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        import synth
        got_ws, got_rank, got_local = bench.dist_info()
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        bench.barrier(ws)
        t = bench.max_over_ranks(1.0 + rank, ws, device="cpu")
        w = synth.Workload("mr", 42, T=2, P=2, C=8, hd=8)
        x = synth.make_inputs(w, seed=rank)["x"]
        out[rank] = (t, float(np.abs(x).sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings_and_use_distinct_seeds():
    ws = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_child, args=(r, ws, port, out)) for r in range(ws)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0            # max over ranks
    assert res[0][1] != res[1][1]                   # rank r draws seed r: independent replicas


def test_single_rank_helpers_need_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
