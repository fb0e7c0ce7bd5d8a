"""The multi-rank path of bench.py on CPU (gloo, world size 2).

The operator shards over independent (batch, head) units, so ranks share no
data; bench.py only exchanges the step time (max over ranks) and gives each
rank its own seed.  These tests run that host logic with two gloo ranks.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    from hybrid_gated_linear_attn_b300.inputs import WORKLOADS, prefill_inputs
    w, r, local = bench.dist_setup()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        t = bench.max_over_ranks(1.5 + r, w)                 # each rank's own step time
        wl = WORKLOADS["tiny_f32"]
        q = prefill_inputs(wl, seed=bench.rank_seed(wl.seed, r))["q"]
        checksum = float(q.double().sum())
        out[r] = (w, r, local, t, checksum)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time_and_draw_their_own_inputs():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(out)
    assert sorted(res) == [0, 1]
    for r, (w, rr, local, t, _) in res.items():
        assert (w, rr, local) == (2, r, r)
        assert t == 2.5                                      # max over ranks of 1.5 + rank
    assert res[0][4] != res[1][4]                            # weak scaling: different sequences per rank


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    args = bench.argparse.Namespace(steps=1, warmup=0, sample_heads=1, gpus=2)
    assert bench.run_reference(args, world=2, rank=1) == 0   # other ranks exit 0 without work
