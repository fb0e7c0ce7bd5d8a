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


def test_bench_gpus_2_launches_two_ranks_by_itself():
    """A plain ``bench.py --gpus 2`` (no launcher) runs two ranks under
    torch.distributed.run; the measured step is replaced by a CPU stand-in
    (tests/bench_stub_main.py), so this checks the launch, the gloo group
    and the max over ranks."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_PORT")}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bench_stub_main.py"), "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [json.loads(x) for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.stdout
    assert lines[0]["n_gpus"] == 2 and lines[0]["ms_per_step"] == 2.0


def test_bench_refuses_a_world_size_other_than_gpus():
    import subprocess
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bench_stub_main.py"), "--gpus", "2",
                          "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 2 and "WORLD_SIZE=1" in out.stderr
