#!/usr/bin/env python3
"""Benchmark of the Lizard hybrid attention operator on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one prefill of the Llama-3-8B-shaped workload (B4 H32 L4096
d128 bf16, w64, m4 meta keys, alpha 1): gate log-sigmoid and log-space
cumulative decay, intra- and inter-chunk gated linear attention, window +
meta-sink softmax, alpha combine and the state hand-off, all in the library's
kernels.  The decode step (64 sequences x H32, d128, w64, m4, fp32 state) is
timed in the same run and reported under "decode", and the backward pass of
the same prefill (dq, dk, dv, dg, d meta, d alpha for a seeded upstream
gradient: the training step of the operator) under "backward".  Inputs are seeded
synthetic tensors (no dataset, no weights) larger than L2 and resident in HBM
before the timed region.

Rank 0 prints one JSON line.  With N > 1 (torchrun) every rank runs its own
batch of sequences (weak scaling, no data-path collective); the step time is
the max over ranks.  ``--impl reference`` times the fp64 CPU oracle on this
host's cores instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from hybrid_gated_linear_attn_b300.inputs import (WORKLOADS, decode_initial_state,  # noqa: E402
                                                  decode_step_inputs, prefill_inputs, torch_dtype)

METRIC = "prefill tokens/s & % bf16 TC roofline; decode tokens/s & HBM GB/s (1 B300)"
PREFILL_WL = WORKLOADS["llama3_8b"]
DECODE_WL = WORKLOADS["decode"]
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
PREFILL_KERNEL_SRC = ["csrc/prefill_ws.cuh", "csrc/prefill_cont.cuh", "csrc/sm100.cuh", "csrc/common.cuh"]
DECODE_KERNEL_SRC = ["csrc/decode.cuh", "csrc/common.cuh"]
BACKWARD_KERNEL_SRC = ["csrc/backward_tc.cuh", "csrc/prefill_ws.cuh", "csrc/sm100.cuh", "csrc/common.cuh"]


# --------------------------------------------------------------------------
# algorithmic work (per launch)
# --------------------------------------------------------------------------

def prefill_bytes(wl, B=None) -> int:
    """q, k, v, g read and y written once (5 d elements per token and head),
    plus the final state write per head: S (fp32 d x d) and the ring's w keys
    and values."""
    B = wl.B if B is None else B
    es = 2 if wl.dtype == "bf16" else 4
    units = B * wl.H
    return units * (wl.L * 5 * wl.dk * es + wl.dk * wl.dv * 4 + 2 * wl.w * wl.dk * es)


def backward_bytes(wl, B=None) -> int:
    """q, k, v, g and the upstream gradient dy read, dq, dk, dv, dg written
    once (9 d elements per token and head)."""
    B = wl.B if B is None else B
    es = 2 if wl.dtype == "bf16" else 4
    return B * wl.H * wl.L * 9 * wl.dk * es


def prefill_flops(wl, B=None) -> int:
    """4 d_k d_v (state update and readout) + 2 d (2w + m) (window scores,
    meta scores and weighted values) per token and head."""
    B = wl.B if B is None else B
    return B * wl.H * wl.L * (4 * wl.dk * wl.dv + 2 * wl.dk * (2 * wl.w + wl.m))


def decode_bytes(wl, B=None) -> int:
    """Per sequence and head: S read and written (fp32), the ring's w keys and
    values read, q, k, v, g in and y out, the ring slot written."""
    B = wl.B if B is None else B
    es = 2 if wl.dtype == "bf16" else 4
    per = 2 * wl.dk * wl.dv * 4 + 2 * wl.w * wl.dk * es + 5 * wl.dk * es + 2 * wl.dk * es
    return B * wl.H * per


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


def source_hash(files) -> str:
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "hybrid_gated_linear_attn_b300")
    for f in files:
        with open(os.path.join(pkg, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, files) -> float | None:
    """DRAM bytes per launch recorded from an ncu capture of `kernel`, if the
    kernel's sources are unchanged since (profiles/dram_traffic.txt)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = source_hash(files)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and parts[1] == want:
            return float(parts[2])
    return None


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) >= 9:
                    try:
                        rows.append((float(p[1]), float(p[2]), float(p[3]), p[4:9]))
                    except ValueError:
                        continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # under load: power well above idle
        pmax = max(r[2] for r in rows)
        load = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in load for i, flag in enumerate(r[3][1:5]) if flag.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": pmax, "samples": len(load), "reasons": reasons}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_name(wl) -> str:
    """The bench workload, named the same way by both arms."""
    return f"llama3_8b prefill B{wl.B} H{wl.H} L{wl.L} d{wl.dk} w{wl.w} m{wl.m} {wl.dtype}"


def rank_seed(base: int, rank: int) -> int:
    """Each rank draws its own sequences (weak scaling over the batch)."""
    return base + 1000 * rank


# --------------------------------------------------------------------------
# the CPU oracle arm
# --------------------------------------------------------------------------

def oracle_prefill_sample(inp, wl, heads):
    from oracle import oracle as O
    cores = O.default_threads()
    B, H = wl.B, wl.H
    units = [(b, h) for b in range(B) for h in range(H)][:heads]
    q, k, v, g = (inp[n] for n in ("q", "k", "v", "g"))
    flat = lambda t: t.reshape(B * H, wl.L, -1)[:len(units)]  # noqa: E731
    t0 = time.perf_counter()
    O.forward(flat(q), flat(k), flat(v), flat(g), inp["mu"], wl.alpha, wl.w, threads=cores)
    dt = time.perf_counter() - t0
    tokens = len(units) * wl.L / H   # token positions of a whole sequence (all heads)
    return tokens / dt, dt, cores, len(units)


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    wl = PREFILL_WL
    inp = prefill_inputs(wl)
    heads = wl.B * wl.H if args.sample_heads is None else args.sample_heads
    vals = []
    for _ in range(args.warmup if args.warmup < 1 else 1):
        oracle_prefill_sample(inp, wl, min(heads, 8))
    total = 0.0
    cores = 1
    nunits = 0
    for _ in range(args.steps):
        v, dt, cores, nunits = oracle_prefill_sample(inp, wl, heads)
        vals.append(v)
        total += dt
    value = statistics.median(vals)
    sample = (f"{nunits} of {wl.B * wl.H} (batch, head) units of the llama3_8b prefill workload per step "
              f"(L={wl.L}), fp64, one thread per unit; tokens/s counts whole-sequence positions")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload_name(wl), "global_batch": wl.B, "seq_len": wl.L,
                   "implementation": "fp64 CPU oracle"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

def time_loop(fn, steps, warmup, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps  # ms


def per_launch_ms(fn, steps, stream):
    """Average duration of the launches `fn` enqueues, event-bracketed one by
    one on the launching stream."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def run_ours(args, world, rank, local):
    from hybrid_gated_linear_attn_b300 import LizardState, lizard_attn_decode_step, lizard_attn_prefill
    from hybrid_gated_linear_attn_b300 import lizard_attn as LA
    from hybrid_gated_linear_attn_b300 import lizard_attn_backward, lizard_check_device_status, lizard_gate_projection
    from hybrid_gated_linear_attn_b300.inputs import gate_projection_inputs

    torch.cuda.set_device(local)
    LA.library()  # fails loudly if the CUDA library is missing
    stream = torch.cuda.current_stream()
    peaks, peak_src = load_peaks()
    wl = PREFILL_WL
    Bl = wl.B  # sequences per rank

    # ---- prefill (the step) ----
    inp_cpu = prefill_inputs(wl, seed=rank_seed(wl.seed, rank))
    q, k, v, g, mu = (inp_cpu[n].cuda() for n in ("q", "k", "v", "g", "mu"))
    y = torch.empty_like(v)
    st = LizardState(Bl, wl.H, wl.dk, wl.dv, wl.w, dtype=q.dtype)

    def step():
        lizard_attn_prefill(q, k, v, g, mu, wl.alpha, wl.w, y=y, state=st, stream=stream)

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    with ClockSampler(local) as clocks:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ms = time_loop(step, args.steps, 0, stream)
        ms = max_over_ranks(ms, world)
        # one prefill kernel per step at this shape (B*H = 128 units: no
        # sequence segments), so the timed average is that kernel's duration
        launch_ms = ms

        # ---- decode (a10), same run ----
        dwl = DECODE_WL
        init = decode_initial_state(dwl, seed=rank_seed(dwl.seed, rank))
        dst = LizardState(dwl.B, dwl.H, dwl.dk, dwl.dv, dwl.w, dtype=torch.bfloat16)
        dst.S.copy_(init["S"])
        dst.ring_k.copy_(init["ring_k"])
        dst.ring_v.copy_(init["ring_v"])
        dst.pos.copy_(init["pos"])
        dmu = init["mu"].cuda()
        pool = [{n: t.cuda() for n, t in decode_step_inputs(dwl, s, seed=rank_seed(dwl.seed, rank)).items()}
                for s in range(8)]
        dy = torch.empty(dwl.B, dwl.H, dwl.dv, dtype=torch.bfloat16, device="cuda")
        ctr = [0]

        def dstep():
            p = pool[ctr[0] % len(pool)]
            ctr[0] += 1
            lizard_attn_decode_step(p["q"], p["k"], p["v"], p["g"], dmu, dwl.alpha, dst, y=dy, stream=stream)

        dsteps = max(args.steps, 64)
        dms = time_loop(dstep, dsteps, max(args.warmup, 3), stream)
        dms = max_over_ranks(dms, world)
        dlaunch_ms = dms  # one kernel per decode step: the timed average is its duration
        # The same steps alternating between two states (2 x 134 MB, above
        # L2): no step finds the state it updates left in L2 by the one before.
        dst2 = LizardState(dwl.B, dwl.H, dwl.dk, dwl.dv, dwl.w, dtype=torch.bfloat16)
        for n in ("S", "ring_k", "ring_v", "pos"):
            getattr(dst2, n).copy_(getattr(dst, n))
        states = (dst, dst2)

        def dstep2():
            p = pool[ctr[0] % len(pool)]
            st_ = states[ctr[0] % 2]
            ctr[0] += 1
            lizard_attn_decode_step(p["q"], p["k"], p["v"], p["g"], dmu, dwl.alpha, st_, y=dy, stream=stream)

        dms2 = max_over_ranks(time_loop(dstep2, dsteps, max(args.warmup, 3), stream), world)
        del dst2, states

        # ---- backward of the prefill (training), same run ----
        gen = torch.Generator().manual_seed(rank_seed(wl.seed + 11, rank))
        dy_b = torch.randn(q.shape, generator=gen).to(q.dtype).cuda()

        def bstep():
            lizard_attn_backward(q, k, v, g, mu, wl.alpha, wl.w, dy_b, stream=stream)

        bsteps = max(3, min(args.steps, 10))
        bms = max_over_ranks(time_loop(bstep, bsteps, max(args.warmup, 2), stream), world)

        # ---- gate projection of the same layer (x [B, L, 4096] -> g), same run ----
        dmodel = 4096
        proj = gate_projection_inputs(Bl, wl.L, dmodel, wl.H, wl.dk, seed=rank_seed(wl.seed + 23, rank))
        px, pw = proj["x"].cuda(), proj["W"].cuda()
        pg = torch.empty(Bl, wl.H, wl.L, wl.dk, dtype=torch.bfloat16, device="cuda")

        def pstep():
            lizard_gate_projection(px, pw, wl.H, g=pg, stream=stream)

        psteps = max(3, min(args.steps, 10))
        pms = max_over_ranks(time_loop(pstep, psteps, max(args.warmup, 2), stream), world)
        pflops = 2.0 * Bl * wl.L * wl.H * wl.dk * dmodel

        # ---- the decay-stress and long-context prefill workloads, same run ----
        extra, extra_bwd = {}, {}
        for name in ("decay_stress", "long_context", "d64"):
            xwl = WORKLOADS[name]
            xin = prefill_inputs(xwl, seed=rank_seed(xwl.seed, rank))
            xq, xk, xv, xg, xmu = (xin[n].cuda() for n in ("q", "k", "v", "g", "mu"))
            xy = torch.empty_like(xv)
            xst = LizardState(xwl.B, xwl.H, xwl.dk, xwl.dv, xwl.w, dtype=xq.dtype)

            def xstep():
                lizard_attn_prefill(xq, xk, xv, xg, xmu, xwl.alpha, xwl.w, y=xy, state=xst, stream=stream)

            xsteps = max(3, min(args.steps, 10))
            xms = max_over_ranks(time_loop(xstep, xsteps, max(args.warmup, 2), stream), world)
            extra[name] = (xwl, xms, xsteps)
            if name == "d64":  # its backward too (the tensor-core path on zero-padded tiles)
                xdy = torch.randn(xq.shape, generator=torch.Generator().manual_seed(rank_seed(xwl.seed + 11, rank)))
                xdy = xdy.to(xq.dtype).cuda()

                def xbstep():
                    lizard_attn_backward(xq, xk, xv, xg, xmu, xwl.alpha, xwl.w, xdy, stream=stream)

                xbms = max_over_ranks(time_loop(xbstep, xsteps, max(args.warmup, 2), stream), world)
                extra_bwd[name] = (xwl, xbms, xsteps)
                del xdy
            del xq, xk, xv, xg, xmu, xy, xst, xin
    lizard_check_device_status(stream)
    clock = clocks.summary()

    # ---- e2e through the public call with host buffers ----
    pinned = {n: inp_cpu[n].pin_memory() for n in ("q", "k", "v", "g", "mu")}
    y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    dq, dk_, dv_, dg, dmu2 = (torch.empty_like(t, device="cuda") for t in
                              (pinned["q"], pinned["k"], pinned["v"], pinned["g"], pinned["mu"]))
    # One call per sequence of the batch, pipelined over three streams: the
    # copy in of sequence b + 1 and the copy out of sequence b - 1 overlap
    # the prefill of sequence b (PCIe is full duplex).
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(Bl)]
    ev_done = [torch.cuda.Event() for _ in range(Bl)]
    st_b = [st.batch(b, b + 1) for b in range(Bl)]

    def e2e_step():
        s_in.wait_stream(stream)  # the previous step's calls have read their inputs
        with torch.cuda.stream(s_in):
            dmu2.copy_(pinned["mu"], non_blocking=True)
            for b in range(Bl):
                for dst, n in ((dq, "q"), (dk_, "k"), (dv_, "v"), (dg, "g")):
                    dst[b].copy_(pinned[n][b], non_blocking=True)
                ev_in[b].record(s_in)
        for b in range(Bl):
            stream.wait_event(ev_in[b])
            lizard_attn_prefill(dq[b:b + 1], dk_[b:b + 1], dv_[b:b + 1], dg[b:b + 1], dmu2, wl.alpha, wl.w,
                                y=y[b:b + 1], state=st_b[b], stream=stream)
            ev_done[b].record(stream)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                y_host[b].copy_(y[b], non_blocking=True)
        stream.wait_stream(s_out)  # the step ends when its last copy out has landed

    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms = max_over_ranks(time_loop(e2e_step, e2e_steps, 2, stream), world)
    h2d = sum(t.numel() * t.element_size() for t in pinned.values())
    d2h = y_host.numel() * y_host.element_size()

    tokens_rank = Bl * wl.L
    value = world * tokens_rank / (ms * 1e-3)
    nbytes = prefill_bytes(wl)
    nflops = prefill_flops(wl)
    achieved_gbs = nbytes / (launch_ms * 1e-3) / 1e9
    achieved_tfs = nflops / (launch_ms * 1e-3) / 1e12
    d_nbytes = decode_bytes(dwl)
    d_gbs = d_nbytes / (dlaunch_ms * 1e-3) / 1e9
    b_nbytes = backward_bytes(wl)
    b_gbs = b_nbytes / (bms * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1)-family tensors, no dataset)",
        "config": {"workload": workload_name(wl),
                   "also_timed": f"decode {dwl.B}x{dwl.H} d{dwl.dk} w{dwl.w} m{dwl.m}; backward and gate projection "
                                 f"of the same layer",
                   "global_batch": world * Bl, "seq_len": wl.L, "parallelism": f"dp{world} (independent sequences)",
                   "l2": "inputs larger than L2 (680 MB read/written per prefill step, 339 MB per decode step)"},
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved_gbs / peaks["hbm_gbs"], "peak_source": peak_src,
                     "traffic": ncu_traffic("prefill", PREFILL_KERNEL_SRC),
                     "kernel": "prefill", "launch_ms": launch_ms, "algorithmic_bytes": nbytes},
        "tensor": {"achieved_tflops": achieved_tfs, "peak_tflops": peaks["bf16_tflops"],
                   "frac": achieved_tfs / peaks["bf16_tflops"], "algorithmic_flops": nflops},
        "decode": {"value": world * dwl.B / (dms * 1e-3), "unit": "tokens/s", "ms_per_step": dms,
                   "steps": dsteps,
                   "roofline": {"bound": "hbm", "achieved": d_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": d_gbs / peaks["hbm_gbs"], "peak_source": peak_src,
                                "traffic": ncu_traffic("decode", DECODE_KERNEL_SRC),
                                "launch_ms": dlaunch_ms, "algorithmic_bytes": d_nbytes},
                   "rotating_states": {"ms_per_step": dms2, "value": world * dwl.B / (dms2 * 1e-3),
                                       "achieved_gbs": d_nbytes / (dms2 * 1e-3) / 1e9,
                                       "frac": d_nbytes / (dms2 * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                       "note": "two states in turn: no step reads a state left in L2"}},
        "backward": {"value": world * tokens_rank / (bms * 1e-3), "unit": "tokens/s", "ms_per_step": bms,
                     "steps": bsteps,
                     "train_value": world * tokens_rank / ((ms + bms) * 1e-3),
                     "train_unit": "tokens/s (prefill + backward)",
                     "roofline": {"bound": "hbm", "achieved": b_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": b_gbs / peaks["hbm_gbs"], "peak_source": peak_src,
                                  "traffic": ncu_traffic("backward", BACKWARD_KERNEL_SRC),
                                  "kernel": "backward call (chunk states, query side, key side)",
                                  "launch_ms": bms, "algorithmic_bytes": b_nbytes}},
        "gate_projection": {"value": world * tokens_rank / (pms * 1e-3), "unit": "tokens/s", "ms_per_step": pms,
                            "steps": psteps, "shape": f"x [{Bl}, {wl.L}, {dmodel}] x W^T [{dmodel}, {wl.H * wl.dk}]",
                            "roofline": {"bound": "tensor", "achieved": pflops / (pms * 1e-3) / 1e12,
                                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                         "frac": pflops / (pms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                                         "peak_source": peak_src, "traffic": None, "kernel": "gate_proj_kernel",
                                         "launch_ms": pms, "algorithmic_flops": pflops}},
        "prefill_workloads": {
            name: {"workload": f"{name} prefill B{xwl.B} H{xwl.H} L{xwl.L} d{xwl.dk} w{xwl.w} m{xwl.m} {xwl.dtype}",
                   "value": world * xwl.B * xwl.L / (xms * 1e-3), "unit": "tokens/s", "ms_per_step": xms,
                   "steps": xsteps,
                   "roofline": {"bound": "hbm", "achieved": prefill_bytes(xwl) / (xms * 1e-3) / 1e9,
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": prefill_bytes(xwl) / (xms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                "peak_source": peak_src, "traffic": None, "launch_ms": xms,
                                "algorithmic_bytes": prefill_bytes(xwl)},
                   "tensor_frac": prefill_flops(xwl) / (xms * 1e-3) / 1e12 / peaks["bf16_tflops"]}
            for name, (xwl, xms, xsteps) in extra.items()},
        "backward_workloads": {
            name: {"workload": f"{name} backward B{xwl.B} H{xwl.H} L{xwl.L} d{xwl.dk} w{xwl.w} m{xwl.m} {xwl.dtype}",
                   "value": world * xwl.B * xwl.L / (xms * 1e-3), "unit": "tokens/s", "ms_per_step": xms,
                   "steps": xsteps,
                   "roofline": {"bound": "hbm", "achieved": backward_bytes(xwl) / (xms * 1e-3) / 1e9,
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": backward_bytes(xwl) / (xms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                "peak_source": peak_src, "traffic": None, "launch_ms": xms,
                                "algorithmic_bytes": backward_bytes(xwl)}}
            for name, (xwl, xms, xsteps) in extra_bwd.items()},
        "e2e": {"value": world * tokens_rank / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": args.steps * 1,
        "clocks": clock,
    }

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        heads = wl.B * wl.H if args.sample_heads is None else args.sample_heads
        cv, cdt, cores, nunits = oracle_prefill_sample(inp_cpu, wl, heads)
        line["cpu_baseline"] = {"value": cv, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"{nunits} (batch, head) units of the same prefill workload, fp64, "
                                          f"{cdt:.1f} s; tokens/s counts whole-sequence positions"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_profile_case(args):
    """Launch one operator of one workload W + K times and print nothing else:
    the program that ncu captures on a small case.  ``--batch`` overrides the
    workload's batch (sequences)."""
    from hybrid_gated_linear_attn_b300 import LizardState, lizard_attn_decode_step, lizard_attn_prefill
    from hybrid_gated_linear_attn_b300 import lizard_attn_backward, lizard_check_device_status

    wl = WORKLOADS[args.workload]
    if args.batch:
        wl = wl.replace(B=args.batch)
    if args.seq_len:
        wl = wl.replace(L=args.seq_len)
    if args.profile_case == "prefill":
        inp = prefill_inputs(wl)
        q, k, v, g, mu = (inp[n].cuda() for n in ("q", "k", "v", "g", "mu"))
        y = torch.empty_like(v)
        st = LizardState(wl.B, wl.H, wl.dk, wl.dv, wl.w, dtype=q.dtype)
        fn = lambda: lizard_attn_prefill(q, k, v, g, mu, wl.alpha, wl.w, y=y, state=st)  # noqa: E731
    elif args.profile_case == "gate_projection":
        from hybrid_gated_linear_attn_b300 import lizard_gate_projection
        from hybrid_gated_linear_attn_b300.inputs import gate_projection_inputs
        proj = gate_projection_inputs(wl.B, wl.L, 4096, wl.H, wl.dk)
        px, pw = proj["x"].cuda(), proj["W"].cuda()
        pg = torch.empty(wl.B, wl.H, wl.L, wl.dk, dtype=torch.bfloat16, device="cuda")
        fn = lambda: lizard_gate_projection(px, pw, wl.H, g=pg)  # noqa: E731
    elif args.profile_case == "backward":
        inp = prefill_inputs(wl)
        q, k, v, g, mu = (inp[n].cuda() for n in ("q", "k", "v", "g", "mu"))
        dy = torch.randn(q.shape, generator=torch.Generator().manual_seed(wl.seed + 11)).to(q.dtype).cuda()
        fn = lambda: lizard_attn_backward(q, k, v, g, mu, wl.alpha, wl.w, dy)  # noqa: E731
    else:
        init = decode_initial_state(wl)
        st = LizardState(wl.B, wl.H, wl.dk, wl.dv, wl.w, dtype=torch_dtype(wl.dtype))
        for n in ("S", "ring_k", "ring_v", "pos"):
            getattr(st, n).copy_(init[n])
        mu = init["mu"].cuda()
        p = {n: t.cuda() for n, t in decode_step_inputs(wl, 0).items()}
        fn = lambda: lizard_attn_decode_step(p["q"], p["k"], p["v"], p["g"], mu, wl.alpha, st)  # noqa: E731
    for _ in range(args.warmup + args.steps):
        fn()
    lizard_check_device_status()
    torch.cuda.synchronize()
    return 0


def relaunch(n: int) -> int:
    """``--gpus N`` without a launcher: run this same script as N local ranks
    under torch.distributed.run (one process per GPU, rendezvous on
    127.0.0.1) and return its exit status; rank 0 prints the JSON line."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(sys.argv[0]), *sys.argv[1:]]
    return subprocess.call(cmd)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sample-heads", type=int, default=None,
                    help="(batch, head) units in the oracle's timed sample (default: the whole workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["prefill", "decode", "backward", "gate_projection"], default=None,
                    help="only launch this operator W + K times (a small program for ncu); no JSON line")
    ap.add_argument("--workload", default=None, help="workload of --profile-case (default: the bench's)")
    ap.add_argument("--batch", type=int, default=0, help="batch override for --profile-case")
    ap.add_argument("--seq-len", type=int, default=0, help="prompt length override for --profile-case prefill")
    args = ap.parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and not args.profile_case:
        return relaunch(args.gpus)
    world, rank, local = dist_setup()
    if not args.profile_case and world != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if args.profile_case:
        if args.workload is None:
            args.workload = "decode" if args.profile_case == "decode" else "llama3_8b"
        return run_profile_case(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    try:
        return run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
