#!/usr/bin/env python3
"""Benchmark of the split-backward MLP stage on GB300 (one JSON line).

A step is one replay of a stage's whole F/B/W op list over m microbatches
(every forward, input-gradient and weight-gradient pass, fp32 weight
gradients accumulated in microbatch order) with the inputs resident in HBM.

Default workload: one stage of a GPT-3-style block, h=6144, ffn=24576,
seq 3072, microbatch 1, bf16, m=24, replaying the stage-0 list of an 8-stage
ZB-H2 ordering (all W deferred into the warm-up/cool-down slots).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c4|c3|c2]
  python bench.py --sweep [--sweep-points 512x1024,...] [--sweep-m 32]

N > 1 runs N independent replicas (one per GPU, launched by torchrun): the
path has no exchange between GPUs, so "value" sums the replicas' work over
the slowest replica's time.  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload (host cores), the baseline arm.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "F/B/W TFLOP/s and stage tokens/sec on 1 GB300; % of dense BF16 tensor peak"
UNIT = "TFLOP/s"

WORKLOADS = {
    # name: (h, f, M, m, schedule, pipeline depth the list comes from, description)
    "c4": (6144, 24576, 3072, 24, "ZBH2", 8,
           "one stage h=6144 ffn=24576 seq 3072 microbatch 1 m=24, ZB-H2 stage-0 list of an "
           "8-stage pipeline, all W deferred, fp32 dW accumulate"),
    "c3": (4096, 16384, 3072, 16, "ZBH1", 8,
           "one stage h=4096 ffn=16384 seq 3072 microbatch 1 m=16, ZB-H1 stage-0 list of an "
           "8-stage pipeline, deferred W held in HBM"),
    "c2": (1024, 4096, 2048, 8, "ZBH1", 4,
           "P=4 stages h=1024 ffn=4096 microbatch 4x512 m=8, ZB-H1 replayed for all stages "
           "on one GPU"),
}


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm": d["hbm_gbs"], "bf16": d["bf16_tflops"],
                "bf16_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def _gemm_source_sha():
    h = hashlib.sha256()
    for n in ("gemm_tc.cu", "gemm_core.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "split_backward_gemms_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload):
    """DRAM bytes per GEMM of the workload's step mix, from the ncu
    figures committed as data under profiles/ (gemm_tc_<workload>.json),
    while they were taken on the current GEMM source; else None."""
    path = os.path.join(ROOT, "profiles", f"gemm_tc_{workload}.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        if d.get("source_sha") != _gemm_source_sha():
            return None
        return float(d["traffic_bytes_per_gemm"])
    except (OSError, KeyError, TypeError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def reduce_max(value: float, device, world_size: int) -> float:
    """Largest value over the ranks (the slowest replica's time)."""
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    if world_size > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_step: float, steps: int, world_size: int, seconds_max: float) -> float:
    """Whole-job throughput of independent replicas: every rank's work over
    the slowest rank's time."""
    return work_per_step * steps * world_size / seconds_max


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _cpu_sample(h, f, tokens, seed=0):
    """Seeded host inputs for the oracle sample (the same draw recipe)."""
    from split_backward_gemms_gb300 import inputs
    stages, X0, dY = inputs.pipeline_draws(1, 1, tokens, h, f, seed=seed)
    return stages[0], X0[0], dY[0]


def cpu_oracle_rate(h, f, tokens, repeats=1):
    """Time the fp64 oracle's F, B and W on a `tokens`-row slice; TFLOP/s."""
    import numpy as np

    from oracle import block as ob
    st, X, G = _cpu_sample(h, f, tokens)
    X, G, W1, W2 = (a.astype(np.float64) for a in (X, G, st.W1, st.W2))
    best = None
    for _ in range(repeats):
        t0 = time.perf_counter()
        H, A, _ = ob.forward(X, W1, W2)
        _, dH, _ = ob.backward_input(G, W1, W2, H)
        ob.backward_weight(X, A, dH, G)
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    flops = 12.0 * tokens * h * f
    return flops / best / 1e12, best


def run_reference(args, wl):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    h, f, M, m, sched, Pl, desc = WORKLOADS[wl]
    sched = args.schedule or sched
    tokens = 256
    from oracle import block as ob  # noqa: F401  (the oracle is the reference arm)
    import numpy as np
    st, X, G = _cpu_sample(h, f, tokens)
    X, G, W1, W2 = (a.astype(np.float64) for a in (X, G, st.W1, st.W2))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        H, A, _ = ob.forward(X, W1, W2)
        _, dH, _ = ob.backward_input(G, W1, W2, H)
        ob.backward_weight(X, A, dH, G)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    flops = 12.0 * tokens * h * f
    tot = sum(times)
    value = flops * len(times) / tot / 1e12
    cores = os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": desc, "h": h, "f": f, "M": M, "m": m, "schedule": sched},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"F+B+W of one microbatch's first {tokens} tokens at "
                                   f"h={h}, f={f} per step, fp64 numpy on host cores"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def pass_bytes(M, h, f):
    """Compulsory HBM bytes of one pass (each tensor read or written once;
    bf16 activations and weights, fp32 weight gradients read and written)."""
    F = 2 * (M * h + h * f + 2 * M * f) + 2 * (M * f + f * h + M * h)
    B = 2 * (M * h + f * h + M * f + M * f) + 2 * (M * f + h * f + M * h)
    W = 2 * (M * f + M * h) + 8 * f * h + 2 * (M * h + M * f) + 8 * h * f
    return {"F": F, "B": B, "W": W}


class SmClockReader:
    """SM clock read through NVML (libnvidia-ml, read-only queries), sampled
    every 5 ms by a thread while a sweep point's passes run."""

    def __init__(self, index: int = 0):
        import ctypes
        import threading
        self._threading = threading
        self.ok = False
        try:
            self.lib = ctypes.CDLL("libnvidia-ml.so.1")
            if self.lib.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                return
            self.mhz = ctypes.c_uint()
            self.ok = True
        except OSError:
            pass
        self.samples, self.thread, self.run = [], None, False

    def read(self):
        import ctypes
        if self.ok and self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(self.mhz)) == 0:
            return self.mhz.value
        return None

    def start(self):
        self.samples, self.run = [], True

        def loop():
            while self.run:
                v = self.read()
                if v is not None:
                    self.samples.append(v)
                time.sleep(0.005)
        if self.ok:
            self.thread = self._threading.Thread(target=loop, daemon=True)
            self.thread.start()

    def stop(self):
        self.run = False
        if self.thread is not None:
            self.thread.join()
        return statistics.median(self.samples) if self.samples else None


def run_sweep(args):
    """Per-pass kernel sweep: F, B and W standalone at each (M, h), f = 4h,
    W accumulating over m microbatches (4 distinct input sets, cycled)."""
    import torch

    from split_backward_gemms_gb300 import build as B
    B.build()
    from split_backward_gemms_gb300 import zb

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks = _peaks()
    stream = torch.cuda.current_stream()
    if args.sweep_points:
        points = [tuple(int(v) for v in p.split("x")) for p in args.sweep_points.split(",")]
    else:
        points = [(M, h) for M in (512, 2048, 8192, 16384) for h in (1024, 2048, 4096, 8192)]
    m, sets = args.sweep_m, 4
    for M, h in points:
        f = 4 * h
        gen = torch.Generator(device=dev).manual_seed(M * 31 + h)
        bf = torch.bfloat16
        W1 = (torch.randn(h, f, device=dev, generator=gen) * 0.02).to(bf)
        W2 = (torch.randn(f, h, device=dev, generator=gen) * 0.02).to(bf)
        dW1 = torch.zeros(h, f, device=dev)
        dW2 = torch.zeros(f, h, device=dev)
        b1 = (torch.randn(f, device=dev, generator=gen) * 0.02).to(bf) if args.bias else None
        b2 = (torch.randn(h, device=dev, generator=gen) * 0.02).to(bf) if args.bias else None
        db1 = torch.zeros(f, device=dev) if args.bias else None
        db2 = torch.zeros(h, device=dev) if args.bias else None
        blk = zb.make_block(M, h, f, has_bias=args.bias)
        S = []
        for _ in range(sets):
            t = {"X": torch.randn(M, h, device=dev, generator=gen).to(bf),
                 "dY": torch.randn(M, h, device=dev, generator=gen).to(bf),
                 "H": torch.empty(M, f, device=dev, dtype=bf), "A": torch.empty(M, f, device=dev, dtype=bf),
                 "Y": torch.empty(M, h, device=dev, dtype=bf), "dH": torch.empty(M, f, device=dev, dtype=bf),
                 "dX": torch.empty(M, h, device=dev, dtype=bf)}
            zb.zb_forward(blk, t["X"], W1, W2, b1, b2, t["H"], t["A"], t["Y"], stream)
            zb.zb_backward_input(blk, t["dY"], W1, W2, t["H"], t["dH"], t["dX"], stream)
            S.append(t)
        passes = {
            "F": lambda t, j: zb.zb_forward(blk, t["X"], W1, W2, b1, b2, t["H"], t["A"], t["Y"], stream),
            "B": lambda t, j: zb.zb_backward_input(blk, t["dY"], W1, W2, t["H"], t["dH"], t["dX"], stream),
            "W": lambda t, j: zb.zb_backward_weight(blk, t["X"], t["A"], t["dH"], t["dY"], dW1, dW2,
                                                    db1, db2, j > 0, stream),
        }
        pb = pass_bytes(M, h, f)
        clock = SmClockReader(torch.cuda.current_device())
        for name, fn in passes.items():
            for j in range(3):
                fn(S[j % sets], j)
            torch.cuda.synchronize()
            # each point is compared with the burst peak: let the previous
            # (possibly power-capped) point's clock recover first
            time.sleep(args.sweep_rest)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            clock.start()
            e0.record(stream)
            for j in range(m):
                fn(S[j % sets], j)
            e1.record(stream)
            torch.cuda.synchronize()
            sm_mhz = clock.stop()
            ms = e0.elapsed_time(e1) / m
            flops = 4.0 * M * h * f
            t_flop = flops / (peaks["bf16"] * 1e12)
            t_byte = pb[name] / (peaks["hbm"] * 1e9)
            bound = "tensor" if t_flop >= t_byte else "hbm"
            print(json.dumps({
                "sweep": True, "pass": name, "M": M, "h": h, "f": f, "microbatches": m, "bias": args.bias,
                "us_per_pass": 1e3 * ms, "tflops": flops / (ms / 1e3) / 1e12, "sm_mhz": sm_mhz,
                "gb_per_s": pb[name] / (ms / 1e3) / 1e9,
                "roofline": {"bound": bound, "time_us": 1e6 * max(t_flop, t_byte),
                             "frac": max(t_flop, t_byte) / (ms / 1e3),
                             "peak": peaks["bf16"] if bound == "tensor" else peaks["hbm"],
                             "unit": "TFLOP/s" if bound == "tensor" else "GB/s",
                             "peak_kind": "burst (%s)" % peaks["source"]},
            }), flush=True)
        zb.zb_sync_status(stream)
        del S, W1, W2, dW1, dW2
        torch.cuda.empty_cache()
    return 0


def measure_post_validated_adamw(zb, h, f, dev, stream, peaks, steps=5, warmup=3):
    """Post-update validation step of two pipeline stages, each holding one
    h x f block's weights (W1 and W2, fp32 master copies with AdamW moments and
    a bf16 weight copy).  max_norm sits between stage 0's partial gradient
    norm and the global one, so stage 0 steps, rolls back and steps again:
    the protocol's worst case.  HBM-bound: 30 bytes per element per pass
    (read theta, m, v, g; write theta, m, v, bf16 theta)."""
    import torch
    P = 2
    gen = torch.Generator(device=dev).manual_seed(77)
    n = h * f
    stages, tensors = [], []
    for s in range(P):
        st = []
        for _ in range(2):
            th = torch.randn(n, device=dev, generator=gen) * 0.02
            d = {"theta": th, "m": torch.zeros_like(th), "v": torch.zeros_like(th),
                 "grad": torch.randn(n, device=dev, generator=gen) * (1.0 + s),
                 "weight_bf16": th.to(torch.bfloat16), "stage": s}
            st.append(d)
            tensors.append(d)
        stages.append(st)
    nbytes = zb.zb_grad_stats_scratch_bytes()
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    states = [torch.zeros(2, dtype=torch.float64, device=dev) for _ in stages]

    def stats_all():
        for st, o in zip(stages, states):
            zb.zb_grad_stats([d["grad"] for d in st], [n, n], o, scratch, nbytes, stream)

    for _ in range(warmup):
        stats_all()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(steps):
        stats_all()
    g1.record(stream)
    torch.cuda.synchronize()
    stats_ms = g0.elapsed_time(g1) / steps
    stats_bytes = 4.0 * 2 * n * P  # every gradient element read once
    stats_gbs = stats_bytes / (stats_ms / 1e3) / 1e9
    sq = [float(o[0]) for o in states]
    c = (sq[0] * (sq[0] + sq[1])) ** 0.25  # geometric mean of the two partial norms
    dec = torch.empty(P * 40, dtype=torch.uint8, device=dev)
    hp = zb.make_adamw(max_norm=c, step=10)
    for _ in range(warmup):
        zb.zb_post_validated_adamw(P, states, tensors, hp, dec, stream)
    torch.cuda.synchronize()
    rolled = [d["rolled_back"] for d in zb.decisions_from_bytes(dec.cpu().numpy().tobytes(), P)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        zb.zb_post_validated_adamw(P, states, tensors, hp, dec, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    zb.zb_sync_status(stream)
    ms = e0.elapsed_time(e1) / steps
    elems = 2 * n * P + 2 * n * sum(rolled)
    algo = 30.0 * elems
    gbs = algo / (ms / 1e3) / 1e9
    return {"workload": f"post-validated AdamW, {P} stages x (W1, W2) of h={h} f={f} "
                        f"({2 * n / 1e6:.0f}M fp32 parameters per stage), stage 0 rolls back",
            "ms": ms, "rolled_back": rolled, "algorithmic_bytes": algo,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm"]},
            "launches_per_step": 3,
            "grad_stats": {"what": "sum of squares and NaN/Inf count of both stages' gradients "
                                   "(the staged-reduce inputs), 4 bytes per element",
                           "ms": stats_ms, "bytes": stats_bytes,
                           "roofline": {"bound": "hbm", "achieved": stats_gbs, "peak": peaks["hbm"],
                                        "unit": "GB/s", "frac": stats_gbs / peaks["hbm"]}}}


class Workload:
    """Device tensors, op list and executor plan of one benchmark workload."""


def make_ops(zb, sched, Pl, m, multi):
    """The op list a workload replays: the whole pipeline, or the stage-0
    list of a Pl-stage ordering replayed as one stage.  ZB1P / ZB2P are the
    heuristic scheduler's lists under p M_B and 2p M_B at equal pass times
    (this block's M_W = M_B, so the memory ratio is 1)."""
    if sched in ("ZB1P", "ZB2P"):
        limit = Pl if sched == "ZB1P" else 2 * Pl
        _, ops, _ = zb.zb_auto_schedule(Pl, m, 1.0, 1.0, 1.0, 0.0, limit, 1.0)
    else:
        ops = zb.zb_make_schedule(sched, Pl, m)
    if not multi:
        ops = [(k, 0, j) for k, s, j in ops if s == 0]
    return ops


def setup_workload(zb, dev, name, schedule=None, streams=0, seed=1000, executor="streams"):
    """Seeded synthetic weights (N(0, 0.02)), inputs and last-stage gradients
    (N(0, 1)) in HBM, the op list and a planned workspace."""
    import torch
    w = Workload()
    w.name = name
    w.h, w.f, w.M, w.m, sched, w.Pl, w.desc = WORKLOADS[name]
    w.sched = schedule or sched
    if w.sched != sched:
        w.desc += "; ordering replayed instead: " + w.sched
        if w.sched in ("ZBV", "1F1B-I"):
            w.desc += " (two chunks of one block per stage: 2P blocks)"
    w.multi = name == "c2"
    w.P = w.Pl if w.multi else 1
    # ZB-V / interleaved 1F1B: two chunks per stage, one MLP block each, so
    # the model is a chain of 2 P blocks (stage s holds two of them)
    w.chunks = 2 if w.sched in ("ZBV", "1F1B-I") else 1
    if w.chunks > 1 and not w.multi:
        raise ValueError("two-chunk orderings are replayed on the pipeline workload only")
    w.L = w.P * w.chunks
    h, f, M, m = w.h, w.f, w.M, w.m
    gen = torch.Generator(device=dev).manual_seed(seed)
    bf = torch.bfloat16
    w.W = [{"W1": (torch.randn(h, f, device=dev, generator=gen) * 0.02).to(bf),
            "W2": (torch.randn(f, h, device=dev, generator=gen) * 0.02).to(bf),
            "dW1": torch.zeros(h, f, device=dev), "dW2": torch.zeros(f, h, device=dev)}
           for _ in range(w.L)]
    w.X0 = [torch.randn(M, h, device=dev, generator=gen).to(bf) for _ in range(m)]
    w.dY = [torch.randn(M, h, device=dev, generator=gen).to(bf) for _ in range(m)]
    if w.chunks > 1:
        w.ops = zb.zb_make_interleaved_schedule(w.sched, w.Pl, w.chunks, m)
    else:
        w.ops = make_ops(zb, w.sched, w.Pl, m, w.multi)
    w.blk = zb.make_block(M, h, f)
    # multi-stage replays run each stage's F, B and W ops on lanes of their
    # own (3P streams; the P=4, h=1024 pipeline: 995 TF/s with a lane per
    # stage, 1008-1069 with a W lane too, 1089 with separate F and B lanes);
    # a one-stage replay puts its W passes on a second stream
    n_streams = streams if streams > 0 else (min(3 * w.P, 12) if w.multi else 2)
    w.executor = executor
    w.pl = zb.make_pipeline(w.P, m, w.blk, timing=True, streams=n_streams, chunks=w.chunks,
                            layout=w.sched if w.chunks > 1 else zb.ZB_LAYOUT_CYCLIC, executor=executor)
    w.need, w.peak_live = zb.zb_schedule_workspace_size(w.pl, w.ops)
    w.ws_t = torch.empty(max(w.need, 256), dtype=torch.uint8, device=dev)
    w.ops_c = zb.ops_array(w.ops)
    w.step_flops = 12.0 * M * h * f * m * w.L  # F, B and W: 4 M h f each per microbatch and block
    return w


def time_workload(zb, dev, w, steps, warmup, use_graph=True):
    """Warm-up replays, then `steps` replays of one captured CUDA graph
    between CUDA events on the launching stream (no per-op timing)."""
    import torch
    stream = torch.cuda.current_stream()
    st = zb.zb_run_stats()
    for _ in range(warmup):
        zb.zb_run_stage_schedule(w.pl, w.W, w.X0, w.dY, None, None, w.ops_c, w.ws_t, w.ws_t.numel(), st,
                                 stream)
    torch.cuda.synchronize()
    zb.zb_sync_status(stream)
    launches = st.n_gemm_launches
    w.pl.timing = 0
    graph = None
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                zb.zb_run_stage_schedule(w.pl, w.W, w.X0, w.dY, None, None, w.ops_c, w.ws_t,
                                         w.ws_t.numel(), None, side)
        stream.wait_stream(side)
        graph.replay()
        torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        if graph is not None:
            graph.replay()
        else:
            zb.zb_run_stage_schedule(w.pl, w.W, w.X0, w.dY, None, None, w.ops_c, w.ws_t, w.ws_t.numel(),
                                     None, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    zb.zb_sync_status(stream)
    ms = e0.elapsed_time(e1) / steps
    w.pl.timing = 1
    return {"ms_per_step": ms, "value": w.step_flops / (ms / 1e3) / 1e12,
            "tokens_per_s": w.m * w.M / (ms / 1e3),
            "gemm_launches_per_step": launches}


def other_workloads(zb, dev, steps, warmup):
    """The other configurations in the same run, each as its own short
    timed region: the P=4, h=1024 pipeline under 1F1B (fused backward), under
    ZB-H1 and ZB-H2 (split backward, W lanes), under the heuristic ZB-2p and
    the two-chunk orderings, same streams and graphs, and the h=4096
    one-stage ZB-H1 step; then the same pipeline orderings and the h=4096
    step with the persistent executor (one kernel per step).  A configuration
    that fails is reported with its error; the others and the main result
    stand."""
    import torch
    out = {}
    runs = [("c2", s, "streams") for s in ("1F1B", "ZBH1", "ZBH2", "ZB2P", "1F1B-I", "ZBV")] + [("c3", "ZBH1", "streams")]
    runs += [("c2", s, "persistent") for s in ("1F1B", "ZBH1", "ZBH2", "ZB2P", "1F1B-I", "ZBV")]
    runs += [("c3", "ZBH1", "persistent")]
    for name, sched, executor in runs:
        key = f"{name}_{sched}" + ("_persistent" if executor == "persistent" else "")
        try:
            w = setup_workload(zb, dev, name, sched, executor=executor)
            r = time_workload(zb, dev, w, steps, warmup)
        except Exception as exc:  # noqa: BLE001  (reported in the line; the main result stands)
            out[key] = {"schedule": sched, "executor": executor, "error": f"{type(exc).__name__}: {exc}"[:300]}
            torch.cuda.empty_cache()
            continue
        if w.chunks > 1:
            wl = ("P=4 stages x 2 chunks = 8 MLP blocks h=1024 ffn=4096, microbatch 4x512 m=8, all "
                  "stages on one GPU")
        elif name == "c2":
            wl = "P=4 stages h=1024 ffn=4096 microbatch 4x512 m=8, all stages on one GPU"
        else:
            wl = w.desc.split(",")[0]
        r.update({"workload": wl, "schedule": sched, "executor": executor, "unit": UNIT,
                  "pct_of_burst_peak": 100.0 * r["value"] / _peaks()["bf16"]})
        if executor == "streams":
            r["streams"] = w.pl.streams
        out[key] = r
        del w
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=tuple(WORKLOADS), default="c4")
    ap.add_argument("--schedule", choices=("1F1B", "ZBH1", "ZBH2", "ZB1P", "ZB2P", "ZBV", "1F1B-I"), default=None,
                    help="ordering to replay instead of the workload's own (c4: ZBH2, c3 and c2: ZBH1); "
                         "ZBV and 1F1B-I (c2 only) give each stage two chunks of one block each")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other configurations' short timed regions (the P=4, h=1024 "
                         "pipeline under 1F1B and ZB-H1, the h=4096 step)")
    ap.add_argument("--extra-steps", type=int, default=10, help="timed steps of each other configuration")
    ap.add_argument("--e2e-copies", choices=("one", "per-microbatch"), default="one",
                    help="e2e uploads: one copy per tensor kind of a contiguous [m, M, h] input set, "
                         "or one copy per microbatch tensor")
    ap.add_argument("--no-e2e-both", action="store_true",
                    help="measure e2e with the --e2e-result read-back only (default: both modes)")
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--e2e-mode", choices=("graph", "hybrid"), default="graph",
                    help="graph: one graph per step holds the step, the next step's upload and the "
                         "read-back; hybrid: a graph holds the step and read-back, the uploads are "
                         "issued from the host on a copy stream")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--executor", choices=("streams", "persistent"), default="streams",
                    help="streams: one launch per GEMM on stream lanes; persistent: every GEMM of the "
                         "step in one persistent kernel ordered on the device")
    ap.add_argument("--streams", type=int, default=0,
                    help="streams of the replay (0: an F, a B and a W lane per stage for a "
                         "pipeline, 3P <= 12; a one-stage replay puts its W passes on a second stream)")
    ap.add_argument("--e2e-result", choices=("stats", "dW"), default="stats",
                    help="what the e2e step reads back for the line's e2e value: the stages' "
                         "gradient statistics (sum of squares, NaN/Inf count; computed at the OPT "
                         "markers) or the full fp32 dW; the other mode is reported beside it")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step's kernels from the host instead of replaying one "
                         "captured CUDA graph per step")
    ap.add_argument("--no-optimizer", action="store_true",
                    help="skip the post-validated AdamW measurement (after the timed step)")
    ap.add_argument("--sweep", action="store_true",
                    help="per-pass kernel sweep (one JSON line per pass and point)")
    ap.add_argument("--sweep-points", default="",
                    help="comma list of MxH points, e.g. 3072x6144 (default: the M x h grid)")
    ap.add_argument("--sweep-m", type=int, default=32, help="microbatches timed per pass")
    ap.add_argument("--sweep-rest", type=float, default=0.5,
                    help="seconds of idle before each timed pass of the sweep (clock recovery)")
    ap.add_argument("--bias", action="store_true",
                    help="sweep with biases: F adds b1/b2, W also accumulates db1 = colsum dH, db2 = colsum dY")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args, args.workload)
    if args.sweep:
        return run_sweep(args)

    import torch
    import torch.distributed as dist

    ws, rank, local = _dist()
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", init_method="env://")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from split_backward_gemms_gb300 import build as B
    if rank == 0:
        B.build()
    if ws > 1:
        dist.barrier()
    from split_backward_gemms_gb300 import zb

    wk = setup_workload(zb, dev, args.workload, args.schedule, args.streams, seed=1000 + rank,
                        executor=args.executor)
    h, f, M, m, sched, Pl, desc = wk.h, wk.f, wk.M, wk.m, wk.sched, wk.Pl, wk.desc
    # P counts MLP blocks (stages x chunks): per-block work, weights, results
    multi, P, W, X0, dY = wk.multi, wk.L, wk.W, wk.X0, wk.dY
    blk, pl, need, peak_live, ws_t, ops_c = wk.blk, wk.pl, wk.need, wk.peak_live, wk.ws_t, wk.ops_c
    stream = torch.cuda.current_stream()

    def step(stats, pipe=None):
        zb.zb_run_stage_schedule(pipe or pl, W, X0, dY, None, None, ops_c, ws_t, ws_t.numel(), stats,
                                 stream)

    st = zb.zb_run_stats()
    for _ in range(args.warmup):
        step(st)
    torch.cuda.synchronize()
    zb.zb_sync_status(stream)
    def capture(Ws, Xs, Gs):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                zb.zb_run_stage_schedule(pl, Ws, Xs, Gs, None, None, ops_c, ws_t, ws_t.numel(), None, side)
        stream.wait_stream(side)
        return g

    graph = None
    if not args.no_graph:
        # the executor only enqueues work: one step captured on a side stream
        # (its helper streams and events exist already) replays as a graph
        launches_per_step = st.n_gemm_launches
        pl.timing = 0
        graph = capture(W, X0, dY)
        graph.replay()
        torch.cuda.synchronize()
        zb.zb_sync_status(stream)

    clocks = ClockSampler(torch.cuda.current_device())
    sums = {"gemm_ms": 0.0, "gemm_launches": 0, "kind": [0.0] * 4}
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
            sums["gemm_launches"] += launches_per_step
            continue
        step(st)
        sums["gemm_ms"] += st.gemm_ms
        sums["gemm_launches"] += st.n_gemm_launches
        for i in range(4):
            sums["kind"][i] += st.kind_ms[i]
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    zb.zb_sync_status(stream)
    ms_max = reduce_max(e0.elapsed_time(e1), dev, ws)

    flop_mb = 12.0 * M * h * f  # F, B and W: 4 M h f each per microbatch
    step_flops = flop_mb * m * P
    value = job_rate(step_flops, args.steps, ws, ms_max / 1e3) / 1e12
    tokens_s = job_rate(m * M, args.steps, ws, ms_max / 1e3)
    kind_ms, kind_steps = sums["kind"], args.steps
    kind_basis = "CUDA events around each op in the timed region"
    if pl.streams > 1 or graph is not None:
        # per-pass times from a short serial replay: on overlapping streams an
        # op's events also count the time it waited for SMs
        pl_serial = zb.make_pipeline(wk.P, m, blk, timing=True, streams=1, chunks=wk.chunks,
                                     layout=wk.sched if wk.chunks > 1 else zb.ZB_LAYOUT_CYCLIC)
        st_serial = zb.zb_run_stats()
        step(st_serial, pl_serial)
        kind_ms, kind_steps = [0.0] * 4, 2
        for _ in range(kind_steps):
            step(st_serial, pl_serial)
            for i in range(4):
                kind_ms[i] += st_serial.kind_ms[i]
        torch.cuda.synchronize()
        kind_basis = "serial replay after the timed region, CUDA events around each op"
    kind_tf = {}
    for i, name in enumerate(("F", "B", "W")):
        kms = kind_ms[i]
        kind_tf[name] = (4.0 * M * h * f * m * P * kind_steps / (kms / 1e3) / 1e12) if kms > 0 else None
    peaks = _peaks()
    # the rate per GEMM: 2 M h f flops each, six GEMMs per stage and
    # microbatch (a W pass's two run in one grouped launch, so GEMMs, not
    # launches, are counted here)
    gemm_flops = 2.0 * M * h * f
    gemms = 6 * m * P * args.steps
    avg_gemm_ms = sums["gemm_ms"] / max(1, gemms)
    overlapped = pl.streams > 1 or graph is not None
    if overlapped:
        # launches on different streams overlap (a W kernel starts in the
        # tail of an F/B kernel), so events around one launch also count the
        # time it waited for SMs: use the timed region's duration instead,
        # a lower bound on the kernel's own rate
        avg_gemm_ms = ms_max / max(1, gemms)
    achieved = gemm_flops / (avg_gemm_ms / 1e3) / 1e12
    roof_peak = peaks["bf16_sustained"]
    # the recorded traffic is the one-launch kernels' (stream executor)
    traffic = _profiled_traffic(args.workload) if args.executor == "streams" else None

    # ----------------------------------------------- projected P-stage pipeline
    # per-pass times measured above (executor CUDA events), fed to the
    # library's simulator of the orderings: a projection, not a measurement
    tfb = [kind_ms[i] / (m * P * kind_steps) for i in range(3)]
    projection = None
    if all(t > 0 for t in tfb) and not multi:  # concurrent stages blur per-pass times
        projection = {"label": "simulated %d-stage pipeline from the measured per-pass times" % Pl,
                      "P": Pl, "m": m, "T_F_ms": tfb[0], "T_B_ms": tfb[1], "T_W_ms": tfb[2],
                      "T_comm_ms": 0.0, "bubble_rate": {}, "pipeline_tokens_per_s": {}}
        for kind in ("1F1B", "ZBH1", "ZBH2"):
            res, _ = zb.zb_simulate_schedule(kind, Pl, m, tfb[0], tfb[1], tfb[2], 0.0)
            projection["bubble_rate"][kind] = res.bubble_rate
            projection["pipeline_tokens_per_s"][kind] = m * M / (res.cost / 1e3)
        # heuristic schedules under 1F1B-sized and doubled memory; this block's
        # B swaps H for dH, so M_W = M_B (mw_ratio 1)
        for name, limit in (("ZB-1p", Pl), ("ZB-2p", 2 * Pl)):
            res, _, _ = zb.zb_auto_schedule(Pl, m, tfb[0], tfb[1], tfb[2], 0.0, limit, 1.0)
            projection["bubble_rate"][name] = res.bubble_rate
            projection["pipeline_tokens_per_s"][name] = m * M / (res.cost / 1e3)
        # two chunks per stage (each half the stage's layers): cyclic 1F1B-I
        # and the V-shaped ZB-V; peak in M_B = peak chunk activations / 2
        projection["peak_M_B"] = {}
        for name, kind in (("1F1B-I", "1F1B-I"), ("ZB-V", "ZBV")):
            if kind == "1F1B-I" and m % Pl:
                continue
            res, _ = zb.zb_simulate_interleaved_schedule(kind, Pl, 2, m, tfb[0], tfb[1], tfb[2], 0.0)
            projection["bubble_rate"][name] = res.bubble_rate
            projection["pipeline_tokens_per_s"][name] = m * M / (res.cost / 1e3)
            projection["peak_M_B"][name] = res.peak_live_microbatches / 2
        projection["pinned"] = {
            "1F1B": "closed form (P-1)/(m+P-1) at any times",
            "ZBH1": "Table 2 at equal times and at T_W = T_F/2; a reading of the W placement otherwise",
            "ZBH2": "Table 2 at equal times and at T_W = T_F/2; a reading of the W placement otherwise",
            "ZB-1p": "Table 5's printed bubbles at Table 9's times; = ZB-H1 at equal times",
            "ZB-2p": "Table 5's printed bubbles at Table 9's times; = ZB-H2 at equal times",
            "1F1B-I": "closed form (P-1)/(vm+P-1) at equal times",
            "ZB-V": "ordering rule pinned only at equal times (zero bubble, peak p M_B); the value "
                    "at these unequal measured times comes from an unpinned reading"}

    # ------------------------------------------------------------- end to end
    # Through the public API with host buffers: every step uploads its inputs
    # from pinned host memory and reads back its result, in two modes: the
    # stages' gradient statistics (the per-step metric a training loop
    # reads; the weight gradients stay on the GPU for the optimizer) and the
    # full fp32 weight gradients.  Two input and gradient sets alternate so
    # that step k+1's upload and step k's read-back run on copy streams
    # while the other step computes.
    one_copy = args.e2e_copies == "one"
    if one_copy:
        # each input set is one [m, M, h] buffer per tensor kind, uploaded
        # with one copy each; the microbatches are views into it
        pin_all = torch.stack(X0).cpu().pin_memory()
        pin_g_all = torch.stack(dY).cpu().pin_memory()
        pin, pin_g = list(pin_all.unbind(0)), list(pin_g_all.unbind(0))
    else:
        pin = [x.cpu().pin_memory() for x in X0]
        pin_g = [g.cpu().pin_memory() for g in dY]
    h2d = sum(x.numel() * x.element_size() for x in pin + pin_g)
    up_stream = torch.cuda.Stream(device=dev)
    down_stream = torch.cuda.Stream(device=dev)
    pl.timing = 0

    def measure_e2e(want_dw):
        sets = []
        whole = []  # one_copy: the [m, M, h] device buffers of each set
        for a in range(2):
            if one_copy:
                xa = torch.empty((m,) + tuple(X0[0].shape), dtype=X0[0].dtype, device=dev)
                ga = torch.empty((m,) + tuple(dY[0].shape), dtype=dY[0].dtype, device=dev)
                xa.copy_(pin_all)
                ga.copy_(pin_g_all)
                whole.append((xa, ga))
                Xs_, Gs_ = list(xa.unbind(0)), list(ga.unbind(0))
            else:
                Xs_ = X0 if a == 0 else [torch.empty_like(x) for x in X0]
                Gs_ = dY if a == 0 else [torch.empty_like(g) for g in dY]
            Ws_ = [dict(w, dW1=torch.empty_like(w["dW1"]), dW2=torch.empty_like(w["dW2"])) for w in W]
            if not want_dw:
                for w in Ws_:
                    w["grad_stats"] = torch.zeros(2, dtype=torch.float64, device=dev)
            sets.append((Xs_, Gs_, Ws_))
        if want_dw:
            host_out = [(torch.empty(h, f, pin_memory=True), torch.empty(f, h, pin_memory=True))
                        for _ in range(P)]
            d2h = sum(a.numel() * 4 + b.numel() * 4 for a, b in host_out)
        else:
            host_out = [torch.empty(2, dtype=torch.float64, pin_memory=True) for _ in range(P)]
            d2h = 16 * P
        in_ready = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        down_done = [torch.cuda.Event(), torch.cuda.Event()]

        def copy_in(a):
            # this step's inputs from pinned host memory (on the current stream)
            if one_copy:
                whole[a][0].copy_(pin_all, non_blocking=True)
                whole[a][1].copy_(pin_g_all, non_blocking=True)
                return
            for j in range(m):
                sets[a][0][j].copy_(pin[j], non_blocking=True)
                sets[a][1][j].copy_(pin_g[j], non_blocking=True)

        def upload(a):
            # set a's inputs were last read by the step two back (done[a])
            up_stream.wait_event(done[a])
            with torch.cuda.stream(up_stream):
                copy_in(a)
                in_ready[a].record(up_stream)

        def read_back(Ws):
            for s_ in range(P):
                if want_dw:
                    host_out[s_][0].copy_(Ws[s_]["dW1"], non_blocking=True)
                    host_out[s_][1].copy_(Ws[s_]["dW2"], non_blocking=True)
                else:
                    host_out[s_].copy_(Ws[s_]["grad_stats"], non_blocking=True)

        def capture_e2e(a):
            # one graph per set: its step and, in parallel branches, the
            # upload of the other set's inputs (for the next step) and the
            # read-back of the other set's result (the previous step's,
            # complete when this graph starts); replays follow each other on
            # one stream, one host call per step.  The last step's result is
            # read back after the last replay (see e2e_run).
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    fork = torch.cuda.Event()
                    fork.record(side)
                    up_stream.wait_event(fork)
                    with torch.cuda.stream(up_stream):
                        copy_in(1 - a)
                        joined = torch.cuda.Event()
                        joined.record(up_stream)
                    down_stream.wait_event(fork)
                    with torch.cuda.stream(down_stream):
                        read_back(sets[1 - a][2])
                        down_joined = torch.cuda.Event()
                        down_joined.record(down_stream)
                    Xs_, Gs_, Ws_ = sets[a]
                    zb.zb_run_stage_schedule(pl, Ws_, Xs_, Gs_, None, None, ops_c, ws_t, ws_t.numel(), None,
                                             side)
                    side.wait_event(joined)
                    side.wait_event(down_joined)
            stream.wait_stream(side)
            return g

        def capture_step(a):
            # --e2e-mode hybrid: one graph per set holds its step and read-back;
            # the uploads are issued from the host on their own stream
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device=dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                with torch.cuda.graph(g, stream=side):
                    Xs_, Gs_, Ws_ = sets[a]
                    zb.zb_run_stage_schedule(pl, Ws_, Xs_, Gs_, None, None, ops_c, ws_t, ws_t.numel(), None,
                                             side)
                    read_back(Ws_)
            stream.wait_stream(side)
            return g

        step_gpu_ms = []
        hybrid = graph is not None and args.e2e_mode == "hybrid"
        e2e_graphs = [capture_e2e(0), capture_e2e(1)] if graph is not None and not hybrid else None
        step_graphs = [capture_step(0), capture_step(1)] if hybrid else None

        def e2e_run(steps):
            if step_graphs is not None:
                for ev in done:
                    ev.record(stream)
                upload(0)
                for k in range(steps):
                    a = k % 2
                    if k + 1 < steps:
                        upload(1 - a)  # overlaps this step's compute
                    stream.wait_event(in_ready[a])
                    step_graphs[a].replay()
                    done[a].record(stream)
                torch.cuda.synchronize()
                return
            if e2e_graphs is not None:
                # step 0's inputs, then each replay uploads the next step's;
                # events around each replay give its GPU time (diagnostic)
                marks = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
                with torch.cuda.stream(up_stream):
                    copy_in(0)
                stream.wait_stream(up_stream)
                marks[0].record(stream)
                for k in range(steps):
                    e2e_graphs[k % 2].replay()
                    marks[k + 1].record(stream)
                # the last step's result (the earlier ones were read back
                # inside the following step's graph)
                read_back(sets[(steps - 1) % 2][2])
                torch.cuda.synchronize()
                step_gpu_ms[:] = [marks[k].elapsed_time(marks[k + 1]) for k in range(steps)]
                return
            for ev in done + down_done:
                ev.record(stream)
            upload(0)
            for k in range(steps):
                a = k % 2
                if k + 1 < steps:
                    upload(1 - a)  # overlaps this step's compute
                stream.wait_event(in_ready[a])
                stream.wait_event(down_done[a])  # set a's gradients were downloaded
                Xs, Gs, Ws = sets[a]
                zb.zb_run_stage_schedule(pl, Ws, Xs, Gs, None, None, ops_c, ws_t, ws_t.numel(), None, stream)
                done[a].record(stream)
                down_stream.wait_event(done[a])
                with torch.cuda.stream(down_stream):
                    read_back(Ws)
                    down_done[a].record(down_stream)
            torch.cuda.synchronize()

        e2e_run(2)
        # the host link's rate for this step's inputs, alone (CUDA events on
        # the copy stream): an upload slower than a step makes e2e copy-bound
        torch.cuda.synchronize()
        u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        u0.record(up_stream)
        with torch.cuda.stream(up_stream):
            copy_in(0)
        u1.record(up_stream)
        torch.cuda.synchronize()
        upload_ms = u0.elapsed_time(u1)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e2e_clocks = ClockSampler(torch.cuda.current_device())
        e2e_clocks.start()
        time.sleep(0.3)
        t0 = time.perf_counter()
        e2e_run(args.e2e_steps)
        e2e_s = reduce_max(time.perf_counter() - t0, dev, ws)
        e2e_clk = e2e_clocks.stop()
        zb.zb_sync_status(stream)
        # graph mode reads back one result more than it runs steps (the first
        # graph's branch reads the other set's buffers before any step wrote
        # them): count every byte that crossed
        d2h_step = d2h * (args.e2e_steps + 1) / args.e2e_steps if e2e_graphs is not None else d2h
        return {"value": job_rate(step_flops, args.e2e_steps, ws, e2e_s) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h_step, "steps": args.e2e_steps,
                "upload_alone_ms": upload_ms, "h2d_gb_per_s": h2d / (upload_ms * 1e6),
                "mode": args.e2e_mode if graph is not None else "eager",
                "copies": args.e2e_copies,
                "clocks": e2e_clk,
                "step_gpu_ms": [round(x, 2) for x in step_gpu_ms] or None,
                "result": ("fp32 weight gradients" if want_dw else
                           "gradient statistics per stage (sum of squares, NaN/Inf count)"),
                "timing": ("host wall clock around the steps; per step one CUDA graph: the step, in "
                           "parallel branches the next step's upload and the previous step's read-back "
                           "(the last step's read-back after the last graph)"
                           if e2e_graphs is not None else
                           "host wall clock around the steps; per step one CUDA graph (the step, "
                           "the read-back), the next step's upload issued from the host on a "
                           "copy stream" if step_graphs is not None else
                           "host wall clock around synchronised steps; uploads and downloads "
                           "double-buffered on their own streams")}

    first = args.e2e_result
    e2e = measure_e2e(first == "dW")
    if not args.no_e2e_both:
        other = measure_e2e(first != "dW")
        e2e["other_result"] = {k: other[k] for k in ("value", "d2h_bytes_per_step", "result", "clocks")}

    optimizer = None
    if not args.no_optimizer:
        optimizer = measure_post_validated_adamw(zb, h, f, dev, stream, _peaks())

    extra = None
    if not args.no_extra and ws == 1:
        extra = other_workloads(zb, dev, args.extra_steps, args.warmup)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        tokens = 1024
        rate, secs = cpu_oracle_rate(h, f, tokens)
        cpu = {"value": rate, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"fp64 numpy F+B+W of one microbatch's first {tokens} tokens at h={h}, "
                         f"f={f} ({secs:.1f} s)"}

    # bytes one step touches: per stage W1, W2 (bf16) and dW1, dW2 (fp32,
    # read and written); per stage and microbatch X, dY, Y and dX (M x h)
    # and H, A and dH (M x f), all bf16
    wt_b = P * (2 * h * f * 2 + 2 * h * f * 4)
    act_b = P * m * (4 * M * h * 2 + 3 * M * f * 2)
    l2_b = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
    l2_note = ("inputs larger than L2: a step touches %.0f MB of weights and fp32 gradients and %.0f MB "
               "of activations, against %.0f MB of L2" % (wt_b / 1e6, act_b / 1e6, l2_b / 1e6))

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": desc, "h": h, "f": f, "M": M, "m": m, "P": wk.P, "chunks": wk.chunks,
                       "schedule": sched, "list_from_P": Pl, "streams": pl.streams, "executor": args.executor,
                       "cuda_graph": graph is not None,
                       "parallelism": "replicas" if ws > 1 else "single GPU",
                       "l2": l2_note},
            "tokens_per_s": tokens_s,
            "tflops": kind_tf, "tflops_basis": kind_basis,
            "pct_of_peak": {"burst": 100.0 * value / ws / peaks["bf16"],
                            "sustained": 100.0 * value / ws / peaks["bf16_sustained"]},
            "peak_live_bytes": peak_live, "workspace_bytes": need,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": roof_peak,
                         "unit": "TFLOP/s", "frac": achieved / roof_peak, "traffic": traffic,
                         "traffic_per": "GEMM (2 M h f flops; a grouped W launch is two)",
                         "kernel": "zb_gemm_bf16_tc_kernel (all six GEMMs of F/B/W)",
                         "launch_duration": ("timed region / GEMMs (streams overlap)" if overlapped
                                             else "CUDA events around each launch, per GEMM"),
                         "peak_kind": f"bf16_tflops_sustained ({peaks['source']})",
                         "frac_of_burst": achieved / peaks["bf16"]},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "projection": projection,
            "optimizer": optimizer,
            "other_configs": extra,
            "gpu_launches": sums["gemm_launches"],
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
