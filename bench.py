#!/usr/bin/env python3
"""Benchmark: one functional MLP training step = one persistent-kernel launch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5] [--impl ours|reference]
                    [--stage-profile] [--launches-only]

Prints ONE JSON line for the headline workload (the GEMM-bound bf16 step, the
largest of the workloads; --config picks another).  `value` is whole-job
steps/s from the CUDA-event device time of exactly K single-step launches with
an L2 flush (a write of a buffer larger than L2) between them, outside the
events.  Beside it, for the headline and every other workload:
  * back_to_back: batches of launches on one stream with the state fed back
    (in-place updates), median of >= 5 batches;
  * graph: the same batches captured once as a CUDA graph and replayed,
    median of >= 5 replays (the pages time graph-captured steps);
  * clocks: nvidia-smi samples taken while that workload's timed loops ran.
`e2e` repeats the metric through the public API with host-resident batches
(tk_run_host): each step copies x (and y) from pinned host memory, overlapped
with the previous step on the library's copy stream, runs the step and reads
the loss back.  With N > 1 each rank runs an independent replica on its own
GPU (the step has no data-parallel exchange), times are max-reduced over ranks
and `value` sums the replicas.

--impl reference times the CPU oracle (the method's plain restatement) on the
host cores instead: each timed step evaluates a uniform random fraction of
every op's outputs, sized so the run stays within a few minutes, and the
throughput is scaled back to whole steps.

--stage-profile prints the per-stage timing of one step (work and grid-barrier
time per stage, from the kernel's %globaltimer stamps) instead.
--launches-only runs W + K launches of the workload and nothing else (for
profilers).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from persistent_step_megakernel_gb300 import synthetic as S  # noqa: E402

METRIC = "MLP train steps/sec (µs/step, device-timed) and % of roofline on 1 GB300"
UNIT = "steps/s"
L2_FLUSH_BYTES = 256 << 20           # > 129 MB L2
KERNEL = "tk_persistent"
HEADLINE = "c5"                      # the largest workload
DTYPE_TAG = {"float32": "f32", "bfloat16": "bf16", "float16": "f16"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def roofline(cfg, seconds, traffic):
    hbm, tflops, src = peaks()
    flops, nbytes = cfg.flops(), cfg.compulsory_bytes()
    t_mem = nbytes / (hbm * 1e9)
    # float32 GEMMs run on CUDA cores here; the tensor roofline applies to bf16/fp16
    t_tc = flops / (tflops * 1e12) if cfg.dtype != "float32" else 0.0
    if t_tc > t_mem:
        achieved = flops / seconds / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s",
                "frac": achieved / tflops, "traffic": traffic, "peak_source": src,
                "roofline_us": t_tc * 1e6}
    achieved = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": traffic, "peak_source": src, "roofline_us": t_mem * 1e6}


def kernel_source_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "persistent_step_megakernel_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(config_key: str):
    """DRAM bytes per launch from a committed ncu summary of the same kernel source."""
    path = os.path.join(ROOT, "profiles", f"{KERNEL}_{config_key}.md")
    if not os.path.exists(path):
        return None
    sha, traffic = None, None
    for line in open(path):
        if line.startswith("source_sha:"):
            sha = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = int(float(line.split(":", 1)[1].strip()))
    return traffic if sha == kernel_source_sha() else None


class Clocks:
    """nvidia-smi sampling while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        """Median SM clock over the samples taken while the GPU was busy (all
        samples when none reported utilisation), the maximum, and every
        throttle reason seen."""
        parsed = []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                clock, top = float(parts[0]), float(parts[1])
            except ValueError:
                continue
            try:
                util = float(parts[7])
            except ValueError:
                util = 0.0
            try:
                power = float(parts[2])
            except ValueError:
                power = None
            active = {n for n, v in zip(names, parts[3:7]) if v.lower().startswith("active")}
            parsed.append((clock, top, util, power, active))
        if not parsed:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_busy": 0}
        busy = [p for p in parsed if p[2] > 0]
        use = busy or parsed
        powers = [p[3] for p in use if p[3] is not None]
        return {"sm_mhz": statistics.median(p[0] for p in use), "sm_max_mhz": max(p[1] for p in use),
                "reasons": sorted(set().union(*(p[4] for p in parsed))), "samples": len(parsed),
                "samples_busy": len(busy), "power_w_max": max(powers) if powers else None}


def dist_setup(world: int, backend: str = "nccl"):
    """One process per GPU (torchrun's environment); None for a single process."""
    if world <= 1:
        return None
    import torch.distributed as dist
    dist.init_process_group(backend)
    return dist


def replica_value(us_per_step_max: float, world: int) -> float:
    """Whole-job steps/s of `world` independent replicas timed by the slowest rank."""
    return world * 1e6 / us_per_step_max


def allmax(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def device_inputs(cfg, prog, device):
    import numpy as np
    import torch
    arrays = S.mlp_inputs(cfg, prog)
    out = []
    for a, s in zip(arrays, prog.inputs):
        if s.dtype == "bfloat16":
            t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(a))
        out.append(t.to(device))
    return out


def input_bytes(cfg) -> int:
    prog = S.mlp_step_program(cfg, export="state")
    size = {"float32": 4, "float16": 2, "bfloat16": 2}
    total = 0
    for s in prog.inputs:
        n = 1
        for d in s.shape:
            n *= d
        total += n * size[s.dtype]
    return total


def batch_steps_for(cfg) -> int:
    """Steps per back-to-back batch: 100, or 20 for steps above a millisecond."""
    return 20 if cfg.flops() > 1e11 else 100


# Planner options of every program the bench builds (set from the command line).
OPTIONS = {}


def setup(cfg, device, **options):
    import torch
    from persistent_step_megakernel_gb300.runtime import TrainStep
    prog = S.mlp_step_program(cfg, export="state")
    step = TrainStep(prog, device.index, **{**OPTIONS, **options})
    ins = device_inputs(cfg, prog, device)
    outs, ws = step.allocate(ins)
    stream = torch.cuda.current_stream(device)
    return {"prog": prog, "step": step, "ins": ins, "outs": outs, "ws": ws, "stream": stream,
            "launch": step.launcher(ins, outs, ws, stream)}


def measure(cfg, device, dist, steps, warmup, batches, batch_steps, graph=True, clocks_gpu=None):
    """Device µs/step of the timed program three ways; the launches counted."""
    import torch
    ctx = setup(cfg, device)
    launch, stream = ctx["launch"], ctx["stream"]
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    for _ in range(warmup):
        launch()
        flush.zero_()
    torch.cuda.synchronize(device)
    ev = lambda: torch.cuda.Event(enable_timing=True)
    clocks = Clocks(clocks_gpu) if clocks_gpu is not None else None
    launches = 0
    barrier(dist)
    torch.cuda.synchronize(device)
    if clocks:
        clocks.__enter__()
    # 1. single steps, L2 flushed between them (the headline value)
    starts, ends = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    for k in range(steps):
        starts[k].record(stream)
        launch()
        ends[k].record(stream)
        flush.zero_()
    launches += steps
    torch.cuda.synchronize(device)
    flushed = [1e3 * s.elapsed_time(e) for s, e in zip(starts, ends)]
    # 2. back-to-back batches with the state fed back
    b2b = []
    for _ in range(batches):
        flush.zero_()
        a, b = ev(), ev()
        a.record(stream)
        for _ in range(batch_steps):
            launch()
        b.record(stream)
        launches += batch_steps
        torch.cuda.synchronize(device)
        b2b.append(1e3 * a.elapsed_time(b) / batch_steps)
    # 3. the batch captured as one CUDA graph, replayed
    graph_res = None
    if graph:
        graph_res = {}
        try:
            side = torch.cuda.Stream(device)
            side.wait_stream(stream)
            glaunch = ctx["step"].launcher(ctx["ins"], ctx["outs"], ctx["ws"], side)
            with torch.cuda.stream(side):
                glaunch()
            torch.cuda.synchronize(device)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                for _ in range(batch_steps):
                    glaunch()
            g.replay()
            torch.cuda.synchronize(device)
            reps = []
            for _ in range(batches):
                flush.zero_()
                a, b = ev(), ev()
                a.record(stream)
                g.replay()
                b.record(stream)
                launches += batch_steps
                torch.cuda.synchronize(device)
                reps.append(1e3 * a.elapsed_time(b) / batch_steps)
            graph_res = {"us_median": statistics.median(reps), "us_samples": reps, "steps_per_replay": batch_steps}
            del g
        except Exception as e:  # reported, not fatal: the other timings stand
            graph_res = {"error": f"{type(e).__name__}: {e}"[:300]}
    torch.cuda.synchronize(device)
    barrier(dist)
    if clocks:
        clocks.__exit__(None, None, None)
    status = ctx["step"].status(ctx["ws"])
    ctx.update({
        "status": status, "stats": ctx["step"].stats, "resources": ctx["step"].resource_usage(),
        "clocks": clocks.summary() if clocks else None, "launches": launches,
        "flushed": {"us_mean": statistics.mean(flushed), "us_median": statistics.median(flushed),
                    "us_min": min(flushed), "steps": steps},
        "back_to_back": {"us_median": statistics.median(b2b), "us_samples": b2b, "steps_per_batch": batch_steps},
        "graph": graph_res})
    return ctx


def time_e2e(ctx, steps, device):
    """Through the public API with host batches (tk_run_host): every step
    copies its x (and y) from page-locked host memory, on the library's copy
    stream while the previous step computes, runs the step and copies its
    loss back to host memory; the timed region ends when the last loss is on
    the host.  The batches alternate between two host copies."""
    import torch
    step, ins, outs, ws, prog = ctx["step"], ctx["ins"], ctx["outs"], ctx["ws"], ctx["prog"]
    names = [s.buffer for s in prog.inputs]
    batch = [names.index("x")] + ([names.index("y")] if "y" in names else [])
    host = [[ins[i].cpu().pin_memory() for i in batch] for _ in range(2)]
    alt = [torch.empty_like(ins[i]) for i in batch]
    loss_host = torch.empty((steps,) + tuple(outs[0].shape), dtype=outs[0].dtype).pin_memory()
    stream = torch.cuda.current_stream(device)
    h2d = sum(t.numel() * t.element_size() for t in host[0])
    d2h = outs[0].numel() * outs[0].element_size()

    def run(n):
        step.run_host(ins, outs, ws, batch, alt, [host[s & 1] for s in range(n)], [0],
                      [[loss_host[s]] for s in range(n)], stream=stream)
        stream.synchronize()

    run(3)
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    return steps / dt, h2d, d2h


# ------------------------------------------------------------ the oracle

def oracle_sampled(cfg, seconds: float, steps: int, warmup: int, seed: int = 0):
    """The oracle as it stands on a bounded sample of whole steps.

    Each sampled step evaluates, for every op, the same uniform random
    fraction of its outputs (at least one output); the operand buffers are
    primed with a constant (the timing of the oracle's loops does not depend on
    the values), so no full step has to run first.  Each op's time is scaled
    by its outputs / evaluated outputs, and the sum is one whole step.
    Returns (whole steps/s, fraction, threads)."""
    import numpy as np
    import oracle
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    o = oracle.Oracle(prog)
    o.set_inputs([S.storage_to_float64(a, s.dtype) for a, s in zip(arrays, prog.inputs)])
    have = {s.buffer for s in prog.inputs}
    for op in prog.operations:
        if op.output.buffer not in have:
            n = int(np.prod(op.output.shape)) if op.output.shape else 1
            o.set(op.output.buffer, np.full(n, 0.5))
            have.add(op.output.buffer)
    rng = np.random.default_rng(seed)
    sizes = [int(np.prod(op.output.shape)) if op.output.shape else 1 for op in prog.operations]

    def sampled_step(frac):
        """Seconds per op scaled to all of its outputs."""
        full = []
        for i, n in enumerate(sizes):
            k = max(1, int(round(frac * n)))
            idx = np.arange(n) if k >= n else np.sort(rng.choice(n, k, replace=False))
            t0 = time.perf_counter()
            o.eval_op_sampled(i, idx)
            full.append((time.perf_counter() - t0) * n / min(k, n))
        return sum(full)

    # calibrate on a small sample, then aim at `seconds` of sampled work in total
    frac = min(1.0, 64.0 / max(sizes))
    t0 = time.perf_counter()
    est = sampled_step(frac)
    while time.perf_counter() - t0 < 0.2 and frac < 1.0:
        frac = min(1.0, frac * 8)
        t0 = time.perf_counter()
        est = sampled_step(frac)
    frac = min(1.0, frac * seconds / max(1, steps + warmup) / max(1e-9, time.perf_counter() - t0))
    for _ in range(warmup):
        sampled_step(frac)
    whole = [sampled_step(frac) for _ in range(steps)]
    return 1.0 / statistics.mean(whole), frac, oracle.threads()


def cpu_baseline(cfg, seconds=15.0):
    value, frac, threads = oracle_sampled(cfg, seconds, steps=5, warmup=1)
    return {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"5 {cfg.key} steps, each evaluating a {frac:.3g} fraction of every op's outputs "
                      f"(uniform random indices, ~{seconds:.0f} s on the host cores); scaled to whole steps"}


def run_reference(args, rank, world):
    """The oracle on host cores as the reference arm (rank 0 only)."""
    if rank != 0:
        return 0
    cfg = S.CONFIGS[args.config]
    value, frac, threads = oracle_sampled(cfg, 90.0, args.steps, args.warmup)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_TAG[cfg.dtype],
            "data": "synthetic", "config": {"workload": cfg.description, "global_batch": cfg.batch * world,
                                            "dims": list(cfg.dims), "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"each step evaluates a {frac:.3g} fraction of every op's outputs "
                                       f"(uniform random indices, operands primed); throughput scaled to "
                                       f"whole steps"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------ modes

def stage_profile(cfg, device, warmup=5):
    """Per-stage work and barrier time of one step, with the L2 flushed before
    the step and warm (back to back), from the kernel's %globaltimer stamps."""
    import torch
    from persistent_step_megakernel_gb300.runtime import TrainStep
    prog = S.mlp_step_program(cfg, export="state")
    step = TrainStep(prog, device.index, profile=1, **OPTIONS)
    ins = device_inputs(cfg, prog, device)
    outs, ws = step.allocate(ins)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    per_stage = {}
    for t in step.tasks():
        per_stage.setdefault(t["stage"], []).append(
            f"{t['kind']}:{t['op'] or 'copy'}" + (f"[{t['m']}x{t['n']}x{t['k']}/{t['tile_n']}]" if t["m"] else ""))

    def timeline(best, s):
        """Median over the blocks with tensor-core tiles in stage s of the
        time from the stage's start to: the producer done, the first operand
        tile landed, the MMA issue done, the first accumulator ready, the
        epilogue's last store issued, the epilogue done (its stores complete),
        the barrier arrival (µs)."""
        rows = [r for r in best["stamps"][s] if r[3] > 0 and r[0] > 0]
        if not rows:
            return None
        med = lambda i: round(statistics.median((r[i] - r[0]) / 1e3 for r in rows), 2)
        return {"blocks": len(rows), "producer_done": med(2), "first_tile": med(3), "mma_done": med(4),
                "first_acc": med(5), "stores_issued": med(8), "epilogue_done": med(6), "arrive": med(1)}

    def run(flushed):
        runs = []
        for k in range(warmup + 3):
            if flushed:
                flush.zero_()
            step.run(ins, outs, ws)
            if flushed or k >= warmup:
                torch.cuda.synchronize(device)
            if k >= warmup:
                runs.append(step.profile(ws))
        best = min(runs, key=lambda r: r["total_us"])
        bars = best["barrier_us"]
        stages = [{"stage": s, "work_us": round(w, 2),
                   "barrier_us": round(bars[s], 2) if s < len(bars) else None,
                   "tasks": per_stage.get(s, []), "tc_timeline": timeline(best, s)}
                  for s, w in enumerate(best["work_us"])]
        return {"stages": stages, "total_us": best["total_us"], "prologue_us": best["prologue_us"],
                "barrier_us_median": statistics.median(bars) if bars else None,
                "barrier_us_max": max(bars) if bars else None}

    flushed = run(True)
    warm = run(False)
    return {"workload": cfg.description, "key": cfg.key, "grid_blocks": step.stats["grid_blocks"],
            "flushed": flushed, "warm": warm, "status": step.status(ws)}


def config_record(cfg, m):
    flushed_us = m["flushed"]["us_mean"]
    return {"us_per_step": flushed_us, "status": m["status"][0],
            "roofline": roofline(cfg, flushed_us * 1e-6, traffic_from_profiles(cfg.key)),
            "back_to_back_us": m["back_to_back"]["us_median"],
            "graph_us": (m["graph"] or {}).get("us_median"),
            "graph_error": (m["graph"] or {}).get("error"),
            "stages": m["stats"]["stages"], "grid_barriers": m["stats"]["grid_barriers"],
            "tensor_core_ops": m["stats"]["tensor_core_ops"],
            "steps": m["flushed"]["steps"], "clocks": m["clocks"], "gpu_launches": m["launches"]}


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=HEADLINE, choices=sorted(S.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batches", type=int, default=5, help="back-to-back batches and graph replays (>= 5)")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--stage-profile", action="store_true", help="print per-stage timing of one step")
    ap.add_argument("--launches-only", action="store_true", help="W + K launches and nothing else")
    ap.add_argument("--cta-pairs", type=int, choices=[0, 1, 2], default=None,
                    help="tensor-core GEMMs on pairs of SMs (1: cta_group::2 MMAs, 2: B shared by multicast) "
                         "or one SM per tile (0); default: the planner's")
    args = ap.parse_args()
    if args.cta_pairs is not None:
        OPTIONS["cta_pairs"] = args.cta_pairs
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch
    from persistent_step_megakernel_gb300.build import build
    if rank == 0 or world == 1:
        build()
    dist = dist_setup(world)
    if dist is not None:
        build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    cfg = S.CONFIGS[args.config]

    if args.launches_only:
        ctx = setup(cfg, device)
        for _ in range(args.warmup + args.steps):
            ctx["launch"]()
        torch.cuda.synchronize(device)
        status = ctx["step"].status(ctx["ws"])
        print(json.dumps({"launches": args.warmup + args.steps, "workload": cfg.key, "status": status}))
        return 0 if status[0] == 0 else 1
    if args.stage_profile:
        print(json.dumps(stage_profile(cfg, device)))
        return 0

    m = measure(cfg, device, dist, args.steps, args.warmup, max(5, args.batches), batch_steps_for(cfg),
                graph=not args.no_graph, clocks_gpu=local)
    if m["status"][0] != 0:
        raise SystemExit(f"device status {m['status']}")
    us = allmax(dist, m["flushed"]["us_mean"], device)
    e2e_value, h2d, d2h = time_e2e(m, min(args.steps, 300), device)
    e2e_value = world / allmax(dist, 1.0 / e2e_value, device)
    value = replica_value(us, world)
    in_mb = input_bytes(cfg) / 1e6
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": DTYPE_TAG[cfg.dtype], "data": "synthetic",
        "config": {"workload": cfg.description, "global_batch": cfg.batch * world, "dims": list(cfg.dims),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"flushed between timed steps (256 MiB write); inputs {in_mb:.1f} MB"},
        "us_per_step": {"mean": us, "median": m["flushed"]["us_median"], "min": m["flushed"]["us_min"],
                        "back_to_back_median": m["back_to_back"]["us_median"],
                        "graph_median": (m["graph"] or {}).get("us_median")},
        "back_to_back": m["back_to_back"], "graph": m["graph"],
        "roofline": roofline(cfg, us * 1e-6, traffic_from_profiles(cfg.key)),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": m["launches"],
        "kernel": KERNEL,
        "plan": {k: m["stats"][k] for k in ("stages", "grid_barriers", "grid_blocks", "fused_epilogues",
                                             "inlined_ops", "tensor_core_ops", "materialized_ops")},
        "resources": m["resources"],
        "clocks": m["clocks"],
    }
    del m
    if not args.no_others and rank == 0:
        others = {}
        for key, c in S.CONFIGS.items():
            if key == cfg.key:
                continue
            k = 100 if c.flops() > 1e11 else 300
            o = measure(c, device, None, k, 5, 5, batch_steps_for(c), graph=not args.no_graph, clocks_gpu=local)
            others[key] = config_record(c, o)
            del o
        line["other_configs"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
