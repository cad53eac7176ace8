#!/usr/bin/env python3
"""Benchmark: one functional MLP training step = one persistent-kernel launch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c2] [--impl ours|reference]

Prints ONE JSON line.  `value` is whole-job steps/s from CUDA-event device time
of exactly K steps (an L2 flush -- a write of a buffer larger than L2 -- runs
between timed steps, outside the events).  `e2e` repeats the metric through the
public API with host-resident batches: each step copies x (and y) from pinned
host memory, runs the step and reads the loss back.  With N > 1 each rank runs
an independent replica on its own GPU (the step has no data-parallel exchange),
times are max-reduced over ranks and `value` sums the replicas.

--impl reference times the CPU oracle (the method's plain restatement) on the
host cores instead: each timed step evaluates a uniform random fraction of every
op's outputs, sized so the run stays within a few minutes, and the throughput
is scaled back to whole steps.
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
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None

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
        self.lines = []
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
                self.lines = [l for l in out.splitlines() if l.strip()]
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


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


def time_device(cfg, steps, warmup, device, dist, clocks_gpu=None):
    """Mean device µs/step over exactly `steps` launches, plus status and plan stats."""
    import torch
    from persistent_step_megakernel_gb300.runtime import TrainStep
    prog = S.mlp_step_program(cfg, export="state")
    step = TrainStep(prog, device.index)
    ins = device_inputs(cfg, prog, device)
    outs, ws = step.allocate(ins)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        step.run(ins, outs, ws)
        flush.zero_()
    torch.cuda.synchronize(device)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    clocks = Clocks(clocks_gpu) if clocks_gpu is not None else None
    barrier(dist)
    torch.cuda.synchronize(device)
    if clocks:
        clocks.__enter__()
    for k in range(steps):
        starts[k].record(stream)
        step.run(ins, outs, ws)
        ends[k].record(stream)
        flush.zero_()
    torch.cuda.synchronize(device)
    barrier(dist)
    if clocks:
        clocks.__exit__(None, None, None)
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    status = step.status(ws)
    return {"us_mean": 1e3 * sum(ms) / len(ms), "us_median": 1e3 * statistics.median(ms),
            "us_min": 1e3 * min(ms), "status": status, "stats": step.stats,
            "resources": step.resource_usage(), "clocks": clocks.summary() if clocks else None,
            "step": step, "ins": ins, "outs": outs, "ws": ws, "prog": prog}


def time_e2e(cfg, ctx, steps, device):
    """Through the public API with host batches: H2D x(,y) -> step -> D2H loss."""
    import torch
    step, ins, outs, ws, prog = ctx["step"], ctx["ins"], ctx["outs"], ctx["ws"], ctx["prog"]
    names = [s.buffer for s in prog.inputs]
    batch = [names.index("x")] + ([names.index("y")] if "y" in names else [])
    host = {i: ins[i].cpu().pin_memory() for i in batch}
    loss_host = torch.empty_like(outs[0], device="cpu").pin_memory()
    stream = torch.cuda.current_stream(device)
    h2d = sum(host[i].numel() * host[i].element_size() for i in batch)
    d2h = loss_host.numel() * loss_host.element_size()
    for _ in range(3):
        for i in batch:
            ins[i].copy_(host[i], non_blocking=True)
        step.run(ins, outs, ws)
        loss_host.copy_(outs[0], non_blocking=True)
        stream.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        for i in batch:
            ins[i].copy_(host[i], non_blocking=True)
        step.run(ins, outs, ws)
        loss_host.copy_(outs[0], non_blocking=True)
        stream.synchronize()
    dt = time.perf_counter() - t0
    return steps / dt, h2d, d2h


def oracle_steps_per_s(cfg, seconds=10.0):
    """The oracle as it stands, whole steps on the host cores, for ~`seconds`."""
    import oracle
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    vals = [S.storage_to_float64(a, s.dtype) for a, s in zip(arrays, prog.inputs)]
    o = oracle.Oracle(prog)
    o.set_inputs(vals)
    n, t0 = 0, time.perf_counter()
    while True:
        o.run()
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "sample": f"{n} whole {cfg.key} steps (all ops, all elements) in {dt:.1f} s on the host cores"}


def run_reference(args, rank, world):
    """The oracle on host cores as the reference arm (rank 0 only)."""
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    cfg = S.CONFIGS[args.config]
    prog = S.mlp_step_program(cfg, export="state")
    arrays = S.mlp_inputs(cfg, prog)
    o = oracle.Oracle(prog)
    o.set_inputs([S.storage_to_float64(a, s.dtype) for a, s in zip(arrays, prog.inputs)])
    t0 = time.perf_counter()
    o.run()                                    # one whole step: all buffers exist
    t_full = time.perf_counter() - t0
    budget = 90.0
    frac = min(1.0, budget / max(1e-9, (args.steps + args.warmup) * t_full))
    rng = np.random.default_rng(0)
    sizes = [int(np.prod(op.output.shape)) if op.output.shape else 1 for op in prog.operations]

    def sampled_step():
        for i, n in enumerate(sizes):
            k = max(1, int(round(frac * n)))
            idx = np.arange(n) if k >= n else rng.choice(n, k, replace=False)
            o.eval_op_sampled(i, idx)

    for _ in range(args.warmup):
        sampled_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sampled_step()
    dt = time.perf_counter() - t0
    value = frac * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": {"float32": "f32", "bfloat16": "bf16",
                                                                "float16": "f16"}[cfg.dtype],
            "data": "synthetic", "config": {"workload": cfg.description, "global_batch": cfg.batch * world,
                                            "dims": list(cfg.dims), "l2": "n/a (CPU)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
                             "sample": f"each step evaluates a {frac:.4f} fraction of every op's outputs "
                                       f"(uniform random indices); throughput scaled to whole steps"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=30)
    ap.add_argument("--config", default="c2", choices=sorted(S.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-others", action="store_true", help="skip the other configs' µs/step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
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

    r = time_device(cfg, args.steps, args.warmup, device, dist, clocks_gpu=local)
    if r["status"][0] != 0:
        raise SystemExit(f"device status {r['status']}")
    us = allmax(dist, r["us_mean"], device)
    e2e_value, h2d, d2h = time_e2e(cfg, r, min(args.steps, 500), device)
    e2e_value = allmax(dist, 1.0 / e2e_value, device)
    e2e_value = world / e2e_value
    value = replica_value(us, world)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": {"float32": "f32", "bfloat16": "bf16", "float16": "f16"}[cfg.dtype],
        "data": "synthetic",
        "config": {"workload": cfg.description, "global_batch": cfg.batch * world, "dims": list(cfg.dims),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between timed steps (256 MiB write)"},
        "us_per_step": {"mean": us, "median": r["us_median"], "min": r["us_min"]},
        "roofline": roofline(cfg, us * 1e-6, traffic_from_profiles(cfg.key)),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "kernel": KERNEL,
        "plan": {k: r["stats"][k] for k in ("stages", "grid_barriers", "grid_blocks", "fused_epilogues",
                                             "inlined_ops", "tensor_core_ops", "materialized_ops")},
        "resources": r["resources"],
        "clocks": r["clocks"],
    }
    line["us_per_barrier_upper_bound"] = us / max(1, r["stats"]["grid_barriers"])
    del r
    if not args.no_others and rank == 0:
        others = {}
        for key, c in S.CONFIGS.items():
            if key == cfg.key:
                continue
            k = 200 if c.flops() < 1e10 else 20
            o = time_device(c, k, 5, device, None)
            others[key] = {"us_per_step": o["us_mean"], "status": o["status"][0],
                           "roofline": roofline(c, o["us_mean"] * 1e-6, traffic_from_profiles(key)),
                           "stages": o["stats"]["stages"], "tensor_core_ops": o["stats"]["tensor_core_ops"],
                           "steps": k, "warmup": 5}
            del o
        line["other_configs"] = others
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_steps_per_s(cfg)
    if rank == 0:
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
