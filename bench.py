#!/usr/bin/env python3
"""Benchmark of the GB300 HSDP fully_shard data path.

One step = one pass of the whole hot path over one HSDP unit (all rank_size
virtual ranks on this GPU): all-gather copy-in fused with the all-gather,
all-gather copy-out, the fused ReduceScatter + AllReduce gradient sync, and
applying the averaged gradients to the actual shards. Default workload: the
large HSDP (2,8) mesh, one 70B-class GQA decoder layer (rank_size 16,
shard_size 8, 855,654,400 bf16 elements per rank).

Metric: achieved HBM GB/s = algorithmic bytes (what the method must read and
write; padding that must be written counts, padding that need not be read
does not) / device time. ``value`` is the whole step; ``kernels`` breaks it
down; ``roofline`` is the dominant kernel against the measured HBM peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

With N > 1 (torchrun), every GPU runs its own independent unit (weak
scaling, no data-path collective); rank 0 prints the line with the max time
over ranks. ``--impl reference`` times the CPU oracle on the host cores on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

KERNELS = ["ag_copy_in", "ag_copy_out", "rs_ar_reduce", "apply_grads"]
METRIC = "achieved HBM GB/s (and % of GB300 peak) for fused RS+AR grad-sync and AG copy-out"
L2_BYTES = 129 * 1024 * 1024
ES = {"f32": 4, "bf16": 2}


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="large_hsdp")
    ap.add_argument("--e2e-steps", type=int, default=3)
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the other workloads' step (reported under per_workload)")
    ap.add_argument("--per-workload-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--scale", type=float, default=1.0,
                    help="scale every dim 0 (small cases for profiler captures only)")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step replayed from a CUDA graph (launch-bound workloads)")
    ap.add_argument("--profile-kernel", default=None,
                    choices=["ag_copy_in", "ag_copy_out", "rs_ar_reduce", "apply_grads", "ag_unshard",
                             "rs_ar_reduce_apply"],
                    help="the small case of an ncu capture: only this kernel, --launches times, on the "
                         "workload scaled by --scale with only its buffers allocated (prints no bench line)")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--grid-limit", type=int, default=0,
                    help="with --profile-kernel: cap the kernel's blocks (fsdp_plan_set_grid_limit)")
    ap.add_argument("--pipeline", type=int, default=4, metavar="LAYERS",
                    help="also measure the pipelined backward over LAYERS layers of --pipeline-workload "
                         "(0: skip)")
    ap.add_argument("--pipeline-workload", default="hsdp_2x4_llama")
    ap.add_argument("--pipeline-large-layers", type=int, default=3,
                    help="also the fused syncs' pipeline over this many large (2,8) layers (0: skip)")
    return ap.parse_args(argv)


# --------------------------------------------------------------------------
# Distributed helpers (one process per GPU; gloo works for CPU tests)
# --------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def dist_init(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def dist_max(value, world, device="cpu"):
    """Max of a float over all ranks (the slowest rank sets the time)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_sum(value, world, device="cpu"):
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch
        import torch.distributed as dist

        if dist.get_backend() == "nccl":
            dist.barrier(device_ids=[torch.cuda.current_device()])
        else:
            dist.barrier()


def host_memory_bytes():
    try:
        return os.sysconf("SC_PHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        return 0


# --------------------------------------------------------------------------
# Bytes the method must move, per launch
# --------------------------------------------------------------------------

def algorithmic_bytes(sizes, param_dt, ag_dt, grad_dt):
    """sizes: dict with W, S, N (elements per rank), shard_total (sum over
    ranks and params of actual shard elements), slice_ag, slice_f32."""
    W, S, N = sizes["W"], sizes["S"], sizes["N"]
    st = sizes["shard_total"]
    bp, ba, bg = ES[param_dt], ES[ag_dt], ES[grad_dt]
    return {
        # read every rank's actual shards; write each rank's slice (data,
        # padding, tail) into all S shard-group members' buffers
        "ag_copy_in": st * bp + W * S * sizes["slice_ag"] * ba,
        # read and write every rank's full parameters (padding not read)
        "ag_copy_out": 2 * W * N * ba,
        # read every rank's full gradients once; write every rank's fused region
        "rs_ar_reduce": W * N * bg + W * sizes["slice_f32"] * 4,
        # read the actual fused elements; write the actual-shard gradients
        "apply_grads": st * 4 + st * bg,
    }


def unfused_bytes(sizes, param_dt, ag_dt, grad_dt):
    """Algorithmic bytes of the calls outside the timed step: the unfused
    forward (copy-in of the own slice, then the all-gather) and the unfused
    gradient sync (RS copy-in, shard-group ReduceScatter, replicate-group
    AllReduce in place, apply). sizes as for algorithmic_bytes plus
    slice_grad."""
    W, S, N, D = sizes["W"], sizes["S"], sizes["N"], sizes["W"] // sizes["S"]
    st = sizes["shard_total"]
    bp, ba, bg = ES[param_dt], ES[ag_dt], ES[grad_dt]
    sa, sg, sf = sizes["slice_ag"], sizes["slice_grad"], sizes["slice_f32"]
    return {
        "ag_copy_in_own_slice": st * bp + W * sa * ba,
        # every rank's own slice read once, written to the S-1 other members
        "ag_gather": (W * sa * ba + W * (S - 1) * sa * ba) if S > 1 else 0,
        # full gradients read (padding not read), whole RS input rows written
        "rs_copy_in": W * N * bg + W * S * sg * bg,
        "rs_reduce": W * S * sg * bg + W * sf * 4,
        "ar_reduce": 2 * W * sf * 4 if D > 1 else 0,
        "apply_grads": st * 4 + st * bg,
    }


def plan_sizes(plan):
    W, S, P = plan.W, plan.S, plan.P
    N = sum(plan.numel(p) for p in range(P))
    st = sum(plan.shard_numel(p, w % S) for w in range(W) for p in range(P))
    return {"W": W, "S": S, "N": N, "shard_total": st}


# --------------------------------------------------------------------------
# Clocks during the timed region
# --------------------------------------------------------------------------

CLOCK_FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
                "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                "clocks_event_reasons.sw_power_cap"]


class ClockSampler:
    def __init__(self, index):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(CLOCK_FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == len(CLOCK_FIELDS):
                rows.append(parts)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")

        sm = [num(r[0]) for r in rows]
        power = [num(r[2]) for r in rows]
        # samples under load: power above the midpoint of the observed range
        lo, hi = min(power), max(power)
        loaded = [s for s, p in zip(sm, power) if p >= lo + 0.5 * (hi - lo)] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(num(r[1]) for r in rows),
                "reasons": reasons, "samples": len(rows), "power_w_max": hi}


# --------------------------------------------------------------------------
# Oracle on the host: the CPU baseline and the reference arm
# --------------------------------------------------------------------------

def scaled_workload(wl, f):
    """The same mesh and parameter list with every dim 0 scaled by f."""
    d0 = [max(1, int(math.ceil(a * f))) for a in wl.d0]
    return d0, wl.inner


def oracle_step(L, wl, shards, grads):
    import oracle as O

    pdt, gdt = wl.param_dtype, wl.grad_dtype
    ag = O.ag_gather(L, O.ag_copy_in(L, shards, pdt, pdt), pdt)
    O.ag_copy_out(L, ag, pdt)
    fused = O.fused_from_grads(L, grads, gdt)
    O.apply_grads(L, fused, "avg", gdt)


def oracle_problem(wl, f):
    import oracle as O
    from hsdp_sharded_parameter_gb300 import workloads as WL

    d0, inner = scaled_workload(wl, f)
    L = O.Layout(d0, inner, wl.rank_size, wl.shard_size)
    shard_sizes = [L.shard_numel(p, w % L.S) for w in range(L.W) for p in range(L.P)]
    grad_sizes = [L.numel(p) for _ in range(L.W) for p in range(L.P)]
    shards = WL.np_tensors(shard_sizes, wl.seed_params, wl.param_std, wl.param_dtype)
    grads = WL.np_tensors(grad_sizes, wl.seed_grads, wl.grad_std, wl.grad_dtype)
    sizes = {"W": L.W, "S": L.S, "N": sum(grad_sizes) // L.W, "shard_total": sum(shard_sizes),
             "slice_ag": L.slice(wl.param_dtype), "slice_f32": L.slice("f32")}
    nbytes = sum(algorithmic_bytes(sizes, wl.param_dtype, wl.param_dtype, wl.grad_dtype).values())
    return L, shards, grads, nbytes, d0


def oracle_calibrate(wl, target_s):
    """Scale factor of the workload's dim 0 so one oracle step on the host
    takes about target_s seconds."""
    f = min(1.0, 2e5 / max(1, wl.numel_per_rank))
    L, shards, grads, nbytes, _ = oracle_problem(wl, f)
    t0 = time.perf_counter()
    oracle_step(L, wl, shards, grads)
    dt = max(time.perf_counter() - t0, 1e-4)
    return min(1.0, f * target_s / dt)


def cpu_baseline(wl, target_s):
    f = oracle_calibrate(wl, target_s)
    L, shards, grads, nbytes, d0 = oracle_problem(wl, f)
    t0 = time.perf_counter()
    oracle_step(L, wl, shards, grads)
    dt = time.perf_counter() - t0
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": (f"one full step (copy-in, gather, copy-out, RS copy-in + fused RS/AR sum, "
                       f"apply AVG) of the oracle on the same mesh and parameter list with every "
                       f"dim 0 scaled by {f:.3g} ({sum(a * b for a, b in zip(d0, wl.inner))} "
                       f"elements per rank, {nbytes / 1e9:.3f} GB algorithmic), single thread"),
            "_sample": (f, L, shards, grads, nbytes)}


def cpu_baseline_mt(wl, sample):
    """The same sample on every host core: the -fopenmp build of the oracle's
    source (loops over ranks, parameters and shard rows split across
    threads; every output byte equal to the oracle's). Reported beside the
    single-thread baseline, not a target."""
    import oracle as O
    from oracle import build as OB

    f, _, shards, grads, nbytes = sample
    try:
        OB.build(threaded=True)
    except Exception as e:  # no OpenMP in the host compiler
        return {"unavailable": f"no -fopenmp build of the oracle: {e}"}
    cores = os.cpu_count() or 1
    O.use_threaded(True)
    try:
        d0, inner = scaled_workload(wl, f)
        L = O.Layout(d0, inner, wl.rank_size, wl.shard_size)
        oracle_step(L, wl, shards, grads)  # warm the thread pool
        t0 = time.perf_counter()
        oracle_step(L, wl, shards, grads)
        dt = time.perf_counter() - t0
    finally:
        O.use_threaded(False)
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle source, -fopenmp build (same bytes as the oracle)", "seconds": round(dt, 3),
            "sample": f"the single-thread baseline's sample, {cores} threads"}


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if world > 1:
        dist_init(world, "gloo")
        barrier(world)
        if rank != 0:
            return 0
    per_step = max(0.2, 150.0 / max(1, args.steps + args.warmup))
    f = oracle_calibrate(wl, per_step)
    L, shards, grads, nbytes, d0 = oracle_problem(wl, f)
    for _ in range(args.warmup):
        oracle_step(L, wl, shards, grads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(L, wl, shards, grads)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = nbytes / dt / 1e9
    sample = (f"each step: the oracle's full step on the same mesh and parameter list with every "
              f"dim 0 scaled by {f:.3g} ({sum(a * b for a, b in zip(d0, wl.inner))} elements per "
              f"rank), single thread on the host")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.grad_dtype, "data": "synthetic",
            "config": {"workload": wl.key, "rank_size": wl.rank_size, "shard_size": wl.shard_size,
                       "elements_per_rank": wl.numel_per_rank, "sampled": True},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# The GPU arm
# --------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    return 6800.0, "fallback (6.8 TB/s)"


def kernel_source_hash():
    """sha256[:16] of the step kernels' source: fsdp_kernels.cu followed by
    the device helpers it includes (fsdp_device.cuh)."""
    import hashlib

    h = hashlib.sha256()
    for f in ("fsdp_kernels.cu", "fsdp_device.cuh"):
        h.update(open(os.path.join(ROOT, "hsdp_sharded_parameter_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (same source hash), else None."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    h = kernel_source_hash()
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[0] == h and parts[1] == kernel \
                and parts[2] == workload:
            return float(parts[3])
    return None


def run_gpu(args, wl):
    import torch

    from hsdp_sharded_parameter_gb300 import capi as C
    from hsdp_sharded_parameter_gb300 import workloads as WL
    from hsdp_sharded_parameter_gb300.runtime import HsdpUnit

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dev = torch.device("cuda", local)

    d0 = wl.d0 if args.scale == 1.0 else scaled_workload(wl, args.scale)[0]
    workload_name = wl.key if args.scale == 1.0 else f"{wl.key}@dim0x{args.scale:g}"
    plan = C.Plan(d0, wl.inner, wl.rank_size, wl.shard_size).upload()
    unit = HsdpUnit(plan, wl.param_dtype, wl.grad_dtype, device=dev, with_unfused=True)
    WL.torch_fill_(unit.shards, wl.seed_params, wl.param_std, wl.param_dtype)
    WL.torch_fill_(unit.grads, wl.seed_grads, wl.grad_std, wl.grad_dtype)
    sizes = plan_sizes(plan)
    sizes["slice_ag"] = plan.slice_numel(wl.param_dtype)
    sizes["slice_f32"] = plan.slice_numel("f32")
    sizes["slice_grad"] = plan.slice_numel(wl.grad_dtype)
    kb = algorithmic_bytes(sizes, wl.param_dtype, wl.param_dtype, wl.grad_dtype)
    step_bytes = sum(kb.values())
    working_set = step_bytes  # every byte of the step is a distinct HBM location
    flush = working_set < 4 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    calls = [lambda: unit.ag_copy_in(fuse_gather=True), unit.ag_copy_out, unit.rs_ar_reduce,
             lambda: unit.apply_grads("avg")]
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        for c in calls:
            c()
        if flush:
            scratch.zero_()
    torch.cuda.synchronize()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    l0 = C.fsdp_launch_count()
    t_start.record(stream)
    for k in range(K):
        if flush:
            scratch.zero_()
        ev[k][0].record(stream)
        for i, c in enumerate(calls):
            c()
            ev[k][i + 1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    launches = C.fsdp_launch_count() - l0
    clk = clocks.stop()

    per_kernel = {n: [ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K)] for i, n in enumerate(KERNELS)}
    step_ms = [ev[k][0].elapsed_time(ev[k][len(calls)]) for k in range(K)]
    total_ms = t_start.elapsed_time(t_end) if not flush else sum(step_ms)
    my_ms = total_ms / K
    ms = dist_max(my_ms, world, dev)
    value = dist_sum(step_bytes, world, dev) / (ms * 1e-3) / 1e9
    peak, peak_src = measured_peaks()
    kernels = {}
    for n in KERNELS:
        avg = sum(per_kernel[n]) / K
        gbs = kb[n] / (avg * 1e-3) / 1e9
        kernels[n] = {"us": round(avg * 1e3, 2), "median_us": round(statistics.median(per_kernel[n]) * 1e3, 2),
                      "bytes": kb[n], "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
    dom = max(KERNELS, key=lambda n: kernels[n]["us"])
    roofline = {"bound": "hbm", "kernel": dom, "achieved": kernels[dom]["gbs"], "peak": peak,
                "unit": "GB/s", "frac": kernels[dom]["frac"], "traffic": ncu_traffic(dom, workload_name),
                "peak_source": peak_src}
    second = "rs_ar_reduce" if dom != "rs_ar_reduce" else "ag_copy_out"
    roofline_2 = {"bound": "hbm", "kernel": second, "achieved": kernels[second]["gbs"], "peak": peak,
                  "unit": "GB/s", "frac": kernels[second]["frac"], "traffic": ncu_traffic(second, workload_name)}

    # Not part of the step, each call timed alone on the same unit: the
    # direct unshard (all three forward steps in one pass, no gathered
    # buffer: it reads each shard once and writes it into every shard-group
    # member's full parameter), and the unfused calls (the own-slice copy-in
    # and the all-gather of the forward; RS copy-in, ReduceScatter, in-place
    # AllReduce and apply of the pages' unfused gradient sync).
    ku = max(3, K // 4)

    def per_launch_us(fn):
        ev_u = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        if flush:  # time each launch alone, the L2 flush outside the events
            ms_u = 0.0
            for _ in range(ku):
                scratch.zero_()
                ev_u[0].record(stream)
                fn()
                ev_u[1].record(stream)
                torch.cuda.synchronize()
                ms_u += ev_u[0].elapsed_time(ev_u[1])
        else:
            ev_u[0].record(stream)
            for _ in range(ku):
                fn()
            ev_u[1].record(stream)
            torch.cuda.synchronize()
            ms_u = ev_u[0].elapsed_time(ev_u[1])
        return ms_u / ku * 1e3

    def entry(us, nbytes):
        gbs = nbytes / (us * 1e-6) / 1e9 if us > 0 else 0.0
        return {"us": round(us, 2), "bytes": nbytes, "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}

    extra = {}
    ub = sizes["shard_total"] * ES[wl.param_dtype] + sizes["W"] * sizes["N"] * ES[wl.param_dtype]
    extra["ag_unshard"] = entry(per_launch_us(unit.unshard_direct), ub)
    extra["ag_unshard"]["replaces_us"] = round(kernels["ag_copy_in"]["us"] + kernels["ag_copy_out"]["us"], 2)
    # the gradient sync in one pass (fused reduce with the apply folded in):
    # reads every gradient once, writes the fused regions and the shard
    # gradients; the apply's read of the fused regions is gone
    ob = sizes["W"] * sizes["N"] * ES[wl.grad_dtype] + sizes["W"] * sizes["slice_f32"] * 4 \
        + sizes["shard_total"] * ES[wl.grad_dtype]
    extra["rs_ar_reduce_apply"] = entry(per_launch_us(lambda: unit.reduce_grads_one_pass("avg")), ob)
    extra["rs_ar_reduce_apply"]["replaces_us"] = round(kernels["rs_ar_reduce"]["us"] + kernels["apply_grads"]["us"], 2)
    ubytes = unfused_bytes(sizes, wl.param_dtype, wl.param_dtype, wl.grad_dtype)
    unfused_calls = {
        "ag_copy_in_own_slice": lambda: unit.ag_copy_in(fuse_gather=False),
        "ag_gather": unit.ag_gather,
        "rs_copy_in": lambda: C.fsdp_rs_copy_in(plan, unit.b_grads, unit.b_rs_in),
        "rs_reduce": lambda: C.fsdp_rs_reduce(plan, unit.b_rs_in, "avg", unit.b_fused),
        "ar_reduce": lambda: C.fsdp_ar_reduce(plan, unit.b_fused, "avg"),
    }
    unfused = {n: entry(per_launch_us(fn), ubytes[n]) for n, fn in unfused_calls.items()}
    sync_us = sum(unfused[n]["us"] for n in ["rs_copy_in", "rs_reduce", "ar_reduce"]) + kernels["apply_grads"]["us"]
    unfused["sync_total"] = {"us": round(sync_us, 2),
                             "replaces_us": round(kernels["rs_ar_reduce"]["us"] + kernels["apply_grads"]["us"], 2),
                             "note": "RS copy-in + ReduceScatter + AllReduce + apply (SUM after the collectives' AVG)"}
    extra["unfused"] = unfused

    if args.graph:
        graph = unit.capture_step()
        ev_g = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ms_g = 0.0
        for _ in range(ku):
            if flush:
                scratch.zero_()
            ev_g[0].record(stream)
            graph.replay()
            ev_g[1].record(stream)
            torch.cuda.synchronize()
            ms_g += ev_g[0].elapsed_time(ev_g[1])
        extra["graph_step"] = {"us": round(ms_g / ku * 1e3, 2),
                               "eager_us": round(sum(kernels[n]["us"] for n in KERNELS), 2)}
        del graph

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, unit, calls, step_bytes, world, dev)

    per_workload = None
    want_per = not args.no_per_workload and args.scale == 1.0 and wl.key == "large_hsdp"
    want_pipe = args.pipeline > 0 and args.scale == 1.0
    if want_pipe or want_per:
        unit.close()
        del unit
        torch.cuda.empty_cache()
    if want_per:
        per_workload = run_per_workload(args, dev, peak)

    pipeline = None
    if want_pipe:
        pipeline = run_pipeline(args, dev, args.pipeline_workload, args.pipeline)
        if args.pipeline_large_layers > 0 and args.pipeline_workload != "large_hsdp":
            pipeline["large_hsdp"] = run_pipeline(args, dev, "large_hsdp", args.pipeline_large_layers,
                                                  ("one_pass", "fused"))

    cpu = cpu_mt = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)
        cpu_mt = cpu_baseline_mt(wl, cpu.pop("_sample"))

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
                "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": wl.grad_dtype, "data": "synthetic",
                "config": {"workload": workload_name, "rank_size": wl.rank_size,
                           "shard_size": wl.shard_size, "dp_size": plan.D, "params": wl.n_params, "elements_per_rank": sizes["N"],
                           "step_bytes": step_bytes,
                           "l2": ("flushed between steps (2x L2 scratch write, outside the step events)"
                                  if flush else "inputs larger than L2 (working set "
                                  f"{working_set / 1e9:.1f} GB >> 129 MB)"),
                           "parallelism": f"{world} independent unit(s), one per GPU"},
                "kernels": kernels, "kernels_outside_step": extra,
                "roofline": roofline, "roofline_second": roofline_2,
                "clocks": clk, "e2e": e2e, "cpu_baseline": cpu, "cpu_baseline_mt": cpu_mt,
                "gpu_launches": launches}
        if per_workload:
            line["per_workload"] = per_workload
        if pipeline:
            line["pipeline"] = pipeline
        print(json.dumps(line), flush=True)
    if not (want_pipe or want_per):
        unit.close()
    return 0


PER_WORKLOADS = ["hsdp_2x4_llama", "ragged_fsdp", "pure_tp_compat"]


def run_per_workload(args, dev, peak):
    """The same step on the other full-size workloads (HSDP (2,4) Llama
    layer, ragged-heavy FSDP, pure-TP compat), each on its own unit after the
    headline workload's unit is freed: per kernel µs, algorithmic GB/s and
    fraction of the measured peak, and the step's GB/s, with the clocks seen
    while they ran. W warm-up steps, then K timed steps; workloads smaller
    than 4x L2 flush it between steps, outside the step's events."""
    import torch

    from hsdp_sharded_parameter_gb300 import capi as C
    from hsdp_sharded_parameter_gb300 import workloads as WL
    from hsdp_sharded_parameter_gb300.runtime import HsdpUnit

    K = max(1, args.per_workload_steps)
    stream = torch.cuda.current_stream()
    out = {}
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    for key in PER_WORKLOADS:
        wl = WL.WORKLOADS[key]
        plan = C.Plan(wl.d0, wl.inner, wl.rank_size, wl.shard_size).upload()
        unit = HsdpUnit(plan, wl.param_dtype, wl.grad_dtype, device=dev)
        WL.torch_fill_(unit.shards, wl.seed_params, wl.param_std, wl.param_dtype)
        WL.torch_fill_(unit.grads, wl.seed_grads, wl.grad_std, wl.grad_dtype)
        sizes = plan_sizes(plan)
        sizes["slice_ag"] = plan.slice_numel(wl.param_dtype)
        sizes["slice_f32"] = plan.slice_numel("f32")
        kb = algorithmic_bytes(sizes, wl.param_dtype, wl.param_dtype, wl.grad_dtype)
        step_bytes = sum(kb.values())
        flush = step_bytes < 4 * L2_BYTES
        scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None
        calls = [lambda: unit.ag_copy_in(fuse_gather=True), unit.ag_copy_out, unit.rs_ar_reduce,
                 lambda: unit.apply_grads("avg")]
        for _ in range(max(3, args.warmup)):
            for c in calls:
                c()
        torch.cuda.synchronize()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(K)]
        for k in range(K):
            if flush:
                scratch.zero_()
            ev[k][0].record(stream)
            for i, c in enumerate(calls):
                c()
                ev[k][i + 1].record(stream)
        torch.cuda.synchronize()
        kernels = {}
        for i, n in enumerate(KERNELS):
            us = sum(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K)) / K * 1e3
            gbs = kb[n] / (us * 1e-6) / 1e9
            kernels[n] = {"us": round(us, 2), "bytes": kb[n], "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
        step_us = sum(ev[k][0].elapsed_time(ev[k][len(calls)]) for k in range(K)) / K * 1e3
        # the gradient sync in one pass (outside the step), back to back
        ob = sizes["W"] * sizes["N"] * ES[wl.grad_dtype] + sizes["W"] * sizes["slice_f32"] * 4 \
            + sizes["shard_total"] * ES[wl.grad_dtype]
        for _ in range(3):
            unit.reduce_grads_one_pass("avg")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            if flush:
                scratch.zero_()
            unit.reduce_grads_one_pass("avg")
        e1.record(stream)
        torch.cuda.synchronize()
        one_us = e0.elapsed_time(e1) / K * 1e3
        one = {"us": round(one_us, 2), "bytes": ob, "gbs": round(ob / (one_us * 1e-6) / 1e9, 1),
               "frac": round(ob / (one_us * 1e-6) / 1e9 / peak, 4),
               "replaces_us": round(kernels["rs_ar_reduce"]["us"] + kernels["apply_grads"]["us"], 2)}
        out[key] = {"rank_size": wl.rank_size, "shard_size": wl.shard_size, "params": wl.n_params,
                    "elements_per_rank": sizes["N"], "steps": K, "step_us": round(step_us, 2),
                    "step_bytes": step_bytes, "step_gbs": round(step_bytes / (step_us * 1e-6) / 1e9, 1),
                    "l2": "flushed between steps" if flush else "working set larger than L2",
                    "kernels": kernels, "rs_ar_reduce_apply": one}
        unit.close()
        plan.close()
        del unit, scratch
        torch.cuda.empty_cache()
    out["clocks"] = clocks.stop()
    return out


def run_pipeline(args, dev, workload, n, modes=("one_pass", "fused", "unfused_4step")):
    """Overlap of the gradient sync with backward compute over a stack of
    layers ("Hyper通信掩盖方案" PR #758 write-up §二.2: the 4-step pipeline):
    the stand-in backward of a layer is bf16 GEMMs (8192^3, cuBLAS) on the
    compute stream, as many as take about one layer's sync; the sync runs
    as the pages' unfused 4-step schedule, as the fused reduce (+ apply at
    the root), or as the one-pass fused sync per layer. Each is timed alone
    (whole GPU), serially after the compute, and pipelined with its kernels
    capped at `cap` blocks while compute runs beside them (one block per SM,
    on the high-priority sync streams; cap 0 = the whole-GPU kernels).
    hidden = (compute + sync - pipelined) / min(compute, sync)."""
    import torch

    from hsdp_sharded_parameter_gb300 import capi as C
    from hsdp_sharded_parameter_gb300 import workloads as WL
    from hsdp_sharded_parameter_gb300.runtime import BackwardPipeline, HsdpUnit

    wl = WL.WORKLOADS[workload]
    unfused = "unfused_4step" in modes
    units = []
    for i in range(n):
        u = HsdpUnit(C.Plan(wl.d0, wl.inner, wl.rank_size, wl.shard_size).upload(), wl.param_dtype,
                     wl.grad_dtype, device=dev, with_unfused=unfused, backward_only=True)
        WL.torch_fill_(u.grads, wl.seed_grads + 100 * i, wl.grad_std, wl.grad_dtype)
        units.append(u)
    a = torch.randn(8192, 8192, device=dev, dtype=torch.bfloat16)
    comp = torch.cuda.current_stream()

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(comp)
        for _ in range(reps):
            fn()
        e.record(comp)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    def set_cap(cap):
        for u in units:
            u.plan.set_grid_limit(cap)

    # size the stand-in backward of one layer to about one layer's fused sync
    t_sync1 = timed(lambda: units[0].reduce_grads("avg"))
    t_mm = timed(lambda: torch.mm(a, a))
    k = max(1, int(round(t_sync1 / t_mm)))

    def compute(L):
        for _ in range(k):
            torch.mm(a, a)

    out = {"layers": n, "workload": wl.key, "gemms_per_layer": k, "gemm": "8192^3 bf16 (cuBLAS)",
           "caps": "blocks of each sync kernel issued while compute may run (one per SM); 0 = whole GPU"}
    t_comp = timed(lambda: [compute(L) for L in reversed(range(n))])
    out["compute_only_ms"] = round(t_comp, 3)
    syncs = {"one_pass": lambda L: units[L].reduce_grads_one_pass("avg"),
             "fused": lambda L: units[L].reduce_grads("avg"),
             "unfused_4step": lambda L: units[L].reduce_grads_unfused("avg")}
    for mode in modes:
        sync = syncs[mode]
        fused, one = mode != "unfused_4step", mode == "one_pass"
        t_sync = timed(lambda: [sync(L) for L in reversed(range(n))])
        res = {"sync_only_ms": round(t_sync, 3), "serial_ms": round(t_comp + t_sync, 3)}
        for cap in (0, 48, 56, 64, 80):
            row = {}
            if cap:
                set_cap(cap)
                row["sync_only_capped_ms"] = round(timed(lambda: [sync(L) for L in reversed(range(n))]), 3)
                set_cap(0)
            t_pipe = timed(lambda: BackwardPipeline(units, "avg", fused, comm_blocks=cap, one_pass=one).run(compute))
            row["pipelined_ms"] = round(t_pipe, 3)
            row["hidden_frac"] = round((t_comp + t_sync - t_pipe) / max(1e-9, min(t_comp, t_sync)), 3)
            res[f"cap_{cap}"] = row
        out[mode] = res
    # per schedule: the cap that hid the most of the shorter of compute and sync
    out["best"] = {m: max(((c, r["hidden_frac"]) for c, r in out[m].items() if c.startswith("cap_")),
                          key=lambda x: x[1]) for m in modes}
    status = [u.plan.status() for u in units]
    out["status_words"] = status
    for u in units:
        u.close()
    return out


def run_e2e(args, unit, calls, step_bytes, world, dev):
    """The same metric end to end: every step copies its inputs (the local
    shards and the full gradients of every rank) from pinned host memory,
    runs the step, and copies its results (the full parameters and the
    averaged shard gradients) back to pinned host memory."""
    import torch

    ins = unit.shards + unit.grads
    outs = unit.full + unit.shard_grads
    need = sum(t.numel() * t.element_size() for t in ins + outs)
    local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", world))
    have = host_memory_bytes()
    if have and need * local_ranks > 0.6 * have:
        # pinned host copies of every rank's inputs and outputs would not fit
        return {"skipped": f"pinned host buffers need {need * local_ranks / 1e9:.0f} GB for "
                           f"{local_ranks} local ranks, host has {have / 1e9:.0f} GB"}
    h_in = [torch.empty(t.numel(), dtype=t.dtype, pin_memory=True) for t in ins]
    h_out = [torch.empty(t.numel(), dtype=t.dtype, pin_memory=True) for t in outs]
    for h, t in zip(h_in, ins):
        h.copy_(t)
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)

    # Three streams: host->device copies, the step, device->host copies.
    # Step k+1's inputs upload while step k's results download (the link is
    # full duplex); the step waits for its inputs and for the previous
    # download to finish reading the outputs it overwrites; an upload waits
    # for the previous step to finish reading the inputs it overwrites.
    compute = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    state = {"done": None, "out": None}

    def one():
        if state["done"] is not None:
            s_in.wait_event(state["done"])
        with torch.cuda.stream(s_in):
            for t, h in zip(ins, h_in):
                t.copy_(h, non_blocking=True)
        ev_in = s_in.record_event()
        compute.wait_event(ev_in)
        if state["out"] is not None:
            compute.wait_event(state["out"])
        for c in calls:
            c()
        state["done"] = compute.record_event()
        s_out.wait_event(state["done"])
        with torch.cuda.stream(s_out):
            for h, t in zip(h_out, outs):
                h.copy_(t, non_blocking=True)
        state["out"] = s_out.record_event()

    one()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        one()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / args.e2e_steps
    dt = dist_max(dt, world, dev)
    value = dist_sum(step_bytes, world, dev) / dt / 1e9
    del h_in, h_out
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(dt * 1e3, 2), "steps": args.e2e_steps}


def run_profile_case(args, wl):
    """One kernel of the step, args.launches times, on the workload with
    every dim 0 scaled by args.scale and only the buffers that kernel reads
    and writes allocated: the case an ncu capture of that kernel runs."""
    import torch

    from hsdp_sharded_parameter_gb300 import capi as C
    from hsdp_sharded_parameter_gb300 import workloads as WL

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    d0 = wl.d0 if args.scale == 1.0 else scaled_workload(wl, args.scale)[0]
    plan = C.Plan(d0, wl.inner, wl.rank_size, wl.shard_size).upload()
    W, S, P = plan.W, plan.S, plan.P
    pdt, gdt = wl.param_dtype, wl.grad_dtype
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}

    def alloc(sizes, dt):
        return [torch.empty(int(n), dtype=tdt[dt], device=dev) for n in sizes]

    shard_sizes = [plan.shard_numel(p, w % S) for w in range(W) for p in range(P)]
    full_sizes = [plan.numel(p) for _ in range(W) for p in range(P)]
    k = args.profile_kernel
    if k in ("ag_copy_in", "ag_unshard"):
        src = alloc(shard_sizes, pdt)
        WL.torch_fill_(src, wl.seed_params, wl.param_std, pdt)
        b_src = plan.bind("shards", pdt, src)
    if k == "ag_copy_in":
        dst = alloc([S * plan.slice_numel(pdt)] * W, pdt)
        b_dst = plan.bind("ag_output", pdt, dst)
        call = lambda: C.fsdp_ag_copy_in(plan, b_src, b_dst, True)  # noqa: E731
    elif k == "ag_unshard":
        dst = alloc(full_sizes, pdt)
        b_dst = plan.bind("full_params", pdt, dst)
        call = lambda: C.fsdp_ag_unshard(plan, b_src, b_dst)  # noqa: E731
    elif k == "ag_copy_out":
        src = alloc([S * plan.slice_numel(pdt)] * W, pdt)
        WL.torch_fill_(src, wl.seed_params, wl.param_std, pdt)
        dst = alloc(full_sizes, pdt)
        b_src, b_dst = plan.bind("ag_output", pdt, src), plan.bind("full_params", pdt, dst)
        call = lambda: C.fsdp_ag_copy_out(plan, b_src, b_dst)  # noqa: E731
    elif k in ("rs_ar_reduce", "rs_ar_reduce_apply"):
        src = alloc(full_sizes, gdt)
        WL.torch_fill_(src, wl.seed_grads, wl.grad_std, gdt)
        dst = alloc([plan.slice_numel("f32")] * W, "f32")
        b_src, b_dst = plan.bind("grads", gdt, src), plan.bind("fused", "f32", dst)
        call = lambda: C.fsdp_rs_ar_reduce(plan, b_src, b_dst)  # noqa: E731
        if k == "rs_ar_reduce_apply":
            sg = alloc(shard_sizes, gdt)
            b_sg = plan.bind("shard_grads", gdt, sg)
            dst = dst + sg
            call = lambda: C.fsdp_rs_ar_reduce_apply(plan, b_src, b_dst, "avg", b_sg)  # noqa: E731
    else:
        src = alloc([plan.slice_numel("f32")] * W, "f32")
        WL.torch_fill_(src, wl.seed_grads, wl.grad_std, "f32")
        dst = alloc(shard_sizes, gdt)
        b_src, b_dst = plan.bind("fused", "f32", src), plan.bind("shard_grads", gdt, dst)
        call = lambda: C.fsdp_apply_grads(plan, b_src, "avg", b_dst)  # noqa: E731
    plan.set_grid_limit(args.grid_limit)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for i in range(args.launches):
        ev[0].record()
        call()
        ev[1].record()
        torch.cuda.synchronize()
        print(f"{k} {wl.key} dim0 x{args.scale:g} grid limit {args.grid_limit} launch {i}: "
              f"{ev[0].elapsed_time(ev[1]) * 1e3:.1f} us", flush=True)
    print(f"{k}: {sum(t.numel() * t.element_size() for t in src + dst) / 1e9:.2f} GB on the device", flush=True)
    status = plan.status()
    if status:
        print(f"{k}: plan status {status} (a wait inside the kernel ran out)", flush=True)
        return 1
    return 0


def main(argv=None):
    args = parse(argv)
    from hsdp_sharded_parameter_gb300 import workloads as WL

    wl = WL.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.profile_kernel:
        return run_profile_case(args, wl)
    return run_gpu(args, wl)


if __name__ == "__main__":
    sys.exit(main())
