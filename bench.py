#!/usr/bin/env python3
"""Benchmark of the shape-fused Muon step on GB300 (one JSON line on rank 0).

Headline workload: the dense h=4096 transformer (32 layers x 4 shape buckets
of 32 matrices: [4096,12288], [4096,4096], [4096,16384], [16384,4096]; bf16
params/grads, fp32 momentum, 5 quintic Newton-Schulz steps), the largest of
the benchmark configurations.  The line also carries a `per_config` block that
times every configuration the same way: the fp32 64x128 case, the pages' fused
skinny batch 74 x [24, 10240] («MindSpore HyperParallel X 盘古,Muon优化器实现6倍
性能跃升», 矩阵融合优化, Fig. 7), the MoE expert tensor with its skinny group,
the dense model, and the 1000-matrix mixed bag at 5 and 10 steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--impl reference] [--no-per-config] [--no-cpu-baseline] [--no-e2e]

`value` is whole-job algorithmic throughput (GB/s of the compulsory G, M, M',
P, P' traffic for workloads made only of memory-bound skinny groups; TFLOP/s
of the dense count 4 m^2 n + 2 m^3 per matrix per NS step otherwise) with
inputs resident in HBM.  Timing: CUDA events on the launching stream, W
untimed warm-up steps, K timed steps, barrier + synchronize on both sides, max
over ranks.  As in a training loop, every step updates the same buffers;
before each step an untimed write of twice the L2 size flushes it, an untimed
read of as much drains the flush's write-backs, and each step is timed alone
by its own event pair.  `e2e` times the same step through muon_step_host
(host buffers in pinned memory, host->device and device->host copies inside
the timed region).  `--impl reference` times the CPU oracle on the host cores
instead (it never loads the CUDA library).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused Muon step ms & TFLOP/s (or GB/s) per shape group, % roofline, 1×GB300"
DEFAULT_CONFIG = "c4_dense_h4096"
PER_CONFIG = [("c1_fp32_64x128", None), ("c2_skinny_74x24x10240", None),
              ("c3_moe_64x2048x7168_32x24x10240", None), ("c4_dense_h4096", None),
              ("c5_mixed_1000", 5), ("c5_mixed_1000", 10)]
L2_BYTES = 129 * 2 ** 20
SKINNY_MAX_M = 64  # the planner's default skinny threshold (min(rows, cols) <= 64)


def algorithmic_work(shapes, mode, k):
    """(bytes, flops) of one step: compulsory traffic (P, G read; M read+write;
    P write) and the dense NS flops k (4 m^2 n + 2 m^3) per matrix."""
    pb = 4 if mode == "fp32" else 2
    byts, flops = 0, 0
    for s in shapes:
        E = s[0] if len(s) == 3 else 1
        r, c = s[-2], s[-1]
        m, n = min(r, c), max(r, c)
        byts += E * r * c * (pb + 4 + 4 + pb + pb)
        flops += E * k * (4 * m * m * n + 2 * m ** 3)
    return byts, flops


def shape_groups(shapes, mode):
    """The planner's default bucketing restated for the report: exact
    (rows, cols) keys in first-seen order, 3-D parameters contributing E
    members, and the path each group takes by default (skinny for
    min(rows, cols) <= 64 in bf16 mode, tensor above, SIMT in fp32 mode).
    Pure Python, so the reference arm never loads the CUDA library."""
    groups = {}
    for s in shapes:
        E = s[0] if len(s) == 3 else 1
        key = (s[-2], s[-1])
        groups[key] = groups.get(key, 0) + E
    out = []
    for (r, c), b in groups.items():
        path = "simt" if mode == "fp32" else ("skinny" if min(r, c) <= SKINNY_MAX_M else "tensor")
        out.append({"rows": r, "cols": c, "batch": b, "path": path})
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_hash(name):
    path = os.path.join(ROOT, "newton_schulz_bucket_gb300", "csrc", name)
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16] if os.path.exists(path) else None


def ncu_traffic(kernel_file, workload):
    """DRAM bytes (read + write) per launch of the dominant kernel, from the
    committed ncu summary, if it was taken on the current source of that
    kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d:
        return None
    files = d.get("source_files") or [d.get("source_file", kernel_file)]
    want = d.get("source_sha256_16")
    want = want if isinstance(want, list) else [want]
    if [kernel_source_hash(f) for f in files] != want:
        return None
    return d


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"muon_clocks_{os.getpid()}_{time.monotonic_ns()}.csv")

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
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
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, fl in rows for i, v in enumerate(fl) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allmax(world, v):
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(v)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return v


# ---------------------------------------------------------------- CPU oracle


def blas_name():
    """NumPy's BLAS library and version, as its build config reports them."""
    import numpy as np
    try:
        d = np.show_config(mode="dicts")["Build Dependencies"]["blas"]
        return f"{d.get('name', '?')} {d.get('version', '')}".strip()
    except Exception:  # older NumPy: no dict form of the build config
        return "unknown"


def busy_cores(wall, cpu):
    """Host threads the oracle used: its CPU time over its wall time, rounded
    up (at least 1)."""
    return max(1, math.ceil(cpu / wall - 0.05)) if wall > 0 else 1


def host_member_inputs(w):
    """Host fp64 inputs of single members, each drawn alone from its own
    parameter's (or expert's) law, for timing the oracle: the values need not
    match the GPU draw, and an expert tensor is never drawn whole."""
    from newton_schulz_bucket_gb300 import workloads as W

    def get(i, e):
        gs = w.g_std[i]
        std = float(gs[e]) if isinstance(gs, (list, tuple)) else float(gs)
        sub = W.custom([w.shapes[i][-2:]], mode=w.mode, seed=w.seed * 100003 + i * 1009 + e,
                       g_std=std, p_std=float(w.p_std[i]))
        P, G, M = W.make_tensors(sub, "cpu")
        return tuple(t[0].float().double().numpy() for t in (P, G, M))
    return get


def member_flops(rows, cols, k):
    m, n = min(rows, cols), max(rows, cols)
    return k * (4 * m * m * n + 2 * m ** 3)


def workload_groups(w):
    """{(rows, cols): [(param, expert), ...]} in first-seen order."""
    groups = {}
    for i, s in enumerate(w.shapes):
        for e in range(s[0] if len(s) == 3 else 1):
            groups.setdefault((s[-2], s[-1]), []).append((i, e))
    return groups


def time_members(w, members, get):
    """Wall and process-CPU seconds of the oracle on `members` (inputs drawn
    before the timed region)."""
    import numpy as np
    from oracle import muon_ref
    f32 = lambda v: float(np.float32(v))
    a, b, c = (f32(v) for v in w.coeffs)
    inputs = [get(i, e) for (i, e) in members]
    t0, c0 = time.perf_counter(), time.process_time()
    for P, G, M in inputs:
        muon_ref.muon_update_ref(P, G, M, f32(w.beta), f32(w.lr), f32(w.wd), w.ns_steps, a, b, c)
    return time.perf_counter() - t0, time.process_time() - c0


def oracle_estimate(w, budget_s, get):
    """The oracle's time for one whole step of w, from a bounded sample.

    Groups are taken cheapest member first.  Each taken group gets as many
    members as its share of the budget allows (at least one) and is
    extrapolated by its member count.  Once the budget is spent, the groups
    left (whose single member would overrun it) are extrapolated by their
    dense Newton-Schulz FLOPs at the FLOP rate the oracle reached on the
    largest sampled tensor-size group (or by bytes for skinny-size groups).
    Returns (seconds per step, wall, cpu, sample note)."""
    import random
    rng = random.Random(1234)
    groups = workload_groups(w)
    keys = sorted(groups, key=lambda k: member_flops(k[0], k[1], w.ns_steps) + k[0] * k[1])
    total = wall = cpu = 0.0
    rate_flops = None   # oracle FLOP/s on the largest timed tensor-size group
    rate_elem = None    # oracle seconds per element on the largest timed skinny-size group
    timed, left = [], []
    spent = 0.0
    for key in keys:
        mem = groups[key][:]
        rng.shuffle(mem)
        r, c = key
        fl = member_flops(r, c, w.ns_steps)
        # projected seconds of one member from what has been measured so far
        guess = (fl / rate_flops if rate_flops else fl / 2.5e11) + r * c * 2e-8
        if timed and spent + guess > budget_s:
            left.append(key)
            continue
        n = 1
        if guess > 0:
            n = max(1, min(len(mem), int(max(budget_s - spent, 0.0) / max(guess, 1e-6) / 4)))
        dt, dc = time_members(w, mem[:n], get)
        spent += dt
        wall += dt
        cpu += dc
        total += dt * len(mem) / n
        timed.append(f"{n} of {len(mem)} x {list(key)}")
        if min(r, c) > SKINNY_MAX_M:
            rate_flops = fl * n / dt
        else:
            rate_elem = dt / (n * r * c)
    for (r, c) in left:
        cnt = len(groups[(r, c)])
        if min(r, c) > SKINNY_MAX_M and rate_flops:
            total += cnt * member_flops(r, c, w.ns_steps) / rate_flops
        else:
            total += cnt * r * c * (rate_elem or 2e-8)
    note = "timed: " + "; ".join(timed)
    if left:
        note += ("; extrapolated by dense NS FLOPs at the oracle's measured rate: " +
                 "; ".join(f"{len(groups[k])} x {list(k)}" for k in left))
    return total, wall, cpu, note


def headline(w, byts, flops, seconds):
    """GB/s for workloads made only of HBM-bound (skinny, resident) groups,
    else TFLOP/s."""
    if all(g["path"] in ("skinny", "resident") for g in shape_groups(w.shapes, w.mode)):
        return byts / seconds / 1e9, "GB/s"
    return flops / seconds / 1e12, "TFLOP/s"


def config_dict(w, world, in_bytes=None):
    """The `config` of the JSON line (the same for both arms)."""
    d = {"workload": w.name, "shapes": describe_shapes(w.shapes), "ns_steps": w.ns_steps,
         "coeffs": list(w.coeffs), "mode": w.mode,
         "ns_operands": "fp32 (FFMA)" if w.mode == "fp32" else "fp16 (fp32 accumulate)",
         "l2": "same buffers every step; L2 flushed before each step by an untimed "
               f"{2 * L2_BYTES / 1e6:.0f} MB write, then drained by an untimed read of as much; "
               "each step timed alone",
         "parallelism": f"replicas x{world}"}
    return d


def run_reference(args, w, world, rank):
    """--impl reference: the CPU oracle as it stands, on the host cores.  Each
    step times a bounded sample of the workload and extrapolates it to the
    whole step; nothing here loads the CUDA library."""
    if rank != 0:
        return
    byts, flops = algorithmic_work(w.shapes, w.mode, w.ns_steps)
    get = host_member_inputs(w)
    budget = max(1.0, 90.0 / max(1, args.steps))
    smallest = min(workload_groups(w).items(), key=lambda kv: kv[0][0] * kv[0][1])
    for _ in range(args.warmup):   # warms NumPy's BLAS on one member of the smallest group
        time_members(w, smallest[1][:1], get)
    runs = [oracle_estimate(w, budget, get) for _ in range(args.steps)]
    per_step = statistics.mean(r[0] for r in runs)  # extrapolated to the whole workload
    value, unit = headline(w, byts, flops, per_step)
    cores = busy_cores(sum(r[1] for r in runs), sum(r[2] for r in runs))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(w, world),
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores,
                             "host_cores": os.cpu_count(), "blas": blas_name(), "kind": "oracle",
                             "sample": runs[0][3] + " (per step; members drawn before timing)"},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def describe_shapes(shapes):
    from collections import Counter
    c = Counter(tuple(s) for s in shapes)
    return ", ".join(f"{n}x{list(s)}" for s, n in c.items())


# ------------------------------------------------------------------ GPU arm


def executed_flop_fraction(rows, cols):
    """Share of the dense count k (4 m^2 n + 2 m^3) the tensor path executes.
    The Gram matrix (2 m^2 n) and A^2 (2 m^3) are symmetric, so their GEMMs
    compute only the 128 x BN tiles that reach the upper triangle and mirror
    the rest (BN = 256 for m >= 256, else 128); Q Y (2 m^2 n) is dense."""
    m, n = min(rows, cols), max(rows, cols)
    bn = 256 if m >= 256 else 128
    tm_, tn_ = -(-m // 128), -(-m // bn)
    sym = sum(max(tn_ - (t * 128) // bn, 0) for t in range(tm_)) / (tm_ * tn_)
    dense = 4 * m * m * n + 2 * m ** 3
    return (sym * (2 * m * m * n + 2 * m ** 3) + 2 * m * m * n) / dense


def executed_flops(w, groups):
    """Newton-Schulz FLOPs the step executes (the dense count, with the
    symmetric products of tensor-path groups reduced to their computed tiles;
    skinny and resident groups are counted dense)."""
    tot = 0.0
    for g in groups:
        f = member_flops(g["rows"], g["cols"], w.ns_steps) * g["batch"]
        tot += f * (executed_flop_fraction(g["rows"], g["cols"]) if g["path"] == "tensor" else 1.0)
    return tot


def group_entry(info, gms, w, peaks):
    """One group's row: ms, matrices/s and its roofline (HBM when its dense
    FLOPs per compulsory byte fall below the ridge -- every skinny group and
    small-m tensor groups such as [128, 4096] -- else the tensor cores)."""
    shp = [info["rows"], info["cols"]]
    gb, gf = algorithmic_work([[info["batch"]] + shp], w.mode, w.ns_steps)
    ent = {"shape": shp, "batch": info["batch"], "path": info["path"], "ms": gms}
    if not gms:
        return ent
    ent["matrices_per_s"] = info["batch"] / (gms / 1e3)
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if info["path"] in ("skinny", "resident") or gf / gb < ridge:
        ach = gb / (gms / 1e3) / 1e9
        ent.update({"GB_s": ach, "roofline_frac": ach / peaks["hbm_gbs"], "bound": "hbm",
                    "flop_per_byte": gf / gb})
    else:
        # TFLOP/s of the dense count (algorithmic); the executed rate counts
        # only the tiles the symmetric products compute
        ach = gf / (gms / 1e3) / 1e12
        xf = executed_flop_fraction(*shp) if info["path"] == "tensor" else 1.0
        ent.update({"TFLOP_s": ach, "roofline_frac": ach / peaks["bf16_tflops_sustained"],
                    "bound": "tensor", "executed_flop_fraction": xf, "TFLOP_s_executed": ach * xf,
                    "roofline_frac_executed": ach * xf / peaks["bf16_tflops_sustained"]})
    return ent


def roofline_of(w, dg, peaks):
    """The `roofline` object for the dominant group `dg`."""
    if dg.get("bound") == "hbm":
        if dg["path"] == "skinny":
            gram_space = w.ns_steps <= 64
            kfile = "k_skinny_gs.cuh" if gram_space else "k_skinny.cu"
            kernel = ("k_skinny_gs (momentum + Gram-space Newton-Schulz + write, one launch)"
                      if gram_space else "k_momentum_partial + k_skinny_ns")
        elif dg["path"] == "resident":
            kfile = "k_resident.cu"
            kernel = "k_resident (momentum, the k Newton-Schulz steps on chip, write; one launch)"
        else:
            kfile = None
            chain = "k_simt_gemm (fp32 FFMA)" if dg["path"] == "simt" else "k_tc_gemm"
            kernel = f"group {dg['shape']} x {dg['batch']}: {chain} chain and the elementwise passes"
        tr = ncu_traffic(kfile, w.name) if kfile else None
        roof = {"bound": "hbm", "achieved": dg.get("GB_s"), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": dg.get("roofline_frac"), "kernel": kernel,
                "peak_source": peaks["source"] + " hbm_gbs (burst copy)"}
    else:
        tr = ncu_traffic("k_tc_gemm.cu", w.name)
        roof = {"bound": "tensor", "achieved": dg.get("TFLOP_s"), "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": dg.get("roofline_frac"),
                "kernel": f"group {dg['shape']} x {dg['batch']}: its k_tc_gemm launches "
                          "(Gram, polynomial, update per step) and elementwise passes",
                "peak_source": peaks["source"] + " bf16_tflops_sustained",
                "flops_counted": "dense k (4 m^2 n + 2 m^3); the symmetric Gram and A^2 compute "
                                 "only upper-triangle tiles",
                "executed_flop_fraction": dg.get("executed_flop_fraction"),
                "achieved_executed": dg.get("TFLOP_s_executed"),
                "frac_executed": dg.get("roofline_frac_executed")}
    # DRAM bytes of the dominant kernel from one ncu capture, per launch; null
    # once the kernel source changed since the capture
    roof["traffic"] = tr.get("dram_bytes_per_launch") if tr else None
    if tr:
        roof["traffic_detail"] = {k: tr[k] for k in ("dram_read_bytes", "dram_write_bytes",
                                                     "compulsory_read_bytes", "compulsory_write_bytes",
                                                     "note") if k in tr}
    return roof


def plan_options(args):
    """Plan options from the command line: `--path` forces one kernel path
    for every group (default: the planner's choice)."""
    path = getattr(args, "path", "auto")
    return {} if path == "auto" else {"path": path}


def measure(w, args, pkg, torch, dev, local, world, peaks, stream, flush, sample_clocks):
    """Times workload w on this GPU: K timed steps (the whole step, every
    group), then per-group times from a second plan that runs the groups one
    after another.  Returns (summary dict, kernel launches per step)."""
    from newton_schulz_bucket_gb300 import workloads as W
    byts, flops = algorithmic_work(w.shapes, w.mode, w.ns_steps)
    tensors = W.make_tensors(w, dev)
    plan = pkg.MuonPlan(w.shapes, device=local, mode=w.mode, **plan_options(args))
    groups = plan.groups()
    bound = plan.bind(*tensors)
    sp = stream.cuda_stream

    def step():
        plan.step_bound(bound, w.beta, w.lr, w.wd, w.ns_steps, w.coeffs, stream=sp)

    for j in range(args.warmup):
        flush(j)
        step()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clk = ClockSampler(local) if sample_clocks else None
    if clk:
        clk.__enter__()
    t_wall = time.perf_counter()
    for j in range(args.steps):
        flush(j)
        evs[j][0].record(stream)
        step()
        evs[j][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if clk:
        clk.__exit__(None, None, None)
    step_ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    barrier(world)
    launches = plan.kernels_per_step(w.ns_steps)
    plan.close()
    # per-group kernel times from events recorded inside the step graph of a
    # plan that runs the groups one after another
    tplan = pkg.MuonPlan(w.shapes, device=local, mode=w.mode, group_timing=True, max_streams=1,
                         **plan_options(args))
    tbound = tplan.bind(*tensors)
    gtimes = [[] for _ in groups]
    for j in range(min(args.steps, 6) + 1):
        flush(j)
        tplan.step_bound(tbound, w.beta, w.lr, w.wd, w.ns_steps, w.coeffs, stream=sp)
        if j == 0:
            continue  # graph capture
        for g in range(len(groups)):
            gtimes[g].append(tplan.group_elapsed_ms(g))
    torch.cuda.synchronize()
    tplan.close()
    del tensors, bound, tbound
    torch.cuda.empty_cache()

    ms_step = allmax(world, sum(step_ms)) / args.steps
    sec = ms_step / 1e3
    value_1, unit = headline(w, byts, flops, sec)
    per_group = [group_entry(info, statistics.mean(gtimes[g]) if gtimes[g] else None, w, peaks)
                 for g, info in enumerate(groups)]
    dom = max(range(len(groups)), key=lambda g: per_group[g]["ms"] or 0)
    out = {"workload": w.name, "shapes": describe_shapes(w.shapes), "ns_steps": w.ns_steps,
           "value": value_1 * world, "unit": unit, "ms_per_step": ms_step,
           "step_ms_this_rank": {"median": statistics.median(step_ms), "min": min(step_ms),
                                 "max": max(step_ms)},
           "matrices_per_s": sum(g["batch"] for g in groups) * world / sec,
           "tflops": flops * world / sec / 1e12, "gbs": byts * world / sec / 1e9,
           "tflops_executed": executed_flops(w, groups) * world / sec / 1e12,
           "per_group": per_group, "roofline": roofline_of(w, per_group[dom], peaks),
           "wall_s_timed": t_wall}
    if clk:
        out["clocks"] = clk.summary()
    return out, launches


def run_e2e(args, w, pkg, torch, dev, local, byts, flops, world):
    """Same step through muon_step_host: H2D of P, G, M and D2H of P', M'
    inside the timed region.  The pinned host buffers are filled on the host
    from the device draw, one parameter at a time."""
    from newton_schulz_bucket_gb300 import workloads as W
    pdt = torch.bfloat16 if w.mode == "bf16" else torch.float32
    el = sum(math.prod(s) for s in w.shapes)
    hP = torch.empty(el, dtype=pdt, pin_memory=True)
    hG = torch.empty(el, dtype=pdt, pin_memory=True)
    hM = torch.empty(el, dtype=torch.float32, pin_memory=True)

    def views(flat):
        out, o = [], 0
        for s in w.shapes:
            n = math.prod(s)
            out.append(flat[o:o + n].view(*s))
            o += n
        return out
    vP, vG, vM = views(hP), views(hG), views(hM)
    P, G, M = W.make_tensors(w, dev)
    for i in range(len(w.shapes)):
        vP[i].copy_(P[i]); vG[i].copy_(G[i]); vM[i].copy_(M[i])
    del P, G, M
    torch.cuda.empty_cache()
    plan = pkg.MuonPlan(w.shapes, device=local, mode=w.mode, host_staging=True, **plan_options(args))
    stream = torch.cuda.Stream(dev)
    # the first host step of a process measured about 600 ms on c4 against
    # 350-460 for the ones after it, so warm up with a few
    for _ in range(max(3, args.warmup // 2)):
        plan.step_host(vP, vG, vM, w.beta, w.lr, w.wd, w.ns_steps, w.coeffs, stream=stream)
    torch.cuda.synchronize()
    barrier(world)
    n = max(6, args.steps // 3)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        plan.step_host(vP, vG, vM, w.beta, w.lr, w.wd, w.ns_steps, w.coeffs, stream=stream)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(n))
    ms = allmax(world, evs[0].elapsed_time(evs[n])) / n
    plan.close()
    del hP, hG, hM, vP, vG, vM
    torch.cuda.empty_cache()
    v, u = headline(w, byts, flops, ms / 1e3)
    pb = 2 if w.mode == "bf16" else 4
    return {"value": v * world, "unit": u, "ms_per_step": ms, "steps": n,
            "step_ms_this_rank": {"median": per[n // 2], "min": per[0], "max": per[-1]},
            "h2d_bytes_per_step": el * (pb + pb + 4), "d2h_bytes_per_step": el * (pb + 4)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--ns-steps", type=int, default=None)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--path", default="auto", choices=["auto", "skinny", "tensor", "simt", "resident"],
                    help="force one kernel path for every group (profiling; default: the planner's)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from newton_schulz_bucket_gb300 import workloads as W
    w = W.get(args.config, args.ns_steps)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, w, world, rank)
        return

    import torch
    import newton_schulz_bucket_gb300 as pkg

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    drain_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)

    def flush(j):
        # untimed: write twice the L2 size (evicts the previous step's lines),
        # then read as much again so the write-backs of that flush happen here
        # and not inside the next timed step
        with torch.cuda.stream(stream):
            flush_buf.fill_(float(j))
            torch.sum(drain_buf, dim=0, out=sink)

    head, launches = measure(w, args, pkg, torch, dev, local, world, peaks, stream, flush, True)
    byts, flops = algorithmic_work(w.shapes, w.mode, w.ns_steps)

    per_config = None
    if not args.no_per_config:
        per_config = []
        for name, k in PER_CONFIG:
            wc = W.get(name, k)
            if wc.name == w.name and wc.ns_steps == w.ns_steps:
                ent = {kk: vv for kk, vv in head.items() if kk != "wall_s_timed"}
            else:
                ent, _ = measure(wc, args, pkg, torch, dev, local, world, peaks, stream, flush, True)
                ent.pop("wall_s_timed", None)
                if rank == 0 and world == 1 and not args.no_cpu_baseline:
                    # the oracle on a smaller sample (about 5 s) of this configuration
                    bc, fc = algorithmic_work(wc.shapes, wc.mode, wc.ns_steps)
                    t, wall, cpu_s, note = oracle_estimate(wc, 5.0, host_member_inputs(wc))
                    cv, cu = headline(wc, bc, fc, t)
                    ent["cpu_baseline"] = {"value": cv, "unit": cu, "ms_per_step": t * 1e3,
                                           "cores": busy_cores(wall, cpu_s), "kind": "oracle",
                                           "sample": note}
            per_config.append(ent)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, pkg, torch, dev, local, byts, flops, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        t, wall, cpu_s, note = oracle_estimate(w, 20.0, host_member_inputs(w))
        cv, cu = headline(w, byts, flops, t)
        cpu = {"value": cv, "unit": cu, "cores": busy_cores(wall, cpu_s),
               "host_cores": os.cpu_count(), "blas": blas_name(), "kind": "oracle",
               "sample": note + " (members drawn before timing)", "ms_per_step": t * 1e3,
               "wall_s": wall}

    if rank == 0:
        line = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
                "step_ms_this_rank": head["step_ms_this_rank"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16" if w.mode == "bf16" else "f32",
                "data": "synthetic: seeded Gaussian G, M0, P (per-config stds); no dataset",
                "config": dict(config_dict(w, world), **plan_options(args)),
                "matrices_per_s": head["matrices_per_s"], "tflops": head["tflops"],
                "gbs": head["gbs"], "tflops_executed": head["tflops_executed"],
                "per_group": head["per_group"], "roofline": head["roofline"],
                "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches * args.steps, "clocks": head.get("clocks"),
                "wall_s_timed": head["wall_s_timed"], "per_config": per_config}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
