#!/usr/bin/env python
"""Throughput of online KV-cache compaction on GB300: KV entries scored + compacted per second.

One step = the whole hot path over one synthetic cache: kvc_score (LSE pass + alpha pass),
kvc_select_topm, kvc_plan_compact, kvc_compact, kvc_free_pages, through the C ABI.  The cache
is restored from a device snapshot between steps, outside the timed CUDA events (the step
mutates it).  One entry = one token position of one (layer, KV head) in the compacted segment.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

N > 1 (torchrun, one rank per GPU): every rank compacts its own replica of the workload (units
are independent; no data-path collective); value = entries of all ranks / max rank time.
--impl reference times the fp64 CPU oracle on the host cores on a bounded sample.
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
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV entries scored+compacted/sec on 1 GB300; % of tensor/HBM roofline"
UNIT = "entries/s"
DEFAULT_WORKLOAD = "qwen3-30b-a3b"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the eager calls only (default: also replay the step as a CUDA graph "
                         "and report the replays)")
    ap.add_argument("--scorer", choices=["te", "actkv"], default="te",
                    help="eviction score: the token-eviction attention-mass score (default) or "
                         "ActKV's action attention smoothed by LRFU")
    ap.add_argument("--variant", choices=["inplace", "sentinel", "fresh"], default="inplace",
                    help="eviction layout after selection: the in-place tail-region compaction "
                         "(default), sentinel dead slots, or compaction into fresh pages")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None,
                    help="override the workload's layer count (small profiling cases)")
    ap.add_argument("--seqs", type=int, default=None,
                    help="keep the workload's first N sequences (small profiling cases)")
    ap.add_argument("--qdist", choices=["normal", "planted4", "aligned"], default=None,
                    help="override the workload's proxy-query distribution (e.g. diffuse 'normal' "
                         "queries, where Attention Matching has mass to recover)")
    ap.add_argument("--am-sweeps", type=int, default=0,
                    help="Attention Matching after the selection: fit the bias and the compact "
                         "values of the kept entries with this many coordinate-descent sweeps "
                         "(0: token eviction alone)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def workload_desc(sp) -> str:
    n = sp.lengths
    nd = f"n{n[0]}" if len(n) == 1 else f"B{len(n)} n{min(n)}..{max(n)} (sum {sum(n)})"
    bud = f"ratio {sp.budget[1]}" if sp.budget[0] == "ratio" else "ActKV budgets 512*1.75^k"
    return (f"{sp.name}: L{sp.L} Hkv{sp.H} G{sp.G} d{sp.d} {nd} P{sp.P} R{sp.R} {bud} "
            f"kv={sp.kv} q={sp.qdist}")


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (100 ms) with timestamps; summarised over a wall-clock window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        uuid = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass
        if uuid:
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        self.lines = [l.strip() for l in self.out.read().splitlines() if l.strip()]
        self.out.close()
        try:
            os.unlink(self.out.name)
        except OSError:
            pass

    def summary(self, t0: float, t1: float):
        import datetime as dt
        rows = []
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((ts, parts))
        window = [p for ts, p in rows if t0 - 0.05 <= ts <= t1 + 0.05] or [p for _, p in rows]
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[2]) for p in window if num(p[2]) is not None]
        smax = [num(p[3]) for p in window if num(p[3]) is not None]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for p in window for i in range(4) if p[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(window)}


# ----------------------------------------------------------------------------- oracle arm

def oracle_sample(case, m, layers: int, threads: int):
    """Times the fp64 oracle (score + select + compact + free) on the first `layers` layers of
    the workload, on host copies.  Returns (seconds, entries, threads used)."""
    import numpy as np
    import torch
    import oracle

    sp = case.spec
    Ls = max(1, min(layers, sp.L))
    kb = case.k_pool[:Ls].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    vb = case.v_pool[:Ls].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    tags = case.tags[:Ls].contiguous().cpu().numpy().astype(np.int32)
    qb = case.q[:, :Ls].contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    bt = case.block_table.cpu().numpy().astype(np.int32)
    nbk = case.nblocks.cpu().numpy().astype(np.int32)
    fi = case.free_ids.cpu().numpy().astype(np.int32)
    ft = case.free_top.cpu().numpy().astype(np.int32)
    units = Ls * sp.H * sum(1 for s, e in zip(case.seg_start, case.seg_end) if e > s)
    used = max(1, min(threads, units))
    t0 = time.perf_counter()
    scores, _ = oracle.score_cache(kb, bt, nbk, case.seg_start, case.seg_end, case.seq_len, qb,
                                   sp.scale, threads=used)
    keep = oracle.select_cache(scores, case.seg_start, case.seg_end, m, threads=used)
    oracle.compact_layers(kb, vb, tags, 0, Ls, bt, case.seg_start, case.seg_end, m, keep)
    oracle.free_blocks(bt, nbk, fi, ft, sp.P, case.seg_start, case.seg_end, m)
    dt_s = time.perf_counter() - t0
    entries = Ls * sp.H * sum(e - s for s, e in zip(case.seg_start, case.seg_end))
    return dt_s, entries, used


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def reference_arm(args):
    """--impl reference: the oracle as it stands, timed on the host cores."""
    import torch
    import workloads

    sp = workloads.spec(args.workload, args.seed)
    import oracle
    oracle.build()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = workloads.build(sp, args.seed, dev)
    m = budgets_oracle(case)
    cores = host_cores()
    # one step = a bounded sample: the smallest number of layers that gives every core a unit
    layers = max(1, min(sp.L, math.ceil(cores / max(1, sp.H))))
    times = []
    entries = 0
    used = 1
    for i in range(args.warmup + args.steps):
        dt_s, entries, used = oracle_sample(case, m, layers, cores)
        if i >= args.warmup:
            times.append(dt_s)
    mean = statistics.mean(times)
    value = entries / mean
    sample = (f"{layers} of {sp.L} layers x {sp.H} KV heads ({entries} entries) per step, "
              f"full oracle chain (score, select, compact, free)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_desc(sp)},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def budgets_oracle(case):
    import oracle
    kind, arg = case.spec.budget
    n = [e - s for s, e in zip(case.seg_start, case.seg_end)]
    if kind == "ratio":
        return [oracle.budget_ratio(x, arg) for x in n]
    return [min(oracle.budget_actkv(k), x) for k, x in zip(arg, n)]


def budgets_lib(case):
    import online_kv_cache_gb300 as kvc
    kind, arg = case.spec.budget
    n = [e - s for s, e in zip(case.seg_start, case.seg_end)]
    if kind == "ratio":
        return [kvc.kvc_budget_from_ratio(x, arg) for x in n]
    return [min(kvc.kvc_budget_actkv(k), x) for k, x in zip(arg, n)]


# ----------------------------------------------------------------------------- our arm

def profile_traffic(kernel: str, workload: str):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            data = json.load(f)
    except (OSError, ValueError):
        return None
    ent = data.get(kernel, {}).get(workload)
    if not ent:
        return None
    src = os.path.join(ROOT, "online_kv_cache_gb300", "csrc", ent.get("source", "score.cu"))
    try:
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    return ent.get("dram_bytes_per_launch") if digest == ent.get("source_sha256_16") else None


# ----------------------------------------------------------------------------- ranks
#
# Units (sequence, layer, KV head) are independent, so N GPUs run N replicas of the
# workload (one per rank, seeded seed + rank) with no exchange on the data path.
# The job ends when the slowest rank does: the step time is the maximum over ranks,
# and the whole-job throughput counts every rank's entries.

def am_flops(sp, n, m, sweeps: int):
    """Algorithmic flops of one Attention Matching fit (2 per multiply-add), summed over the units,
    as (targets, Gram products, fp32 rest).  Targets: Q K^T and P V over all n keys (the kept keys'
    exponentials reuse those logits), bf16 operands on the tensor cores.  Gram products: E^T [E | s],
    Ph^T Ph and Ph^T Y, fp32-accurate (on the tensor cores as split-bf16 products).  fp32 rest, on
    the CUDA cores: the compact probabilities and the two descents (m-long updates of the mass
    gradient, m x d-long updates of the value gradient, per step; their initial gradients)."""
    R, d = sp.R, sp.d
    ft = fg = ff = 0.0
    for nb, mb in zip(n, m):
        mb = min(mb, nb)
        if mb <= 0:
            continue
        units = sp.L * sp.H
        ft += units * 4.0 * R * nb * d
        fg += units * (2.0 * R * mb * (mb + 1) + 2.0 * R * mb * mb + 2.0 * R * mb * d)
        ff += units * (2.0 * R * mb + 2.0 * mb * mb * (d + 1) + sweeps * (2.0 * mb * mb + 2.0 * mb * mb * d))
    return ft, fg, ff


SPLIT_PRODUCTS = 6  # bf16 products per fp32-accurate product (three-part split, terms above 2^-24)


def fp32_peak_tflops() -> float:
    """fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 flops at the 2070 MHz maximum SM
    clock."""
    return 152 * 128 * 2 * 2070e6 / 1e12


def replica_seed(seed: int, rank: int) -> int:
    return seed + rank


def slowest_rank_ms(ms: float, world: int, device) -> float:
    """Maximum over the ranks of a per-rank time (ms); world == 1 returns it unchanged."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(entries_per_rank: int, world: int, ms: float) -> float:
    """Entries per second of the whole job: every rank's entries over the slowest step."""
    return entries_per_rank * world / (ms * 1e-3)


def our_arm(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from online_kv_cache_gb300 import build
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    import online_kv_cache_gb300 as kvc
    import workloads

    import dataclasses
    sp = workloads.spec(args.workload, args.seed)
    if args.layers:
        sp = dataclasses.replace(sp, L=args.layers)
    if args.qdist:
        sp = dataclasses.replace(sp, qdist=args.qdist)
    if args.seqs:
        bud = sp.budget if sp.budget[0] != "actkv" else ("actkv", sp.budget[1][:args.seqs])
        sp = dataclasses.replace(sp, lengths=sp.lengths[:args.seqs], budget=bud)
    if args.variant == "fresh":  # the fresh pages come from the free stack: leave room for them
        sp = dataclasses.replace(sp, headroom=max(sp.headroom, 0.35))
    case = workloads.build(sp, replica_seed(args.seed, rank), dev)
    m = budgets_lib(case)
    aux = None
    if args.scorer == "actkv" or args.am_sweeps > 0:  # per-slot LRFU values / AM biases, moved with their entries
        aux = torch.zeros(case.tags.shape, dtype=torch.float32, device=dev)
    cp = kvc.Compactor(case.k_pool, case.v_pool, case.tags, case.block_table, case.nblocks,
                       case.free_ids, case.free_top, case.seg_start, case.seg_end, case.seq_len, m,
                       sp.R, aux=aux)
    snap = case.snapshot()
    if aux is not None:
        snap.append(aux.clone())
        restore_core = case.restore

        def restore_all(sn):
            restore_core(sn[:-1])
            aux.copy_(sn[-1])
        case.restore = restore_all
    n = [e - s for s, e in zip(case.seg_start, case.seg_end)]
    entries = sp.L * sp.H * sum(n)
    stream = torch.cuda.current_stream()
    stages = ("score_lse", "score_alpha", "select", "am_fit", "plan", "compact", "free")
    nev = len(stages) + 1

    class _NoEvent:
        def record(self, _stream):
            pass

    def step(ev):
        if ev is None:  # under graph capture: no timing events inside the graph
            ev = [_NoEvent()] * nev
        ev[0].record(stream)
        if args.scorer == "actkv":  # both scoring passes, then the LRFU step, in "score_alpha"
            cp.score_action(case.q, sp.scale)
            ev[1].record(stream)
            cp.lrfu(0.9, 0.5)
        else:
            cp.score_lse(case.q, sp.scale, want_lse=args.am_sweeps > 0)
            ev[1].record(stream)
            cp.score_alpha(case.q, sp.scale)
        ev[2].record(stream)
        cp.select()
        ev[3].record(stream)
        if args.am_sweeps > 0:
            # the scoring LSE pass's rows are the fit's (the action scorer writes none)
            cp.am_fit(case.q, sp.scale, args.am_sweeps, lse=None if args.scorer == "actkv" else cp.lse)
        ev[4].record(stream)
        if args.variant == "inplace":
            cp.plan_compact()
            ev[5].record(stream)
            cp.compact()
            ev[6].record(stream)
            cp.free_pages()
        elif args.variant == "fresh":
            fplan = cp.plan_fresh()
            ev[5].record(stream)
            cp.compact(plan=fplan)
            ev[6].record(stream)
            cp.commit_fresh()
        else:  # sentinel: the whole layout step is the "compact" stage
            ev[5].record(stream)
            cp.evict_sentinel()
            ev[6].record(stream)
        ev[7].record(stream)

    for _ in range(args.warmup):
        case.restore(snap)
        step([torch.cuda.Event(enable_timing=True) for _ in range(nev)])
    torch.cuda.synchronize()
    assert kvc.kvc_read_device_status(clear=True) == 0

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    kvc.kvc_launch_count(reset=True)
    w0 = time.time()
    for k in range(args.steps):
        case.restore(snap)  # outside the step's events
        step(events[k])
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    w1 = time.time()
    launches = kvc.kvc_launch_count()
    status = kvc.kvc_read_device_status(clear=True)
    assert status == 0, f"device status {status:#x}"
    per_step = [events[k][0].elapsed_time(events[k][nev - 1]) for k in range(args.steps)]
    per_stage = {s: statistics.mean(events[k][i].elapsed_time(events[k][i + 1])
                                    for k in range(args.steps)) for i, s in enumerate(stages)}
    ms = slowest_rank_ms(statistics.mean(per_step), world, dev)

    # The same step captured once into a CUDA graph (its kernels become graph nodes; the
    # library's calls validate and build their launch parameters on the host once, at
    # capture) and replayed: the step a serving loop would issue.  Each replay runs every
    # kernel of the step; the cache is restored between replays, outside the events.
    graph_ms, graph_nodes = None, 0
    if not args.no_graph:
        g = torch.cuda.CUDAGraph()
        case.restore(snap)
        torch.cuda.synchronize()
        before = kvc.kvc_launch_count()
        with torch.cuda.graph(g):
            step(None)
        graph_nodes = kvc.kvc_launch_count() - before
        for _ in range(args.warmup):
            case.restore(snap)
            g.replay()
        torch.cuda.synchronize()
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        if world > 1:
            dist.barrier()
        for k in range(args.steps):
            case.restore(snap)
            gev[k][0].record(stream)
            g.replay()
            gev[k][1].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        w1 = time.time()
        status = kvc.kvc_read_device_status(clear=True)
        assert status == 0, f"device status {status:#x} (graph replays)"
        graph_ms = slowest_rank_ms(statistics.mean(a.elapsed_time(b) for a, b in gev), world, dev)
        launches = graph_nodes * args.steps
    if clocks:
        time.sleep(0.15)
        clocks.stop()

    # algorithmic work of the step
    plan_used = cp.fresh_plan if args.variant == "fresh" else cp.plan
    moves = int(plan_used.move_count[:sp.L * sp.H * sp.B].sum().item()) if cp.Mtot else 0
    R, d = sp.R, sp.d
    F_alg = 2.0 * R * d * entries  # one Q K^T contraction (each pass executes it once)
    Xp = sum(((min(a, b) + sp.P - 1) // sp.P) * sp.P for a, b in zip(m, n))
    Mtot = sum(min(a, b) for a, b in zip(m, n))
    units = sp.L * sp.H * sum(1 for x in n if x > 0)
    B_alg = (2.0 * d * entries + 2.0 * R * d * units + 12.0 * entries + 4.0 * sp.L * sp.H * Mtot
             + moves * 8.0 * d + 4.0 * sp.L * sp.H * Xp)
    pk = peaks()
    t_roof = max(F_alg / (pk["bf16_tflops"] * 1e12), B_alg / (pk["hbm_gbs"] * 1e9))

    # dominant kernel: the longer scoring pass (each is one persistent kernel; the LSE stage also
    # runs a small combine kernel)
    dom = max(("score_lse", "score_alpha"), key=lambda s: per_stage[s])
    dom_kernel = ("score_pass_kernel<128,2> (alpha pass)" if dom == "score_alpha"
                  else "score_pass_kernel<128,1> (LSE pass)")
    t_dom = per_stage[dom] * 1e-3
    if args.scorer == "actkv":
        # the "score_lse" stage holds both passes of the action attention: time them as one
        # pass each (half the stage) against one Q K^T each
        dom, dom_kernel = "score_lse", "score_pass_kernel<128,1>+<128,2> (action attention, per pass)"
        t_dom = per_stage["score_lse"] * 1e-3 / 2.0
    # a pass reads every K row once and its Q group(s); the alpha pass also writes the scores.
    # The pass is bound by whichever of its flops (at the bf16 peak) or bytes (at the copy
    # peak) takes longer.
    B_pass = 2.0 * d * entries + 2.0 * R * d * units + (4.0 * entries if dom == "score_alpha" else 0.0)
    if F_alg / (pk["bf16_tflops"] * 1e12) >= B_pass / (pk["hbm_gbs"] * 1e9):
        achieved = F_alg / t_dom / 1e12
        roofline = {"bound": "tensor", "kernel": dom_kernel, "achieved": achieved,
                    "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"]}
    else:
        achieved = B_pass / t_dom / 1e9
        roofline = {"bound": "hbm", "kernel": dom_kernel, "achieved": achieved,
                    "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                    "tensor_frac": F_alg / t_dom / 1e12 / pk["bf16_tflops"]}
    roofline.update({"traffic": profile_traffic(dom_kernel, sp.name), "peak_source": pk["source"],
                     "algorithmic_flops_per_launch": F_alg, "algorithmic_bytes_per_launch": B_pass})
    if args.am_sweeps > 0:
        # Attention Matching dominates the step, timed as one stage.  Its roofline time is the
        # sum of each part at the rate it can run on this GPU: the targets at the bf16 tensor
        # peak; the fp32-accurate Gram products as SPLIT_PRODUCTS bf16 products each at the same
        # peak (three tf32 products at half the rate cost the same); the descents and compact
        # probabilities at the fp32 FMA peak of the CUDA cores.  "achieved" is the bf16-equivalent
        # rate, so frac = t_roof / t_stage.
        F_tc, F_gram, F_fp = am_flops(sp, n, m, args.am_sweeps)
        t_am = per_stage["am_fit"] * 1e-3
        bf = pk["bf16_tflops"] * 1e12
        fp_peak = fp32_peak_tflops()
        t_am_roof = (F_tc + SPLIT_PRODUCTS * F_gram) / bf + F_fp / (fp_peak * 1e12)
        t_roof += t_am_roof  # the step: the token-eviction chain's bound plus the fit's
        roofline = {"bound": "tensor", "kernel": "kvc_am_fit (one stage: tensor-core targets and Gram "
                                                 "products, fp32 descents)",
                    "achieved": t_am_roof * pk["bf16_tflops"] / t_am, "peak": pk["bf16_tflops"],
                    "unit": "TFLOP/s", "frac": t_am_roof / t_am, "traffic": None,
                    "peak_source": pk["source"] + "; Gram products counted as %d bf16 products; fp32 "
                                   "part against the derived 152 SMs x 128 FMA/clk x 2 x 2070 MHz = "
                                   "%.1f TFLOP/s" % (SPLIT_PRODUCTS, fp_peak),
                    "algorithmic_flops_per_launch": F_tc + F_gram + F_fp, "targets_flops": F_tc,
                    "gram_flops": F_gram, "fp32_flops": F_fp, "t_roof_ms": t_am_roof * 1e3}
    if args.variant == "sentinel":  # evicted rows written: K and V rows (2d bytes each) and a tag
        compact_bytes = (entries - sp.L * sp.H * Mtot) * (4.0 * d + 4.0)
    else:
        compact_bytes = moves * 8.0 * d + 4.0 * moves
    gbs = compact_bytes / (per_stage["compact"] * 1e-3) / 1e9 if per_stage["compact"] > 0 else 0.0

    line = {
        "metric": METRIC, "value": job_throughput(entries, world, graph_ms or ms), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": graph_ms or ms,
        "ms_per_step_eager": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(sp), "entries_per_step": entries,
                   "l2": "inputs larger than L2 (pools %.1f GB); cache restored from a device "
                         "snapshot between steps, outside the timed events"
                         % (2 * case.k_pool.numel() * 2 / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "eviction_layout": args.variant, "eviction_score": args.scorer,
                   "attention_matching_sweeps": args.am_sweeps,
                   "launch": (f"CUDA graph of the step ({graph_nodes} kernel nodes), replayed"
                              if graph_ms is not None else "eager C-ABI calls")},
        "roofline": roofline,
        "step_roofline": {"t_roof_ms": t_roof * 1e3, "frac": t_roof / ((graph_ms or ms) * 1e-3),
                          "F_alg": F_alg, "B_alg": B_alg, "moves": moves},
        "stages_ms": per_stage,
        "compact_gbs": gbs,
        "gpu_launches": launches,
        "wall_s_timed_region": w1 - w0,
    }
    if clocks:
        line["clocks"] = clocks.summary(w0, w1)

    # the end-to-end and CPU-baseline legs measure the default in-place chain only
    if not args.no_e2e and args.variant == "inplace" and args.scorer == "te" and args.am_sweeps == 0:
        line["e2e"] = e2e_run(args, case, cp, snap, entries, world, dev)
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and args.variant == "inplace"
            and args.scorer == "te" and args.am_sweeps == 0):
        case.restore(snap)  # the oracle reads the pristine cache
        torch.cuda.synchronize()
        line["cpu_baseline"] = cpu_baseline(case, budgets_oracle(case))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def e2e_run(args, case, cp, snap, entries, world, dev):
    """Same metric end to end through the public API with host buffers: every step copies the
    cache and proxy queries from pinned host memory to the device, runs the five calls, and reads
    the selection and the updated bookkeeping (tags, block table, block counts, free stack) back
    into pinned host memory.  When the inputs are large (over 64 MiB: the copy dominates) two
    device copies of the cache alternate between steps, so the copy of step k + 1's inputs (on a
    copy stream) runs while step k computes; small steps run one after another on one stream
    (the second stream's events would cost more than they hide).  Every step's copies in and
    out lie inside the timed region."""
    import torch
    import torch.distributed as dist

    import online_kv_cache_gb300 as kvc

    sp = case.spec
    ins = snap + [case.q]
    h_in = [t.cpu().pin_memory() for t in ins]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    pipelined = h2d > (64 << 20)
    slots = []
    for k in range(2 if pipelined else 1):
        if k == 0:
            dev_ins, c = case.state() + [case.q], cp
        else:  # a second device copy of the cache, with its own compactor
            dev_ins = [t.clone() for t in case.state()] + [case.q.clone()]
            c = kvc.Compactor(*dev_ins[:7], case.seg_start, case.seg_end, case.seq_len, cp.m, sp.R)
        outs = [c.keep, dev_ins[2], dev_ins[3], dev_ins[4], dev_ins[5], dev_ins[6]]
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        slots.append((dev_ins, c, outs, h_out))
    d2h = sum(t.numel() * t.element_size() for t in slots[0][3])
    steps = args.e2e_steps or max(3, min(args.steps, 50))
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    freed = [None, None]

    def run(n):
        for k in range(n):
            dev_ins, c, outs, h_out = slots[k % len(slots)]
            if not pipelined:
                for d_t, h_t in zip(dev_ins, h_in):
                    d_t.copy_(h_t, non_blocking=True)
                c.run(dev_ins[7], sp.scale)
                for h_t, d_t in zip(h_out, outs):
                    h_t.copy_(d_t, non_blocking=True)
                continue
            with torch.cuda.stream(copy_stream):
                if freed[k % 2] is not None:  # step k - 2 is done with this copy
                    copy_stream.wait_event(freed[k % 2])
                for d_t, h_t in zip(dev_ins, h_in):
                    d_t.copy_(h_t, non_blocking=True)
                copied = torch.cuda.Event()
                copied.record(copy_stream)
            stream.wait_event(copied)
            c.run(dev_ins[7], sp.scale)
            for h_t, d_t in zip(h_out, outs):
                h_t.copy_(d_t, non_blocking=True)
            done = torch.cuda.Event()
            done.record(stream)
            freed[k % 2] = done

    run(max(2, args.warmup))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    run(steps)
    stream.wait_stream(copy_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = slowest_rank_ms(e0.elapsed_time(e1) / steps, world, dev)
    return {"value": job_throughput(entries, world, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "pipeline": ("two device copies of the cache: step k + 1's host-to-device copy overlaps step k"
                         if pipelined else "none (inputs of 64 MiB or less: steps in sequence on one stream)"),
            "read_back": ("keep sets, tags, block table, nblocks and free stack; the compacted K/V pools "
                          "stay in device memory by design (the cache is compacted for the decoding that "
                          "follows on the same GPU)")}


def cpu_baseline(case, m):
    """The oracle as it stands on the host cores, on a bounded sample (~10-30 s of CPU work)."""
    sp = case.spec
    cores = host_cores()
    # calibrate with one layer, then size the sample to ~15 s
    dt1, e1, _ = oracle_sample(case, m, 1, cores)
    per_layer = dt1
    layers = max(1, min(sp.L, int(15.0 / max(per_layer, 1e-3))))
    if layers > 1:
        dt_s, entries, used = oracle_sample(case, m, layers, cores)
    else:
        dt_s, entries, used = dt1, e1, max(1, min(cores, sp.H))
    out = {"value": entries / dt_s, "unit": UNIT, "cores": used, "kind": "oracle",
           "sample": f"{layers} of {sp.L} layers x {sp.H} KV heads ({entries} entries): fp64 "
                     f"score + select + compact + free, {dt_s:.1f} s",
           "host_cores": cores}
    # the same oracle on one thread, on one layer when that takes at most ~30 s
    used1 = max(1, min(cores, sp.H * sum(1 for a, b in zip(case.seg_start, case.seg_end) if b > a)))
    if dt1 * used1 <= 30.0:
        dts, es, _ = oracle_sample(case, m, 1, 1)
        out["single_thread"] = {"value": es / dts, "unit": UNIT, "cores": 1,
                                "sample": f"1 of {sp.L} layers x {sp.H} KV heads ({es} entries), {dts:.1f} s"}
    else:
        out["single_thread"] = {"value": None, "skipped": f"one layer would take ~{dt1 * used1:.0f} s on one thread"}
    return out


def main():
    args = parse_args()
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        reference_arm(args)
        return
    our_arm(args)


if __name__ == "__main__":
    main()
