#!/usr/bin/env python
"""Benchmark of the unified paged-KV attention forward on GB300.

One step = one ua_forward over the whole batch of the chosen workload (every
kernel of the path: prefill, split-KV decode, combine). Default workload: the
pure-decode batch (64 sequences, kv_len ~ U[512, 4096], 32 query / 8 KV heads,
head_dim 128, bf16, block_size 16); metric: KV-read GB/s (algorithmic bytes:
every visible K/V row once, plus Q, output, page tables and lengths).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
                    [--impl ours|reference]

Under torchrun each rank runs its own independent batch (weak scaling, no
collective on the data path); rank 0 prints one JSON line. `--impl reference`
times the fp64 CPU oracle (the only other implementation of this path) on a
bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024
WORKLOAD_NAMES = {
    1: "tiny mixed batch: 3 seqs, q [1,5,17], kv [40,130,300], 4/4 heads, d64, bf16, bs16",
    2: "pure decode: 64 seqs, q 1, kv U[512,4096], 32/8 heads, d128, bf16, bs16",
    3: "mixed: 8 prefill (q U[512,2048], ctx U[0,1024]) + 120 decode (kv U[1024,8192]), "
       "32/8 heads, d128, bf16, bs16",
    4: "dense causal prefill: 4 seqs x 4096, 32/32 heads, d128, bf16, bs128, identity table",
    5: "long decode fp8: 8 seqs, kv 131072, 64/8 heads, d128, fp8 e4m3 KV, bs16",
    6: "dense causal prefill over an fp8 cache: 4 seqs x 4096, 32/32 heads, d128, fp8 e4m3 KV, "
       "bs16, random table (not a benchmark configuration: measures the fp8 prefill path)",
    7: "uniform decode: 32 seqs, q 1, kv 8192, 32/8 heads, d128, bf16, bs16 (not a benchmark "
       "configuration: measures split sizing on equal lengths)",
    8: "pure decode at head_dim 256: 64 seqs, q 1, kv U[512,4096], 32/8 heads, bf16, bs16 "
       "(not a benchmark configuration: measures the head_dim 256 decode path)",
}
FLOP_CONFIGS = (4, 6)   # prefill-bound workloads, reported in TFLOP/s


def algorithmic_work(case):
    """(bytes, flops) one forward must move / compute, counting every visible
    K/V row once per KV head, Q and the output once, the used page-table
    entries and the length arrays; flops = 4 * d per (query head, visible key)."""
    cu = case.cu_query_lens.tolist()
    kvl = case.kv_lens.tolist()
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    d, hq, hkv = case.head_dim, case.num_q_heads, case.num_kv_heads
    kv_rows = 0
    vis_pairs = 0
    pages = 0
    for s in range(case.num_seqs):
        ql, kv = cu[s + 1] - cu[s], kvl[s]
        if ql == 0:
            continue
        ctx = kv - ql
        lo = max(0, ctx - case.window + 1) if case.window > 0 else 0
        kv_rows += kv - lo
        pages += -(-kv // case.block_size)
        for i in range(ql):
            pos = ctx + i
            hi = pos + 1 if case.causal else kv
            l0 = max(0, pos - case.window + 1) if case.window > 0 else 0
            vis_pairs += hi - l0
    tq = cu[-1]
    byts = (kv_rows * hkv * d * elt * 2 + 2 * tq * hq * d * 2 + pages * 4 +
            (2 * case.num_seqs + 1) * 4)
    flops = 4 * d * hq * vis_pairs
    return byts, flops


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region (read only)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline; never on the GPU path)
# ---------------------------------------------------------------------------

def _oracle_worker(cfg, budget_s, seq_limit, window=0):
    """Spawned process, one thread: draw the workload, then run the fp64
    oracle sequence by sequence until budget_s of compute has been spent.
    Returns (sequences done, compute seconds)."""
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    import oracle
    import workloads as W
    case = _with_window(W.CONFIGS[cfg](), window)
    r = case.raw()
    cu = r["cu_query_lens"]
    done, spent = [], 0.0
    for s in range(case.num_seqs):
        if spent >= budget_s or len(done) >= seq_limit:
            break
        t0 = time.perf_counter()
        oracle.paged_attention(r["q"][cu[s]:cu[s + 1]], r["k_cache"], r["v_cache"],
                               [0, int(cu[s + 1] - cu[s])], r["kv_lens"][s:s + 1],
                               r["block_tables"][s:s + 1], case.block_size, case.scale,
                               kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                               v_scale=case.v_scale, causal=case.causal, window=case.window)
        spent += time.perf_counter() - t0
        done.append(s)
    return done, spent


def _seq_subcase(case, seqs):
    """A view of `case` restricted to the given sequences (for work counting)."""
    import torch
    import workloads as W
    cu = case.cu_query_lens.tolist()
    qlens = [cu[s + 1] - cu[s] for s in seqs]
    new_cu = [0]
    for q in qlens:
        new_cu.append(new_cu[-1] + q)
    return W.Case(name=case.name, q=case.q[:0], k_cache=case.k_cache[:1], v_cache=case.v_cache[:1],
                  cu_query_lens=torch.tensor(new_cu, dtype=torch.int32),
                  kv_lens=case.kv_lens[list(seqs)], block_tables=case.block_tables[list(seqs)],
                  num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads,
                  head_dim=case.head_dim, block_size=case.block_size, kv_dtype=case.kv_dtype,
                  scale=case.scale, k_scale=case.k_scale, v_scale=case.v_scale,
                  causal=case.causal, window=case.window)


def oracle_throughput(cfg, case, budget_s=12.0, seq_limit=1 << 30):
    """Time the oracle (one process, one thread) on whole sequences of the
    workload for about budget_s; returns (GB/s, cores, sample description)."""
    import concurrent.futures
    import multiprocessing as mp
    with concurrent.futures.ProcessPoolExecutor(
            max_workers=1, mp_context=mp.get_context("spawn")) as ex:
        done, spent = ex.submit(_oracle_worker, cfg, budget_s, seq_limit, case.window).result()
    byts, _ = algorithmic_work(_seq_subcase(case, done))
    sample = (f"{len(done)} of {case.num_seqs} sequences (all heads) of the same workload, "
              f"{spent:.1f} s of single-thread compute")
    return byts / spent / 1e9, 1, sample


def _oracle_steps_worker(cfg, steps, step_budget_s, window=0):
    """Spawned process, one thread: `steps` timed oracle steps, each a run
    over consecutive sequences (cycling) lasting about step_budget_s.
    Returns [(sequence list, seconds)] per step."""
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    import oracle
    import workloads as W
    case = _with_window(W.CONFIGS[cfg](), window)
    r = case.raw()
    cu = r["cu_query_lens"]
    out, s = [], 0
    for _ in range(steps):
        seqs, spent = [], 0.0
        while spent < step_budget_s and len(seqs) < case.num_seqs:
            t0 = time.perf_counter()
            oracle.paged_attention(r["q"][cu[s]:cu[s + 1]], r["k_cache"], r["v_cache"],
                                   [0, int(cu[s + 1] - cu[s])], r["kv_lens"][s:s + 1],
                                   r["block_tables"][s:s + 1], case.block_size, case.scale,
                                   kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                                   v_scale=case.v_scale, causal=case.causal,
                                   window=case.window)
            spent += time.perf_counter() - t0
            seqs.append(s)
            s = (s + 1) % case.num_seqs
        out.append((seqs, spent))
    return out


def _metric_for(cfg):
    if cfg in FLOP_CONFIGS:
        return "prefill TFLOP/s (algorithmic causal flops / step time)", "TFLOP/s"
    return "decode KV-read GB/s (algorithmic K/V+Q+O bytes / step time)", "GB/s"


def _dtype_for(case):
    return "fp8e4m3 KV -> f16 MMA, fp32 accumulate" if case.kv_dtype == "fp8_e4m3" else \
        "bf16 MMA, fp32 accumulate"


def _rate(cfg, byts, flops, seconds):
    return (flops / seconds / 1e12) if cfg in FLOP_CONFIGS else (byts / seconds / 1e9)


# ---- replicas across ranks (weak scaling: an independent batch per GPU) ----

def _with_window(case, window):
    """The workload with a left sliding window of `window` keys (0: none)."""
    return dataclasses.replace(case, window=int(window)) if window else case


def rank_case(cfg, rank):
    """This rank's batch: the workload drawn with seed = rank."""
    import workloads as W
    return W.CONFIGS[cfg](seed=rank)


def max_over_ranks(value, world, device="cpu"):
    """Largest value over the ranks (the job's step time is its slowest rank's)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, world, device="cpu"):
    """Sum over the ranks (work units the whole job processed)."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def run_reference(args):
    """The oracle as the reference arm: host cores only, rank 0 only."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import workloads as W
    import concurrent.futures
    import multiprocessing as mp
    cfg = args.workload
    case = _with_window(W.CONFIGS[cfg](), getattr(args, "window", 0))
    metric, unit = _metric_for(cfg)
    step_budget = max(0.5, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    if getattr(args, "op", "attention") == "append":
        return _reference_append(args, case, step_budget)
    with concurrent.futures.ProcessPoolExecutor(
            max_workers=1, mp_context=mp.get_context("spawn")) as ex:
        res = ex.submit(_oracle_steps_worker, cfg, args.warmup + args.steps, step_budget,
                        case.window).result()
    timed = res[args.warmup:]
    tot_b = tot_f = tot_t = 0.0
    for seqs, secs in timed:
        b, f = algorithmic_work(_seq_subcase(case, seqs))
        tot_b, tot_f, tot_t = tot_b + b, tot_f + f, tot_t + secs
    value = _rate(cfg, tot_b, tot_f, tot_t)
    sample = (f"each step: consecutive whole sequences (all heads) of the workload for about "
              f"{step_budget:.1f} s of single-thread fp64 compute")
    line = {
        "impl": "reference", "metric": metric, "value": value, "unit": unit,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(1, len(timed)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
        "data": "synthetic (seeded N(0,1))",
        "config": {"workload": WORKLOAD_NAMES[cfg], "parallelism": "host, 1 thread",
                   **({"window": case.window} if case.window else {})},
        "cpu_baseline": {"value": value, "unit": unit, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _traffic_record(kernel: str, cfg: int):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources (profiles/traffic.json: {key: {"source_hash", "bytes"}})."""
    try:
        from paged_kv_attention_unified_gb300 import build as B
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(f"{kernel}/workload{cfg}")
        if rec and rec.get("source_hash") == B._digest():
            return float(rec["bytes_per_launch"]), rec.get("note")
    except Exception:
        pass
    return None, None


def run_ours(args):
    import torch
    import torch.distributed as dist
    import workloads as W
    import paged_kv_attention_unified_gb300 as ua
    from paged_kv_attention_unified_gb300 import build as B
    from paged_kv_attention_unified_gb300 import torch_utils as tu

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    B.build()
    cfg = args.workload
    case = _with_window(rank_case(cfg, rank), args.window)   # weak scaling: one batch per GPU
    byts, flops = algorithmic_work(case)
    metric, unit = _metric_for(cfg)
    hbm_peak, tf_peak, peak_src = _peaks()

    # CPU baseline first (spawned process, before the timed GPU region).
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_throughput(cfg, case, budget_s=args.cpu_budget)
        if cfg in FLOP_CONFIGS:
            v = v / max(byts, 1) * flops / 1e3  # GB/s -> TFLOP/s on the same sample mix
        cpu = {"value": v, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample}

    b = tu.to_device(case)
    plan = tu.make_plan(b, num_splits=args.num_splits)
    plan.set_unified_max(args.unified_max)
    info = plan.info
    out = b.new_out()
    stream = torch.cuda.current_stream()
    ua.ua_plan_set_profiling(plan.handle, True)
    for _ in range(args.warmup):
        tu.forward(plan, b, out)
    torch.cuda.synchronize()
    ua.ua_plan_kernel_times(plan.handle)   # discard warm-up timings

    working_set = byts
    flush = None
    if working_set < 2 * L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        if flush is None:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(args.steps):
                tu.forward(plan, b, out)
            t1.record(stream)
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1)
        else:
            ms = 0.0
            for _ in range(args.steps):
                flush.zero_()
                t0 = torch.cuda.Event(enable_timing=True)
                t1 = torch.cuda.Event(enable_timing=True)
                t0.record(stream)
                tu.forward(plan, b, out)
                t1.record(stream)
                torch.cuda.synchronize()
                ms += t0.elapsed_time(t1)
    if world > 1:
        dist.barrier()
    ktimes = ua.ua_plan_kernel_times(plan.handle)
    ms_max = max_over_ranks(ms, world, device="cuda")
    step_s = ms_max / 1e3 / args.steps
    job_bytes = sum_over_ranks(byts, world, device="cuda")
    job_flops = sum_over_ranks(flops, world, device="cuda")
    value = _rate(cfg, job_bytes, job_flops, step_s)

    # dominant kernel and its roofline, credited with the work of the sequences
    # the scheduler gave it (host-only schedule of the same batch)
    kind = max(("prefill", "decode"), key=lambda k: ktimes[k][0])
    kms, kn = ktimes[kind]
    avg_s = kms / 1e3 / max(kn, 1)
    _, pre_t, dec_t, _ = ua.ua_schedule(b.cu_host, b.kv_host, b.num_q_heads, b.num_kv_heads,
                                        b.head_dim, b.block_size, int(b.block_tables.shape[1]),
                                        kv_dtype=b.kv_dtype, causal=b.causal, window=b.window,
                                        num_sms=info.num_sms)
    seqs = sorted({t["seq"] for t in (pre_t if kind == "prefill" else dec_t)})
    k_bytes, k_flops = algorithmic_work(_seq_subcase(case, seqs)) if seqs else (byts, flops)
    if kind == "prefill":
        ach = k_flops / avg_s / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": tf_peak, "unit": "TFLOP/s",
                "frac": ach / tf_peak, "work_per_launch": k_flops}
    else:
        ach = k_bytes / avg_s / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                "frac": ach / hbm_peak, "work_per_launch": k_bytes}
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" \
        else "fallback"
    roof["kernel"] = kind
    roof["kernel_avg_us"] = avg_s * 1e6
    roof["kernel_share"] = kms / max(1e-9, sum(v[0] for v in ktimes.values()))
    traffic, note = _traffic_record(kind, cfg)
    roof["traffic"] = traffic
    if note:
        roof["traffic_note"] = note
    launches = sum(v[1] for v in ktimes.values())

    # end to end through the public API with host buffers, plan included
    e2e = None
    if not args.no_e2e:
        q_h = case.q.pin_memory()
        cu_h = case.cu_query_lens.to(torch.int32).pin_memory()
        kv_h = case.kv_lens.to(torch.int32).pin_memory()
        bt_h = case.block_tables.to(torch.int32).pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        cu_list, kv_list = case.cu_query_lens.tolist(), case.kv_lens.tolist()
        tiles_b = 32 * (info.num_prefill_tiles + info.num_decode_tiles) + \
            32 * info.num_combine_groups + 16
        h2d = q_h.numel() * 2 + cu_h.numel() * 4 + kv_h.numel() * 4 + bt_h.numel() * 4 + tiles_b
        d2h = out_h.numel() * 2
        torch.cuda.synchronize()
        tot = 0.0
        for it in range(args.warmup + args.steps):
            if flush is not None:
                flush.zero_()
                torch.cuda.synchronize()
            t_0 = time.perf_counter()
            b.q.copy_(q_h, non_blocking=True)
            b.cu_query_lens.copy_(cu_h, non_blocking=True)
            b.kv_lens.copy_(kv_h, non_blocking=True)
            b.block_tables.copy_(bt_h, non_blocking=True)
            with tu.make_plan(b, num_splits=args.num_splits) as p2:
                p2.set_unified_max(args.unified_max)
                tu.forward(p2, b, out)
                out_h.copy_(out, non_blocking=True)
                torch.cuda.synchronize()
            if it >= args.warmup:
                tot += time.perf_counter() - t_0
        e2e = {"value": _rate(cfg, byts, flops, tot / args.steps), "unit": unit,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "includes": "H2D of q/lengths/page tables, CPU scheduling + tile upload, "
                           "forward, D2H of the output, per step"}

    plan.close()
    if rank != 0:
        return 0
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": _dtype_for(case),
        "data": "synthetic (seeded N(0,1), random page tables)",
        "config": {"workload": WORKLOAD_NAMES[cfg],
                   "l2": ("inputs larger than L2 (%.2f GB > 0.129 GB)" % (working_set / 1e9))
                   if flush is None else "L2 flushed (256 MB write) between timed steps",
                   "parallelism": "replicas: an independent batch per GPU, no collective",
                   "decode_tiles": info.num_decode_tiles, "prefill_tiles": info.num_prefill_tiles,
                   "split_tokens": info.split_tokens,
                   **({"unified_max": args.unified_max} if args.unified_max is not None else {}),
                   **({"num_splits": args.num_splits} if args.num_splits else {}),
                   **({"window": args.window} if args.window else {})},
        "algorithmic": {"bytes_per_step": byts, "flops_per_step": flops},
        "pct_of_peak": (value / world) / (tf_peak if cfg in FLOP_CONFIGS else hbm_peak),
        "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": int(launches),
        "kernel_ms": {k: v[0] for k, v in ktimes.items()},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def _reference_append(args, case, step_budget):
    """Reference arm of --op append: the oracle's append, rank 0, host cores."""
    import concurrent.futures
    import multiprocessing as mp
    cfg = args.workload
    row = case.num_kv_heads * case.head_dim
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    toks, spent = 0, 0.0
    with concurrent.futures.ProcessPoolExecutor(
            max_workers=1, mp_context=mp.get_context("spawn")) as ex:
        for k in range(args.warmup + args.steps):
            t, sp = ex.submit(_oracle_append_worker, cfg, step_budget).result()
            if k >= args.warmup:
                toks, spent = toks + t, spent + sp
    value = 2 * toks * row * (2 + elt) / spent / 1e9
    sample = (f"each step: the oracle's append over consecutive whole sequences for about "
              f"{step_budget:.1f} s of single-thread work")
    line = {
        "impl": "reference", "metric": "append-KV GB/s (algorithmic new K/V bytes read + cache "
        "bytes written / step time)", "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * spent / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (CPU oracle)", "data": "synthetic (seeded N(0,1))",
        "config": {"workload": WORKLOAD_NAMES[cfg], "op": "append_kv",
                   "parallelism": "host, 1 thread"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---- append-KV (writing the step's new K/V into the paged cache) ----

def append_work(case):
    """Bytes one append moves: the new K and V rows read (bf16) and written
    (cache element size), plus cu_query_lens, kv_lens and one page-table entry
    per new token."""
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    T = int(case.cu_query_lens[-1])
    row = case.num_kv_heads * case.head_dim
    return 2 * T * row * (2 + elt) + 4 * (2 * case.num_seqs + 1) + 4 * T


def _new_kv(case, seed=1):
    import torch
    g = torch.Generator().manual_seed(seed)
    T = int(case.cu_query_lens[-1])
    shape = (T, case.num_kv_heads, case.head_dim)
    return (torch.randn(shape, generator=g).to(torch.bfloat16),
            torch.randn(shape, generator=g).to(torch.bfloat16))


def _oracle_append_worker(cfg, budget_s):
    """Spawned process, one thread: the oracle's append over consecutive
    sequences of the workload for about budget_s. Returns (tokens, seconds)."""
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    import numpy as np
    import oracle
    import workloads as W
    case = W.CONFIGS[cfg]()
    r = case.raw()
    kn, vn = _new_kv(case)
    kn = kn.view(__import__("torch").int16).numpy().view(np.uint16)
    vn = vn.view(__import__("torch").int16).numpy().view(np.uint16)
    cu = r["cu_query_lens"]
    toks, spent, s = 0, 0.0, 0
    while spent < budget_s and s < case.num_seqs:
        t0 = time.perf_counter()
        oracle.append_kv(kn[cu[s]:cu[s + 1]], vn[cu[s]:cu[s + 1]], r["k_cache"], r["v_cache"],
                         [0, int(cu[s + 1] - cu[s])], r["kv_lens"][s:s + 1],
                         r["block_tables"][s:s + 1], case.block_size, kv_dtype=case.kv_dtype,
                         k_scale=case.k_scale, v_scale=case.v_scale)
        spent += time.perf_counter() - t0
        toks += int(cu[s + 1] - cu[s])
        s += 1
    return toks, spent


def run_append(args):
    """One step = ua_append_kv of every new token of the workload's batch (the
    q tokens' K and V) into its paged cache; HBM-bound."""
    import torch
    import concurrent.futures
    import multiprocessing as mp
    import paged_kv_attention_unified_gb300 as ua
    from paged_kv_attention_unified_gb300 import build as B
    from paged_kv_attention_unified_gb300 import torch_utils as tu
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    B.build()
    cfg = args.workload
    case = rank_case(cfg, rank)
    byts = append_work(case)
    hbm_peak, _, peak_src = _peaks()
    T = int(case.cu_query_lens[-1])
    row = case.num_kv_heads * case.head_dim
    elt = 1 if case.kv_dtype == "fp8_e4m3" else 2
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        with concurrent.futures.ProcessPoolExecutor(
                max_workers=1, mp_context=mp.get_context("spawn")) as ex:
            toks, spent = ex.submit(_oracle_append_worker, cfg, args.cpu_budget).result()
        cpu_b = 2 * toks * row * (2 + elt)
        cpu = {"value": cpu_b / spent / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{toks} of {T} new tokens (whole sequences), {spent:.1f} s of "
                         "single-thread fp64-oracle work"}
    b = tu.to_device(case)
    kn, vn = (t.cuda() for t in _new_kv(case))
    plan = tu.make_plan(b)
    ua.ua_plan_set_profiling(plan.handle, True)
    for _ in range(args.warmup):
        tu.append_kv(plan, b, kn, vn)
    torch.cuda.synchronize()
    ua.ua_plan_kernel_times(plan.handle)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    ms = 0.0
    with ClockSampler(torch.cuda.current_device()) as clk:
        for _ in range(args.steps):
            flush.zero_()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            tu.append_kv(plan, b, kn, vn)
            t1.record(stream)
            torch.cuda.synchronize()
            ms += t0.elapsed_time(t1)
    kt = ua.ua_plan_kernel_times(plan.handle)["append"]
    ms_max = max_over_ranks(ms, world, device="cuda")
    job_bytes = sum_over_ranks(byts, world, device="cuda")
    value = job_bytes / (ms_max / 1e3 / args.steps) / 1e9
    avg_s = kt[0] / 1e3 / max(1, kt[1])
    ach = byts / avg_s / 1e9
    roof = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
            "frac": ach / hbm_peak, "work_per_launch": byts, "kernel": "append",
            "kernel_avg_us": avg_s * 1e6, "kernel_share": 1.0,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured"
            else "fallback",
            "traffic": _traffic_record("append", cfg)[0]}
    # end to end: pinned host K/V rows -> device, append, read the error word
    kh, vh = kn.cpu().pin_memory(), vn.cpu().pin_memory()
    tot = 0.0
    for it in range(args.warmup + args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t_0 = time.perf_counter()
        kn.copy_(kh, non_blocking=True)
        vn.copy_(vh, non_blocking=True)
        tu.append_kv(plan, b, kn, vn)
        err = plan.last_device_error()
        if it >= args.warmup:
            tot += time.perf_counter() - t_0
    assert err == 0
    plan.close()
    if rank != 0:
        return 0
    line = {
        "metric": "append-KV GB/s (algorithmic new K/V bytes read + cache bytes written / step time)",
        "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 -> fp8 e4m3 (x / scale, saturating)" if elt == 1 else "bf16 copy",
        "data": "synthetic (seeded N(0,1), random page tables)",
        "config": {"workload": WORKLOAD_NAMES[cfg], "op": "append_kv", "new_tokens": T,
                   "l2": "L2 flushed (256 MB write) between timed steps",
                   "parallelism": "replicas: an independent batch per GPU, no collective"},
        "algorithmic": {"bytes_per_step": byts},
        "pct_of_peak": (value / world) / hbm_peak,
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": byts / (tot / args.steps) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": int(kh.numel() * 2 * 2), "d2h_bytes_per_step": 4,
                "includes": "H2D of the new K/V rows, append, read of the error word"},
        "gpu_launches": int(kt[1]), "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=2, choices=sorted(WORKLOAD_NAMES))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", default="attention", choices=["attention", "append"],
                    help="attention: the forward step (default); append: ua_append_kv of the "
                         "step's new K/V")
    ap.add_argument("--window", type=int, default=0, metavar="W",
                    help="left sliding window of W keys for the attention step (0: none)")
    ap.add_argument("--num-splits", type=int, default=0, metavar="N",
                    help="cut every decode tile into N split pieces (0: automatic sizing)")
    ap.add_argument("--unified-max", type=float, default=None, metavar="PHI",
                    help="decode rows start from the unified max PHI (scaled-score units) "
                         "instead of their first maximum (off by default)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "append":
        return run_append(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
