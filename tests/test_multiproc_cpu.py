"""The N > 1 path on CPU: two gloo ranks, as bench.py runs them under torchrun.

Every rank owns an independent seeded batch (replicas, weak scaling); the only
cross-rank traffic is the step-time maximum and the work sums of the timing
line. No GPU is used: the scheduler is host code and the reductions run over
gloo on 127.0.0.1.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import paged_kv_attention_unified_gb300 as ua
        case = bench.rank_case(1, rank)
        raw = case.raw()
        cu = [int(x) for x in raw["cu_query_lens"]]
        kv = [int(x) for x in raw["kv_lens"]]
        info, pre, dec, grp = ua.ua_schedule(cu, kv, case.num_q_heads, case.num_kv_heads,
                                             case.head_dim, case.block_size,
                                             int(raw["block_tables"].shape[1]))
        rows = sum(t["nrows"] for t in pre) + sum(t["nrows"] for t in dec
                                                  if t["slot"] < 0 or t["kv_lo"] == 0)
        byts, flops = bench.algorithmic_work(case)
        step_ms = 1.0 + rank              # stand-in per-rank timings
        ms_max = bench.max_over_ranks(step_ms, world)
        job_bytes = bench.sum_over_ranks(byts, world)
        job_flops = bench.sum_over_ranks(flops, world)
        results[rank] = dict(first_q=float(raw["q"].flatten()[0]), rows=rows,
                             expect_rows=(cu[-1]) * case.num_q_heads, byts=byts, flops=flops,
                             ms_max=ms_max, job_bytes=job_bytes, job_flops=job_flops,
                             num_tiles=int(info.num_prefill_tiles + info.num_decode_tiles))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert sorted(res) == [0, 1]
    # independent batches: different seeds, different data
    assert res[0]["first_q"] != res[1]["first_q"]
    for r in res.values():
        # every (token, query head) row of the rank's own batch is scheduled once
        assert r["rows"] == r["expect_rows"]
        assert r["num_tiles"] > 0
        # the reductions: slowest rank's time, summed work
        assert r["ms_max"] == 2.0
        assert r["job_bytes"] == res[0]["byts"] + res[1]["byts"]
        assert r["job_flops"] == res[0]["flops"] + res[1]["flops"]


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class Args:
        workload = 1
        steps = 1
        warmup = 3
        gpus = 2

    assert bench.run_reference(Args()) == 0
    assert capsys.readouterr().out == ""


def _reference_line(*extra):
    import json
    import subprocess
    import sys
    env = dict(os.environ, RANK="0")
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "1", "--steps", "1", "--warmup", "3", *extra],
                          capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert proc.returncode == 0, proc.stderr[-2000:]
    lines = [l for l in proc.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, proc.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("op", ["attention", "append"])
def test_reference_arm_rank0_prints_one_contract_line(op):
    """Rank 0 of the reference arm times the oracle on the host (no GPU) and
    prints the contract line: the same metric keys as the CUDA arm, with
    cpu_baseline describing the run and a zero-copy e2e."""
    d = _reference_line("--op", op)
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "config"):
        assert k in d, k
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
