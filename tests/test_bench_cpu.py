"""CPU checks of the benchmark's accounting: the algorithmic bytes and flops
that every roofline fraction divides by, counted here by brute force over
(query row, key) pairs, and the oracle baseline path."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _brute_work(case):
    """Visible (query token, key) pairs and the K/V rows any query reads,
    enumerated one by one from the mask definition."""
    cu = case.cu_query_lens.tolist()
    kv = case.kv_lens.tolist()
    pairs, rows = 0, 0
    for s in range(case.num_seqs):
        ql = cu[s + 1] - cu[s]
        if ql == 0:
            continue
        ctx = kv[s] - ql
        read = set()
        for i in range(ql):
            pos = ctx + i
            for t in range(kv[s]):
                if case.causal and t > pos:
                    continue
                if case.window > 0 and t <= pos - case.window:
                    continue
                pairs += 1
                read.add(t)
        rows += len(read)
    return pairs, rows


@pytest.mark.parametrize("window,causal", [(0, True), (7, True), (0, False), (40, False)])
def test_algorithmic_work_matches_brute_force(window, causal):
    case = W.make_case("acct", [1, 5, 17, 0, 3], [40, 130, 300, 9, 3], 8, 2, 64, 16,
                       window=window, causal=causal, seed=2)
    pairs, rows = _brute_work(case)
    byts, flops = bench.algorithmic_work(case)
    d, hq, hkv = case.head_dim, case.num_q_heads, case.num_kv_heads
    tq = int(case.cu_query_lens[-1])
    pages = sum(-(-k // case.block_size) for q, k in
                zip((case.cu_query_lens[1:] - case.cu_query_lens[:-1]).tolist(),
                    case.kv_lens.tolist()) if q > 0)
    assert flops == 4 * d * hq * pairs
    assert byts == rows * hkv * d * 2 * 2 + 2 * tq * hq * d * 2 + pages * 4 + \
        (2 * case.num_seqs + 1) * 4


def test_fp8_bytes_count_one_byte_per_element():
    case = W.make_case("acct8", [1, 2], [100, 37], 16, 2, 128, 16, kv_dtype=W.FP8, seed=3)
    _, rows = _brute_work(case)
    byts, _ = bench.algorithmic_work(case)
    assert byts == rows * 2 * 128 * 1 * 2 + 2 * 3 * 16 * 128 * 2 + (7 + 3) * 4 + 5 * 4


def test_window_reduces_the_counted_work():
    case = W.CONFIGS[1]()
    full = bench.algorithmic_work(case)
    win = bench.algorithmic_work(bench._with_window(case, 16))
    assert win[0] < full[0] and win[1] < full[1]
    assert bench._with_window(case, 0) is case


def test_oracle_baseline_runs_on_every_host_core():
    rates, cores, sample, raw = bench.oracle_throughput(1, W.CONFIGS[1](), budget_s=0.5,
                                                        rounds=2)
    assert len(rates) == 2 and all(v > 0 for v in rates)
    assert cores == len(os.sched_getaffinity(0)) and "units" in sample
    assert all(b > 0 and f > 0 and t > 0 for b, f, t in raw)


@pytest.mark.parametrize("window", [0, 40])
def test_unit_work_adds_up_to_the_whole_forward(window):
    """The oracle baseline credits each (sequence, KV head) unit with 1/Hkv of
    its sequence's work: over all units that is the whole forward minus the
    length arrays."""
    case = bench._with_window(W.make_case("units", [1, 30, 4], [700, 30, 90], 16, 4, 64, 16,
                                          seed=4), window)
    from oracle import pool
    units = pool.units_of(case.cu_query_lens.tolist(), 4)
    b, f = bench.units_work(case, units)
    tb, tf = bench.algorithmic_work(case)
    assert b == tb - (2 * 3 + 1) * 4 and f == tf


def test_kernel_digest_ignores_comments_but_not_code():
    """The traffic records are keyed by the code of a kernel's sources: a
    comment edit keeps the digest, a code edit changes it, and comment
    markers inside string or character literals are code."""
    from paged_kv_attention_unified_gb300 import build as B
    src = 'int a = 1; // note\n/* block\n note */ const char* s = "x // y /* z */"; char q = \'"\';'
    got = B._strip_comments(src)
    assert "note" not in got and '"x // y /* z */"' in got and "char q = '\"';" in got
    assert B._strip_comments(src.replace("note", "other words")) == got
    assert B._strip_comments(src.replace("a = 1", "a = 2")) != got


def test_traffic_records_belong_to_one_launch_configuration():
    """A committed ncu record is reported only for the launch configuration
    it was taken on: a key that no capture wrote (a windowed run, forced
    splits) yields no traffic, and a record whose digest is not the current
    code's yields none either."""
    import json
    import bench
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    assert "decode/workload2ns8" not in records and "decode/workload2win512" not in records
    assert bench._traffic_record("decode", "2ns8")[0] is None
    assert bench._traffic_record("decode", "2win512")[0] is None
    if "decode/workload2win1024" in records and "decode/workload2" in records:
        assert records["decode/workload2win1024"]["bytes_per_launch"] < \
            records["decode/workload2"]["bytes_per_launch"] / 2   # the window reads 41 % of the cache
    for key, rec in records.items():
        if key.startswith("_"):
            continue
        kernel, cfg = key.split("/")
        got, _, digests = bench._traffic_record(kernel, cfg[len("workload"):])
        if digests["current"] == rec["source_hash"]:
            assert got == rec["bytes_per_launch"]
        else:
            assert got is None
