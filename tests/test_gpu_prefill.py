"""GPU parity of the tcgen05 prefill path (through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_attention_unified_gb300 as ua
from paged_kv_attention_unified_gb300 import torch_utils as tu
import workloads as W

from _helpers import as_f64, assert_close, oracle_full, oracle_full_parallel

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_unified_gb300 import build
    build.build()


def _check(case, decode_rows_max=0, num_splits=0):
    """decode_rows_max=0 sends every sequence the prefill kernel can take to it."""
    b = tu.to_device(case)
    with tu.make_plan(b, num_splits=num_splits, decode_rows_max=decode_rows_max) as plan:
        assert plan.info.num_prefill_tiles > 0
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    return assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)


def test_single_tile_prefill():
    _check(W.make_case("one_tile", [100], [100], 1, 1, 128, 16, seed=1))


def test_tiny_mixed_config_through_prefill():
    _check(W.config1_tiny_mixed(), decode_rows_max=4)


@pytest.mark.parametrize("qpk,hkv", [(1, 2), (2, 2), (4, 2), (8, 1), (16, 1)])
def test_random_gqa(qpk, hkv):
    _check(W.random_small_case(200 + qpk, head_dim=128, num_q_heads=qpk * hkv,
                               num_kv_heads=hkv, max_kv=700, max_seqs=4))


@pytest.mark.parametrize("bs", [16, 32, 64, 128, 256])
def test_block_sizes(bs):
    _check(W.make_case(f"bs{bs}", [300, 77, 1], [300, 500, 40], 8, 2, 128, bs, seed=bs))


def test_head_dim_64():
    _check(W.random_small_case(230, head_dim=64, num_q_heads=8, num_kv_heads=2, max_kv=800))
    _check(W.make_case("d64_long", [700], [1500], 4, 4, 64, 16, seed=231))


def test_window_and_noncausal():
    _check(W.make_case("win", [400, 260], [900, 260], 8, 2, 128, 16, window=150, seed=240))
    _check(W.make_case("win128", [300], [800], 4, 4, 128, 128, window=200, seed=241))
    _check(W.make_case("noncausal", [200, 90], [600, 90], 8, 2, 128, 16, causal=False, seed=242))


def test_nan_poisoned_padding_never_leaks():
    _check(W.make_case("poison", [333, 150], [700, 181], 8, 2, 128, 16, poison=True, seed=250))
    _check(W.make_case("poison128", [333], [459], 4, 4, 128, 128, poison=True, seed=251))


def test_dense_causal_small():
    _check(W.make_case("dense", [1024, 1024], [1024, 1024], 4, 4, 128, 128, table="identity",
                       seed=260))


def test_mixed_prefill_and_decode_in_one_plan():
    case = W.make_case("mixed", [1, 600, 1, 1, 37, 900], [3000, 1400, 70, 5000, 37, 900], 16, 4,
                       128, 16, seed=270)
    _check(case, decode_rows_max=32)


def test_more_tiles_than_ctas_and_repeated_forwards():
    """320 prefill tiles for at most one CTA per SM: CTAs run several tiles in
    a row (rings and barrier phases carry over), and the tile queue re-arms
    between forwards, so three forwards on one plan give the same bits."""
    rng = np.random.default_rng(280)
    ql = [64] * 40
    kv = [64 + int(c) for c in rng.integers(0, 300, 40)]
    case = W.make_case("many_tiles", ql, kv, 32, 8, 128, 16, seed=280)
    b = tu.to_device(case)
    with tu.make_plan(b, decode_rows_max=0) as plan:
        info = plan.info
        assert info.num_prefill_tiles == 320
        assert info.num_prefill_ctas == min(info.num_sms, 320)
        outs = []
        for _ in range(3):
            outs.append(tu.forward(plan, b))
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert_close(as_f64(outs[0]), oracle_full(case), case.kv_dtype, case.name)


def test_block_permutation_gives_identical_bits():
    case = W.make_case("perm", [500, 200], [800, 333], 8, 2, 128, 16, seed=280)
    b = tu.to_device(case)
    with tu.make_plan(b, decode_rows_max=0) as plan:
        a = tu.forward(plan, b).cpu()
    nb = case.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    k2, v2 = torch.empty_like(case.k_cache), torch.empty_like(case.v_cache)
    k2[inv] = case.k_cache
    v2[inv] = case.v_cache
    case2 = W.Case(**{**case.__dict__, "k_cache": k2, "v_cache": v2,
                      "block_tables": inv[case.block_tables.long()].to(torch.int32)})
    b2 = tu.to_device(case2)
    with tu.make_plan(b2, decode_rows_max=0) as plan:
        c = tu.forward(plan, b2).cpu()
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_full_size_dense_prefill_whole_output_and_first_row_exact():
    """The dense causal prefill workload in the benchmark's launch
    configuration: every element against the fp64 oracle, and row 0 of every
    (sequence, head) -- which sees key 0 alone -- equal to V[0] bit for bit."""
    case = W.config4_dense_prefill()
    got = tu.run(case)
    for s in range(case.num_seqs):
        page = int(case.block_tables[s, 0])
        for h in range(case.num_q_heads):
            assert torch.equal(got[4096 * s, h].view(torch.int16),
                               case.v_cache[page, 0, h].view(torch.int16))
    got = as_f64(got)
    torch.cuda.empty_cache()
    exp = oracle_full_parallel(case)
    assert_close(got, exp, case.kv_dtype, f"workload 4 ({case.name})", report=True)


def test_full_size_mixed_config_whole_output():
    case = W.config3_mixed()
    got = as_f64(tu.run(case))
    torch.cuda.empty_cache()
    exp = oracle_full_parallel(case)
    assert_close(got, exp, case.kv_dtype, f"workload 3 ({case.name})", report=True)


def test_bounded_wait_reports_timeout_and_context_survives():
    """The producer is told to issue nothing: every consumer wait runs out
    after 50 ms, the kernel records UA_ERR_DEVICE_TIMEOUT and exits; the same
    plan then runs normally."""
    case = W.make_case("timeout", [256], [256], 4, 4, 128, 16, seed=290)
    b = tu.to_device(case)
    with tu.make_plan(b, decode_rows_max=0) as plan:
        ua.ua_plan_set_debug(plan.handle, 1, 50_000_000)
        tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == ua.UA_ERR_DEVICE_TIMEOUT
        ua.ua_plan_set_debug(plan.handle, 0, 0)
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert_close(as_f64(out), oracle_full(case), W.BF16, "after timeout")


# ---- prefill over an fp8 (e4m3) cache: staged to bf16, then the tcgen05 kernel

def _check_fp8(case, decode_rows_max=0):
    b = tu.to_device(case)
    with tu.make_plan(b, decode_rows_max=decode_rows_max) as plan:
        assert plan.info.num_prefill_tiles > 0
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    return assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)


@pytest.mark.parametrize("qpk,hkv,d,bs", [(4, 2, 128, 16), (1, 4, 64, 32), (8, 1, 128, 64),
                                          (2, 2, 128, 128), (1, 2, 64, 256)])
def test_fp8_prefill_matches_oracle(qpk, hkv, d, bs):
    _check_fp8(W.make_case(f"fp8p_{qpk}_{bs}", [300, 77, 150], [300, 500, 460], qpk * hkv, hkv,
                           d, bs, kv_dtype=W.FP8, seed=400 + bs))


def test_fp8_prefill_window_noncausal_and_poison():
    _check_fp8(W.make_case("fp8p_win", [400, 260], [900, 260], 8, 2, 128, 16, window=150,
                           kv_dtype=W.FP8, seed=410))
    _check_fp8(W.make_case("fp8p_nc", [200, 90], [600, 90], 8, 2, 128, 16, causal=False,
                           kv_dtype=W.FP8, seed=411))
    _check_fp8(W.make_case("fp8p_poison", [333, 150], [700, 181], 8, 2, 128, 16, poison=True,
                           kv_dtype=W.FP8, seed=412))


def test_fp8_mixed_batch_prefill_and_decode():
    """Long sequences through the staged prefill, single tokens through the fp8
    decode kernel, in one plan."""
    case = W.make_case("fp8_mixed", [1, 600, 1, 1, 37, 900], [3000, 1400, 70, 5000, 37, 900], 16,
                       4, 128, 16, kv_dtype=W.FP8, seed=420)
    _check_fp8(case, decode_rows_max=32)


def test_full_size_fp8_dense_prefill_whole_output():
    case = W.config6_dense_prefill_fp8()
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        assert plan.info.num_decode_tiles == 0
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    got = as_f64(out)
    del b, out
    torch.cuda.empty_cache()
    exp = oracle_full_parallel(case)
    assert_close(got, exp, case.kv_dtype, f"workload 6 ({case.name})", report=True)


def test_many_ragged_sequences_through_both_kernels():
    """400 sequences: single tokens, short and long prefills with and without
    prior context, one plan, both kernels, the prefill tile queue busy."""
    rng = np.random.default_rng(500)
    ql, kv = [], []
    for i in range(400):
        kind = i % 4
        q = 1 if kind == 0 else int(rng.integers(2, 40)) if kind == 1 else \
            int(rng.integers(40, 400)) if kind == 2 else int(rng.integers(400, 1200))
        ql.append(q)
        kv.append(q + int(rng.integers(0, 600)))
    case = W.make_case("many_seqs", ql, kv, 16, 4, 128, 16, seed=501)
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        info = plan.info
        assert info.num_prefill_tiles > 152 and info.num_decode_tiles > 0
        out = tu.forward(plan, b)
        out2 = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert_close(as_f64(out), oracle_full_parallel(case), case.kv_dtype, case.name, report=True)


# ---- head_dim 192 / 256: the wide prefill kernel (one 128-row query tile, 64-key tiles)

def _check_wide(case, decode_rows_max=0):
    b = tu.to_device(case)
    with tu.make_plan(b, decode_rows_max=decode_rows_max) as plan:
        assert plan.info.num_prefill_tiles > 0
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    return assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("qpk,hkv,bs", [(1, 2, 16), (2, 2, 32), (4, 1, 64), (8, 1, 128),
                                        (4, 2, 16)])
def test_wide_prefill_matches_oracle(qpk, hkv, bs, d):
    """Ragged prefills with contexts that are not multiples of 16 or 64, and a
    query tile that straddles the 128-row item boundary."""
    _check_wide(W.make_case(f"wide_d{d}_{qpk}_{bs}", [300, 77, 129, 1], [300, 533, 200, 90],
                            qpk * hkv, hkv, d, bs, seed=700 + bs + qpk + d))


@pytest.mark.parametrize("d", [192, 256])
def test_wide_prefill_window_noncausal_poison_and_fp8(d):
    _check_wide(W.make_case("wide_win", [400, 260], [900, 260], 8, 2, d, 16, window=150,
                            seed=710 + d))
    _check_wide(W.make_case("wide_nc", [200, 90], [600, 90], 8, 2, d, 32, causal=False,
                            seed=711 + d))
    _check_wide(W.make_case("wide_poison", [333, 150], [700, 181], 8, 2, d, 16, poison=True,
                            seed=712 + d))
    _check_wide(W.make_case("wide_fp8", [300, 77, 150], [300, 500, 460], 8, 2, d, 16,
                            kv_dtype=W.FP8, seed=713 + d))


def test_wide_prefill_mixed_with_decode_and_repeated():
    """Long prefills in the wide prefill kernel and single tokens in the
    head_dim 256 decode kernel, one plan, both grids overlapping; a second
    forward on the same plan gives the same bits."""
    case = W.make_case("wide_mixed", [1, 600, 1, 1, 37, 900], [3000, 1400, 70, 5000, 37, 900],
                       16, 4, 256, 16, seed=720)
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        assert plan.info.num_prefill_tiles > 0 and plan.info.num_decode_tiles > 0
        out = tu.forward(plan, b)
        out2 = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)


def test_wide_prefill_bounded_wait_reports_timeout_and_context_survives():
    case = W.make_case("wide_timeout", [256], [256], 4, 4, 256, 16, seed=730)
    b = tu.to_device(case)
    with tu.make_plan(b, decode_rows_max=0) as plan:
        ua.ua_plan_set_debug(plan.handle, 1, 50_000_000)
        tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == ua.UA_ERR_DEVICE_TIMEOUT
        ua.ua_plan_set_debug(plan.handle, 0, 0)
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert_close(as_f64(out), oracle_full(case), W.BF16, "wide, after timeout")


def test_full_size_wide_dense_prefill_whole_output_and_first_row_exact():
    """Config 4's shape at head_dim 256 through the wide prefill kernel: every
    element against the fp64 oracle, row 0 of every (sequence, head) equal to
    V[0] bit for bit."""
    case = W.config9_dense_prefill_d256()
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        assert plan.info.num_decode_tiles == 0 and plan.info.num_prefill_tiles > 0
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    got = out.cpu()
    for s in range(case.num_seqs):
        page = int(case.block_tables[s, 0])
        for h in range(case.num_q_heads):
            assert torch.equal(got[4096 * s, h].view(torch.int16),
                               case.v_cache[page, 0, h].view(torch.int16))
    del b, out
    torch.cuda.empty_cache()
    assert_close(as_f64(got), oracle_full_parallel(case), case.kv_dtype,
                 f"workload 9 ({case.name})", report=True)


@pytest.mark.parametrize("d", [128, 192, 256])
def test_one_persistent_cta_runs_every_tile_in_turn(d):
    """One prefill CTA takes every work tile of the batch in sequence, so every
    barrier phase, ring position and TMEM buffer runs on across many tiles
    (a waiter that is a phase away from its barrier shows up here)."""
    case = W.make_case(f"one_cta_{d}", [1024] * 4, [1024] * 4, 8, 8, d, 128, table="identity",
                       seed=740 + d)
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        ua.ua_plan_set_prefill_ctas(plan.handle, 1)
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)
