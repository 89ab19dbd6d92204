"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle."""
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


def _check(case, num_splits=0, decode_rows_max=-1):
    got = as_f64(tu.run(case, num_splits=num_splits, decode_rows_max=decode_rows_max))
    exp = oracle_full(case)
    return assert_close(got, exp, case.kv_dtype, case.name)


def test_tiny_mixed_config():
    _check(W.config1_tiny_mixed())


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("d", [64, 128])
def test_random_bf16(seed, d):
    hkv = [1, 2, 4][seed % 3]
    hq = hkv * [1, 4, 8, 2, 16, 3][seed]
    _check(W.random_small_case(seed, head_dim=d, num_q_heads=hq, num_kv_heads=hkv,
                               block_size=[16, 32, 128][seed % 3], max_kv=900))


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("d", [64, 128])
def test_random_fp8(seed, d):
    _check(W.random_small_case(100 + seed, kv_dtype=W.FP8, head_dim=d, num_q_heads=8 * (seed + 1),
                               num_kv_heads=seed + 1, max_kv=900))


@pytest.mark.parametrize("ns", [1, 2, 3, 16, 128])
def test_forced_splits_match_oracle(ns):
    case = W.make_case("splits", [1, 1, 3, 1], [3000, 700, 2500, 16], 32, 8, 128, 16, seed=5)
    _check(case, num_splits=ns)


def test_splits_agree_with_unsplit_within_rounding():
    case = W.make_case("splits2", [1, 2], [4000, 1500], 16, 2, 128, 16, seed=6)
    a = as_f64(tu.run(case, num_splits=1))
    for ns in (2, 3, 16, 128):
        b = as_f64(tu.run(case, num_splits=ns))
        assert np.max(np.abs(a - b)) <= 2e-2


def test_window_and_noncausal():
    _check(W.random_small_case(40, head_dim=128, num_q_heads=8, num_kv_heads=2, window=37,
                               max_kv=800))
    _check(W.random_small_case(41, head_dim=64, num_q_heads=4, num_kv_heads=4, causal=False,
                               max_kv=500))
    _check(W.random_small_case(42, kv_dtype=W.FP8, head_dim=128, num_q_heads=16, num_kv_heads=2,
                               window=100, max_kv=800), num_splits=5)


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
def test_nan_poisoned_padding_never_leaks(dtype):
    case = W.random_small_case(50, kv_dtype=dtype, head_dim=128, num_q_heads=8, num_kv_heads=2,
                               max_kv=700, poison=True)
    _check(case)
    _check(case, num_splits=7)


def test_block_permutation_gives_identical_bits():
    case = W.random_small_case(60, head_dim=128, num_q_heads=8, num_kv_heads=2, max_kv=900)
    a = tu.run(case)
    nb = case.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    k2, v2 = torch.empty_like(case.k_cache), torch.empty_like(case.v_cache)
    k2[inv] = case.k_cache
    v2[inv] = case.v_cache
    case2 = W.Case(**{**case.__dict__, "k_cache": k2, "v_cache": v2,
                      "block_tables": inv[case.block_tables.long()].to(torch.int32)})
    b = tu.run(case2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_single_visible_key_is_exact():
    case = W.make_case("w1", [7, 1, 20, 1], [7, 33, 50, 3000], 8, 2, 128, 16, window=1, seed=3)
    got = tu.run(case, num_splits=3)
    cu, kvl = case.cu_query_lens.tolist(), case.kv_lens.tolist()
    for s in range(case.num_seqs):
        ql = cu[s + 1] - cu[s]
        for i in range(ql):
            pos = kvl[s] - ql + i
            page = int(case.block_tables[s, pos // 16])
            for h in range(8):
                exp = case.v_cache[page, pos % 16, h // 4]
                assert torch.equal(got[cu[s] + i, h].view(torch.int16), exp.view(torch.int16))


def test_identical_keys_give_mean_of_values():
    case = W.make_case("same_k", [1, 4, 1], [300, 90, 2000], 8, 2, 128, 16, seed=7)
    case.k_cache[:] = case.k_cache[0, 0, 0]
    got = as_f64(tu.run(case))
    exp = oracle_full(case)
    assert_close(got, exp, W.BF16, "identical keys")


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
def test_gather_index_handling_is_bit_exact(dtype):
    case = W.random_small_case(70, kv_dtype=dtype, head_dim=128, num_q_heads=8, num_kv_heads=2,
                               max_kv=600)
    b = tu.to_device(case)
    with tu.make_plan(b, num_splits=3) as plan:
        _, _, dec, _ = ua.ua_schedule(b.cu_host, b.kv_host, 8, 2, 128, 16,
                                      int(b.block_tables.shape[1]), kv_dtype=b.kv_dtype,
                                      num_splits=3, num_sms=plan.info.num_sms)
        rows = sum(t["kv_hi"] - t["kv_lo"] for t in dec)
        elt = 1 if dtype == W.FP8 else 2
        ko = torch.zeros((rows, 128 * elt), dtype=torch.uint8, device="cuda")
        vo = torch.zeros_like(ko)
        ua.ua_gather_kv_debug(plan.handle, b.k_cache, b.v_cache, b.kv_lens, b.block_tables,
                              b.num_blocks, ko, vo, rows)
        torch.cuda.synchronize()
    kraw = case.k_cache.contiguous().view(torch.uint8).reshape(case.num_blocks, 16, 2, 128 * elt)
    vraw = case.v_cache.contiguous().view(torch.uint8).reshape(case.num_blocks, 16, 2, 128 * elt)
    off = 0
    ko, vo = ko.cpu(), vo.cpu()
    for t in dec:
        for key in range(t["kv_lo"], t["kv_hi"]):
            page = int(case.block_tables[t["seq"], key // 16])
            assert torch.equal(ko[off], kraw[page, key % 16, t["kv_head"]])
            assert torch.equal(vo[off], vraw[page, key % 16, t["kv_head"]])
            off += 1
    assert off == rows


def test_out_of_range_page_id_sets_error_word():
    case = W.make_case("bad_page", [1, 1], [100, 64], 8, 2, 128, 16, seed=8)
    b = tu.to_device(case)
    b.block_tables[0, 2] = case.num_blocks + 5   # never dereferenced, reported instead
    with tu.make_plan(b) as plan:
        tu.forward(plan, b)
        assert plan.last_device_error() == ua.UA_ERR_BOUNDS
        assert plan.last_device_error() == 0    # cleared by the read


def test_host_side_validation_launches_nothing():
    case = W.make_case("val", [1], [100], 8, 2, 128, 16, seed=9)
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        out = b.new_out()
        bad_q = b.q.view(-1)[1:]  # not 16-byte aligned
        with pytest.raises(ua.UAError) as e:
            ua.ua_forward(plan.handle, bad_q, b.k_cache, b.v_cache, out, b.cu_query_lens,
                          b.kv_lens, b.block_tables, b.num_blocks, 1, 100, b.scale)
        assert e.value.status == ua.UA_ERR_INVALID_ARG
        with pytest.raises(ua.UAError) as e:
            ua.ua_forward(plan.handle, b.q, b.k_cache, b.v_cache, out, b.cu_query_lens,
                          b.kv_lens, b.block_tables, b.num_blocks, 1, 99, b.scale)  # max_kv short
        assert e.value.status == ua.UA_ERR_INVALID_ARG


def test_oneshot_matches_plan_path():
    case = W.random_small_case(80, head_dim=128, num_q_heads=8, num_kv_heads=2, max_kv=600)
    b = tu.to_device(case)
    a = tu.run(case)
    out = b.new_out()
    ua.ua_forward_oneshot(b.q, b.k_cache, b.v_cache, out, b.cu_host, b.kv_host, b.cu_query_lens,
                          b.kv_lens, b.block_tables, 8, 2, 128, 16, int(b.block_tables.shape[1]),
                          b.num_blocks, b.kv_dtype, b.max_q, b.max_kv, b.scale)
    assert torch.equal(a.view(torch.int16), out.cpu().view(torch.int16))


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_entry_point_matches_plan_path(pinned):
    """ua_forward_host (q, output, lengths and page tables in host memory)
    gives the planned path's output bit for bit, on a mixed batch (both
    kernels) and on a decode batch, from pinned and from pageable memory."""
    for case in (W.make_case("host_mixed", [1, 300, 1, 40], [900, 700, 3000, 40], 16, 4, 128, 16,
                             seed=81),
                 W.random_small_case(82, kv_dtype=W.FP8, head_dim=64, num_q_heads=8,
                                     num_kv_heads=2, max_kv=700)):
        b = tu.to_device(case)
        ref = tu.run(case)
        q_h = case.q.contiguous()
        out_h = torch.empty_like(q_h)
        cu_h, kv_h = case.cu_query_lens.to(torch.int32), case.kv_lens.to(torch.int32)
        bt_h = case.block_tables.to(torch.int32).contiguous()
        if pinned:
            q_h, out_h, cu_h, kv_h, bt_h = (t.pin_memory() for t in (q_h, out_h, cu_h, kv_h, bt_h))
        err = ua.ua_forward_host(q_h, out_h, cu_h, kv_h, bt_h, b.k_cache, b.v_cache,
                                 b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                 b.num_blocks, b.kv_dtype, b.scale, causal=b.causal,
                                 window=b.window, k_scale=b.k_scale, v_scale=b.v_scale)
        assert err == 0
        assert torch.equal(out_h.view(torch.int16), ref.view(torch.int16)), case.name


@pytest.mark.parametrize("cfg", [2, 5, 7, 8])
def test_full_size_decode_configs_whole_output(cfg):
    """The full-size decode workloads in the benchmark's launch configuration
    (automatic splits): every element of the output against the fp64 oracle
    (computed on every host core), max-abs and mean-abs over the whole output."""
    case = W.CONFIGS[cfg]()
    got = as_f64(tu.run(case))
    torch.cuda.empty_cache()
    exp = oracle_full_parallel(case)
    assert_close(got, exp, case.kv_dtype, f"workload {cfg} ({case.name})", report=True)


def test_full_size_window_decode_whole_output():
    """The pure-decode workload with a 1024-key window (the benchmark's
    `--window 1024` case: its 56 last tiles are cut into tail pieces): every
    element against the fp64 oracle."""
    import dataclasses
    case = dataclasses.replace(W.CONFIGS[2](), window=1024)
    got = as_f64(tu.run(case))
    torch.cuda.empty_cache()
    exp = oracle_full_parallel(case)
    assert_close(got, exp, case.kv_dtype, f"workload 2, window 1024 ({case.name})", report=True)


# ---- head_dim 256 (decode kernel only: V fragments read after the softmax)

@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
def test_head_dim_256_random(dtype):
    for seed in (600, 601):
        _check(W.random_small_case(seed, kv_dtype=dtype, head_dim=256, num_q_heads=8,
                                   num_kv_heads=2, max_kv=900))


def test_head_dim_256_splits_window_and_long_prefill():
    case = W.make_case("d256_mix", [1, 1, 130], [3000, 70, 400], 16, 4, 256, 16, seed=610)
    _check(case, num_splits=7)
    _check(W.make_case("d256_win", [1, 50], [2000, 600], 8, 2, 256, 32, window=300, seed=611))
    _check(W.make_case("d256_fp8", [1, 3], [5000, 900], 16, 2, 256, 16, kv_dtype=W.FP8,
                       seed=612), num_splits=16)


def test_head_dim_256_allocation_free_entry_point_matches_oracle():
    # a decode batch: the entry point's fixed scratch sizes split pieces for
    # every row tile of the longest query
    case = W.make_case("d256_static", [1, 1, 1, 1], [3000, 70, 1200, 16], 8, 2, 256, 16, seed=620)
    b = tu.to_device(case)
    out = b.new_out()
    err = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    ua.ua_forward_static_scratch(
        b.q, b.k_cache, b.v_cache, out, b.cu_query_lens, b.kv_lens, b.block_tables,
        b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size, int(b.block_tables.shape[1]),
        b.num_blocks, b.kv_dtype, b.max_q, b.max_kv, b.scale, causal=b.causal, window=b.window,
        k_scale=b.k_scale, v_scale=b.v_scale, num_splits=4, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)


# ---- every other head_dim that is a multiple of 32 up to 256: the decode
# kernel (and at 192 the wide prefill kernel for long prefills)

NEW_DIMS = [32, 96, 160, 192, 224]


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
@pytest.mark.parametrize("d", NEW_DIMS)
def test_other_head_dims_random(d, dtype):
    for seed in (800, 801):
        _check(W.random_small_case(seed + d, kv_dtype=dtype, head_dim=d, num_q_heads=8,
                                   num_kv_heads=2, max_kv=700))


@pytest.mark.parametrize("d", NEW_DIMS)
def test_other_head_dims_splits_window_noncausal_and_poison(d):
    _check(W.make_case(f"d{d}_split", [1, 1, 3, 1], [3000, 70, 1300, 16], 16, 4, d, 16,
                       seed=810 + d), num_splits=7)
    _check(W.make_case(f"d{d}_win", [1, 40], [2000, 600], 8, 2, d, 32, window=300,
                       seed=811 + d))
    _check(W.make_case(f"d{d}_nc", [1, 30], [900, 300], 4, 4, d, 16, causal=False,
                       seed=812 + d))
    _check(W.make_case(f"d{d}_fp8", [1, 3], [4000, 900], 16, 2, d, 16, kv_dtype=W.FP8,
                       poison=True, seed=813 + d), num_splits=16)


@pytest.mark.parametrize("d", [96, 160])
def test_other_head_dims_allocation_free_entry_point(d):
    case = W.make_case(f"d{d}_static", [1, 1, 1, 1], [3000, 70, 1200, 16], 8, 2, d, 16,
                       seed=830 + d)
    b = tu.to_device(case)
    out = b.new_out()
    err = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    ua.ua_forward_static_scratch(
        b.q, b.k_cache, b.v_cache, out, b.cu_query_lens, b.kv_lens, b.block_tables,
        b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size, int(b.block_tables.shape[1]),
        b.num_blocks, b.kv_dtype, b.max_q, b.max_kv, b.scale, causal=b.causal, window=b.window,
        k_scale=b.k_scale, v_scale=b.v_scale, num_splits=4, device_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)


def test_plan_churn_reuses_pooled_memory():
    """A serving loop builds and drops a plan every step: plan memory comes
    from the library's stream-ordered pool and pinned upload blocks, so 200
    more steps leave device memory use where it was, and the results stay
    right."""
    case = W.config1_tiny_mixed()
    b = tu.to_device(case)
    exp = oracle_full(case)

    def step():
        with tu.make_plan(b, num_splits=3) as plan:
            return tu.forward(plan, b)

    for _ in range(20):
        step()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(200):
        out = step()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert abs(free1 - free0) < 64 * 2 ** 20, (free0, free1)
    assert_close(as_f64(out), exp, case.kv_dtype, case.name)
