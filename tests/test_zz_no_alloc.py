"""The allocation-free entry point against the fp64 oracle and the planned path.

ua_forward_static_scratch is for callers that may not allocate device memory
themselves -- code running inside a runtime that owns every device allocation
through its own pool, plugins hosted by such a runtime, or loops where the
device-wide synchronisation cudaMalloc can cause is not acceptable. Its tile
list, split partials and error word live in a static device array inside
libua.so. This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_unified_gb300 as ua
from paged_kv_attention_unified_gb300 import torch_utils as tu
import workloads as W

from _helpers import as_f64, assert_close, oracle_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_unified_gb300 import build
    build.build()


def _static(b, num_splits=0):
    out = b.new_out()
    err = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    ua.ua_forward_static_scratch(
        b.q, b.k_cache, b.v_cache, out, b.cu_query_lens, b.kv_lens, b.block_tables,
        b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size, int(b.block_tables.shape[1]),
        b.num_blocks, b.kv_dtype, b.max_q, b.max_kv, b.scale, causal=b.causal, window=b.window,
        k_scale=b.k_scale, v_scale=b.v_scale, num_splits=num_splits, device_error=err)
    torch.cuda.synchronize()
    return out.cpu(), int(err.item())


def _planned(b, num_splits=0):
    with tu.make_plan(b, num_splits=num_splits) as plan:
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
    return out.cpu()


def test_two_calls_in_a_row_match_the_oracle_and_the_planned_path():
    cases = [
        W.random_small_case(300, head_dim=128, num_q_heads=8, num_kv_heads=2, max_kv=1500),
        W.random_small_case(301, kv_dtype=W.FP8, head_dim=64, num_q_heads=16, num_kv_heads=4,
                            max_kv=900, window=200),
    ]
    for case in cases:                       # two calls in a row, different shapes
        b = tu.to_device(case)
        got, err = _static(b)
        assert err == 0
        assert_close(as_f64(got), oracle_full(case), case.kv_dtype, case.name)
        assert_close(as_f64(got), as_f64(_planned(b)), case.kv_dtype, case.name + " vs plan")


def test_repeated_call_on_the_same_batch_allocates_nothing():
    case = W.make_case("repeat", [1] * 12 + [3], [4000, 17, 900, 2500] * 3 + [64], 32, 8, 128, 16,
                       seed=302)
    b = tu.to_device(case)
    exp = oracle_full(case)
    first, e1 = _static(b, num_splits=16)    # the first call on a device sets itself up
    out = b.new_out()
    err = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(50):
        ua.ua_forward_static_scratch(
            b.q, b.k_cache, b.v_cache, out, b.cu_query_lens, b.kv_lens, b.block_tables,
            b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size,
            int(b.block_tables.shape[1]), b.num_blocks, b.kv_dtype, b.max_q, b.max_kv, b.scale,
            num_splits=16, device_error=err)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0   # no device allocation by the calls
    second = out.cpu()
    assert e1 == 0 and int(err.item()) == 0
    assert_close(as_f64(first), exp, W.BF16, "first call")
    assert_close(as_f64(second), exp, W.BF16, "later call")
    assert torch.equal(first.view(torch.int16), second.view(torch.int16))


def test_lengths_beyond_the_declared_bounds_are_reported():
    """max_q below a sequence's q_len leaves rows outside the tile grid: the
    device records UA_ERR_INVALID_ARG instead of returning them unwritten."""
    case = W.make_case("short_max_q", [1, 3, 2], [500, 300, 40], 8, 2, 128, 16, seed=304)
    b = tu.to_device(case)
    out = b.new_out()
    err = torch.full((1,), -99, dtype=torch.int32, device="cuda")
    ua.ua_forward_static_scratch(
        b.q, b.k_cache, b.v_cache, out, b.cu_query_lens, b.kv_lens, b.block_tables,
        b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size, int(b.block_tables.shape[1]),
        b.num_blocks, b.kv_dtype, 2, b.max_kv, b.scale, device_error=err)   # q_len 3 > 2
    torch.cuda.synchronize()
    assert int(err.item()) == ua.UA_ERR_INVALID_ARG
    got, e = _static(b)                          # the right bound: clean again
    assert e == 0
    assert_close(as_f64(got), oracle_full(case), W.BF16, case.name)


def test_bad_fp8_scale_is_rejected_without_launch():
    case = W.make_case("fp8_scale", [1], [100], 8, 2, 128, 16, kv_dtype=W.FP8, seed=305)
    b = tu.to_device(case)
    for ks in (0.0, float("nan"), float("inf")):
        with pytest.raises(ua.UAError) as e:
            ua.ua_forward_static_scratch(
                b.q, b.k_cache, b.v_cache, b.new_out(), b.cu_query_lens, b.kv_lens,
                b.block_tables, b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size,
                int(b.block_tables.shape[1]), b.num_blocks, b.kv_dtype, b.max_q, b.max_kv,
                b.scale, k_scale=ks, v_scale=b.v_scale)
        assert e.value.status == ua.UA_ERR_INVALID_ARG


def test_oversized_call_is_rejected_without_launch():
    case = W.make_case("big", [1] * 8, [20000] * 8, 64, 8, 128, 16, seed=303)
    b = tu.to_device(case)
    with pytest.raises(ua.UAError) as e:
        _static(b, num_splits=128)   # 8 * 8 * 128 split tiles need more than 16 MiB
    assert e.value.status == ua.UA_ERR_WORKSPACE
