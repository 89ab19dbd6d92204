"""The allocation-free entry point agrees with the planned entry point.

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

from _helpers import as_f64, assert_close

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


def test_two_calls_in_a_row_match_the_planned_path():
    cases = [
        W.random_small_case(300, head_dim=128, num_q_heads=8, num_kv_heads=2, max_kv=1500),
        W.random_small_case(301, kv_dtype=W.FP8, head_dim=64, num_q_heads=16, num_kv_heads=4,
                            max_kv=900, window=200),
    ]
    for case in cases:                       # two calls in a row, different shapes
        b = tu.to_device(case)
        got, err = _static(b)
        ref = _planned(b)
        assert err == 0
        assert_close(as_f64(got), as_f64(ref), case.kv_dtype, case.name)


def test_repeated_call_on_the_same_batch():
    case = W.make_case("repeat", [1] * 12 + [3], [4000, 17, 900, 2500] * 3 + [64], 32, 8, 128, 16,
                       seed=302)
    b = tu.to_device(case)
    ref = _planned(b, num_splits=16)
    first, e1 = _static(b, num_splits=16)
    second, e2 = _static(b, num_splits=16)
    assert e1 == 0 and e2 == 0
    assert_close(as_f64(first), as_f64(ref), W.BF16, "first call")
    assert_close(as_f64(second), as_f64(ref), W.BF16, "second call")
    assert torch.equal(first.view(torch.int16), second.view(torch.int16))


def test_oversized_call_is_rejected_without_launch():
    case = W.make_case("big", [1] * 8, [20000] * 8, 64, 8, 128, 16, seed=303)
    b = tu.to_device(case)
    with pytest.raises(ua.UAError) as e:
        _static(b, num_splits=128)   # 8 * 8 * 128 split tiles need more than 16 MiB
    assert e.value.status == ua.UA_ERR_WORKSPACE
