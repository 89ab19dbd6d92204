"""GPU parity of the fp8-products prefill (e4m3 Q.K^T and e4m3 P.V on the
tensor cores, reading the e4m3 cache directly) against its fp64 oracle, and
its distance from the exact (dequantised) oracle."""
import numpy as np
import pytest
import torch

import paged_kv_attention_unified_gb300 as ua
from paged_kv_attention_unified_gb300 import torch_utils as tu
import workloads as W

from _helpers import as_f64, assert_close, oracle_full, oracle_fp8_products

pytestmark = pytest.mark.gpu

# Against its own oracle the kernel differs only by binary32 exponentials and
# accumulation order, which move a few e4m3 roundings of P by one step.
F8P_MAX_ABS = 2e-2
F8P_MEAN_ABS = 1e-3
# Against the exact attention over the dequantised cache the e4m3 rounding of
# Q and P shows: each carries up to 2^-4 relative error per element, so an
# output of size ~2 may move by ~0.1 where they add up (bound with room).
EXACT_MAX_ABS = 0.15
EXACT_MEAN_ABS = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_unified_gb300 import build
    build.build()


def _run_f8p(case, decode_rows_max=0):
    b = tu.to_device(case)
    with tu.make_plan(b, decode_rows_max=decode_rows_max) as plan:
        ua.ua_plan_set_fp8_products(plan.handle, True)
        assert plan.info.num_prefill_tiles > 0
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    return as_f64(out)


def _check(case, report=False):
    got = _run_f8p(case)
    exp = oracle_fp8_products(case)
    err = np.abs(got - exp)
    assert np.all(np.isfinite(got))
    assert err.max() <= F8P_MAX_ABS, f"{case.name}: max-abs {err.max():.3e}"
    assert err.mean() <= F8P_MEAN_ABS, f"{case.name}: mean-abs {err.mean():.3e}"
    # and within the e4m3-operand bound of the exact attention
    ex = np.abs(got - oracle_full(case))
    assert ex.max() <= EXACT_MAX_ABS, f"{case.name} vs exact: max-abs {ex.max():.3e}"
    assert ex.mean() <= EXACT_MEAN_ABS, f"{case.name} vs exact: mean-abs {ex.mean():.3e}"
    if report:
        from _helpers import PARITY_REPORT
        PARITY_REPORT.append((case.name + " (fp8 products, own oracle)", int(err.size),
                              float(err.max()), float(err.mean())))
        PARITY_REPORT.append((case.name + " (fp8 products, exact oracle)", int(ex.size),
                              float(ex.max()), float(ex.mean())))
    return got


@pytest.mark.parametrize("qpk,hkv,bs", [(1, 2, 16), (4, 2, 32), (8, 1, 128), (2, 4, 64),
                                        (16, 1, 256)])
def test_fp8_products_prefill_matches_its_oracle(qpk, hkv, bs):
    _check(W.make_case(f"f8p_{qpk}_{bs}", [300, 77, 129, 1], [300, 533, 200, 90], qpk * hkv,
                       hkv, 128, bs, kv_dtype=W.FP8, seed=1000 + qpk + bs))


def test_fp8_products_window_noncausal_and_poison():
    _check(W.make_case("f8p_win", [400, 260], [900, 260], 8, 2, 128, 16, kv_dtype=W.FP8,
                       window=150, seed=1010))
    _check(W.make_case("f8p_nc", [200, 90], [600, 90], 8, 2, 128, 32, kv_dtype=W.FP8,
                       causal=False, seed=1011))
    _check(W.make_case("f8p_poison", [333, 150], [700, 181], 8, 2, 128, 16, kv_dtype=W.FP8,
                       poison=True, seed=1012))


def test_fp8_products_one_cta_and_repeated_forwards():
    """One persistent CTA takes every work tile in turn (ring and barrier
    phases, and the Q tiles the softmax warps rewrite, run on across work
    tiles); a second forward gives the same bits."""
    case = W.make_case("f8p_one_cta", [1024] * 3, [1024] * 3, 8, 8, 128, 128, kv_dtype=W.FP8,
                       table="identity", seed=1020)
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        ua.ua_plan_set_fp8_products(plan.handle, True)
        ua.ua_plan_set_prefill_ctas(plan.handle, 1)
        out = tu.forward(plan, b)
        out2 = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    exp = oracle_fp8_products(case)
    assert np.abs(as_f64(out) - exp).max() <= F8P_MAX_ABS


def test_fp8_products_mixed_batch_keeps_decode_exact():
    """Prefill tiles take the fp8 products, decode tiles keep their f16
    products: each part against its own oracle."""
    case = W.make_case("f8p_mixed", [1, 600, 1, 37], [3000, 1400, 70, 900], 16, 4, 128, 16,
                       kv_dtype=W.FP8, seed=1030)
    got = _run_f8p(case, decode_rows_max=-1)
    exact = oracle_full(case)
    f8p = oracle_fp8_products(case)
    cu = case.cu_query_lens.tolist()
    dec_rows = np.r_[cu[0]:cu[1], cu[2]:cu[3]]
    pre_rows = np.r_[cu[1]:cu[2], cu[3]:cu[4]]
    assert_close(got[dec_rows], exact[dec_rows], W.FP8, "decode rows")
    assert np.abs(got[pre_rows] - f8p[pre_rows]).max() <= F8P_MAX_ABS


def test_fp8_products_is_refused_where_it_does_not_apply():
    bf = W.make_case("bf16", [64], [64], 4, 4, 128, 16, seed=1040)
    b = tu.to_device(bf)
    with tu.make_plan(b) as plan:
        with pytest.raises(ua.UAError) as e:
            ua.ua_plan_set_fp8_products(plan.handle, True)
        assert e.value.status == ua.UA_ERR_UNSUPPORTED
    f64 = W.make_case("d64", [64], [64], 4, 4, 64, 16, kv_dtype=W.FP8, seed=1041)
    b = tu.to_device(f64)
    with tu.make_plan(b) as plan:
        with pytest.raises(ua.UAError) as e:
            ua.ua_plan_set_fp8_products(plan.handle, True)
        assert e.value.status == ua.UA_ERR_UNSUPPORTED


def test_fp8_products_dense_prefill_2x2048():
    """A dense causal prefill of two 2048-token sequences (32 query heads over
    8 KV heads, identity page table): the whole output."""
    case = W.make_case("f8p_dense_2x2048", [2048] * 2, [2048] * 2, 32, 8, 128, 128,
                       kv_dtype=W.FP8, table="identity", seed=1050)
    _check(case, report=True)
