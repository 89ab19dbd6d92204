"""GPU parity of the unified-max decode option (FlashDecoding++, "Fused
Attention" notes: a preset value replaces each row's maximum, with a fallback
when the scores leave its range) against the fp64 oracle, through the C ABI.

The option changes only the value subtracted before exponentiation, so the
oracle is the plain softmax attention; a value outside every row's range
must reproduce the default path bit for bit (every row falls back)."""
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


def _run(b, phi, num_splits=0):
    with tu.make_plan(b, num_splits=num_splits) as plan:
        plan.set_unified_max(phi)
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    return out


def _decode_case(dtype, seed, scale=None):
    return W.make_case(f"umax_{dtype}_{seed}", [1, 1, 2, 1, 3, 1], [3000, 17, 900, 1, 2500, 64],
                       32, 8, 128, 16, kv_dtype=dtype, seed=seed, scale=scale)


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
@pytest.mark.parametrize("phi", [1000.0, -1000.0])
def test_out_of_range_phi_falls_back_bit_for_bit(dtype, phi):
    case = _decode_case(dtype, 400)
    b = tu.to_device(case)
    for ns in (0, 3):
        ref = _run(b, None, ns)
        got = _run(b, phi, ns)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
def test_in_range_phi_matches_the_oracle(dtype):
    case = _decode_case(dtype, 401)
    b = tu.to_device(case)
    exp = oracle_full(case)
    ref = _run(b, None)
    differs = False
    # scores are about N(0, 1): row maxima of the first 16 keys lie near 1.7,
    # so these values sit inside the range for most rows (bf16: up to 44
    # above the maximum; e4m3: at most 5.5 below it)
    phis = [0.0, 1.0, 2.0, 10.0, 40.0] if dtype == W.BF16 else [-2.0, 0.0, 1.0]
    for phi in phis:
        for ns in (0, 2, 16):
            got = _run(b, phi, ns)
            assert_close(as_f64(got), exp, dtype, f"{case.name} phi={phi} splits={ns}")
            differs |= not torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert differs, "the unified max never changed a rounding: is it reaching the kernel?"


@pytest.mark.parametrize("dtype", [W.BF16, W.FP8])
def test_wide_scores_take_the_fallbacks(dtype):
    """Scaled scores with a spread of about 20 (maxima near 60): a preset
    value below the later keys' maxima triggers the upward rescale, one far
    above the first maxima the fallback to the row's own maximum."""
    case = _decode_case(dtype, 402, scale=20.0 / np.sqrt(128))
    b = tu.to_device(case)
    exp = oracle_full(case)
    for phi in (-30.0, 0.0, 30.0, 50.0, 70.0, 200.0):
        for ns in (0, 4):
            assert_close(as_f64(_run(b, phi, ns)), exp, dtype, f"{case.name} phi={phi}")


def test_mixed_batch_prefill_tiles_unaffected():
    """Prefill tiles keep the running maximum: a mixed batch with the option on
    matches the oracle, and its prefill rows are bit-identical to the default."""
    case = W.make_case("umax_mixed", [1, 200, 1, 70], [900, 600, 3000, 70], 16, 4, 128, 16,
                       seed=403)
    b = tu.to_device(case)
    ref = _run(b, None)
    got = _run(b, 1.5)
    assert_close(as_f64(got), oracle_full(case), case.kv_dtype, case.name)
    cu = case.cu_query_lens.tolist()
    for s in (1, 3):                       # the prefill sequences (q_len * qpk > 32)
        assert torch.equal(got[cu[s]:cu[s + 1]].view(torch.int16),
                           ref[cu[s]:cu[s + 1]].view(torch.int16))


def test_invalid_values_are_rejected():
    case = _decode_case(W.BF16, 404)
    b = tu.to_device(case)
    with tu.make_plan(b) as plan:
        for bad in (float("nan"), float("inf"), -float("inf"), 1e31):
            with pytest.raises(ua.UAError):
                plan.set_unified_max(bad)
        plan.set_unified_max(3.0)
        plan.set_unified_max(None)
