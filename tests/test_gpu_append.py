"""GPU parity of ua_append_kv (through the C ABI) against the oracle: cache
bytes bit for bit (bf16 words, e4m3 codes), then attention over the result."""
import numpy as np
import pytest
import torch

import oracle
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


def _raw_to_device(a):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    elif a.dtype == np.uint8:
        t = t.view(torch.float8_e4m3fn)
    return t.cuda()


def _to_raw(t):
    t = t.cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def _split_new_tokens(case):
    """Take the new tokens' rows out of the generator's cache (by the page
    table) and blank their slots with NaN: returns (raw, k_new, v_new, caches
    without them)."""
    r = case.raw()
    cu, kvl, bt, bs = r["cu_query_lens"], r["kv_lens"], r["block_tables"], case.block_size
    kc, vc = r["k_cache"].copy(), r["v_cache"].copy()
    T = int(cu[-1])
    k_new = np.zeros((T,) + kc.shape[2:], dtype=kc.dtype)
    v_new = np.zeros_like(k_new)
    blank = np.uint16(0x7FC0) if kc.dtype == np.uint16 else np.uint8(0x7F)
    for s in range(len(kvl)):
        ql = int(cu[s + 1] - cu[s])
        for i in range(ql):
            pos = int(kvl[s]) - ql + i
            blk, slot = int(bt[s, pos // bs]), pos % bs
            k_new[cu[s] + i], v_new[cu[s] + i] = kc[blk, slot], vc[blk, slot]
            kc[blk, slot] = blank
            vc[blk, slot] = blank
    return r, k_new, v_new, kc, vc


@pytest.mark.parametrize("bs,d,hkv", [(16, 128, 8), (32, 64, 2), (128, 128, 4)])
def test_bf16_append_rebuilds_the_cache_bit_exact(bs, d, hkv):
    case = W.make_case(f"app_bf16_{bs}", [1, 9, 130, 1, 33], [40, 90, 130, 700, 200], hkv * 4,
                       hkv, d, bs, seed=300 + bs)
    r, k_new, v_new, kc, vc = _split_new_tokens(case)
    b = tu.to_device(case)
    b.k_cache.copy_(_raw_to_device(kc))
    b.v_cache.copy_(_raw_to_device(vc))
    with tu.make_plan(b) as plan:
        tu.append_kv(plan, b, _raw_to_device(k_new), _raw_to_device(v_new))
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert np.array_equal(_to_raw(b.k_cache), r["k_cache"])
    assert np.array_equal(_to_raw(b.v_cache), r["v_cache"])


def test_fp8_append_codes_bit_exact_including_saturation_and_nan():
    case = W.make_case("app_fp8", [3, 1, 40, 17], [50, 9, 40, 300], 16, 2, 128, 16,
                       kv_dtype=W.FP8, seed=310)
    r = case.raw()
    T = int(r["cu_query_lens"][-1])
    rng = np.random.default_rng(311)
    f = (rng.standard_normal((2, T, 2, 128)) * 3.0).astype(np.float32)
    ks, vs = 0.01, 0.003
    # values at and beyond the saturation point, ties, subnormals, signed zero, NaN
    special = np.array([448 * ks, 464 * ks, 1e4, -1e4, -0.0, 0.0, 2.0 ** -10 * ks,
                        3 * 2.0 ** -10 * ks, np.nan, -np.nan], dtype=np.float32)
    f[0, 0, 0, :special.size] = special
    f[1, 1, 1, :special.size] = special * (vs / ks)
    bits = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    b = tu.to_device(case)
    b.k_scale, b.v_scale = ks, vs
    with tu.make_plan(b) as plan:
        tu.append_kv(plan, b, _raw_to_device(bits[0]), _raw_to_device(bits[1]))
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    k_ref, v_ref = oracle.append_kv(bits[0], bits[1], r["k_cache"], r["v_cache"],
                                    r["cu_query_lens"], r["kv_lens"], r["block_tables"], 16,
                                    kv_dtype="fp8_e4m3", k_scale=ks, v_scale=vs)
    got_k, got_v = _to_raw(b.k_cache), _to_raw(b.v_cache)
    for got, ref in ((got_k, k_ref), (got_v, v_ref)):
        nan = (ref & 0x7F) == 0x7F
        assert np.array_equal(got[~nan], ref[~nan])       # every finite code bit for bit
        assert np.all((got[nan] & 0x7F) == 0x7F)           # NaN stays NaN (either sign)
    assert np.any((k_ref & 0x7F) == 0x7E)                  # saturation was exercised


def test_bad_page_id_is_reported_and_not_written():
    case = W.make_case("app_bad", [4, 4], [20, 36], 4, 4, 64, 16, seed=320)
    r, k_new, v_new, kc, vc = _split_new_tokens(case)
    b = tu.to_device(case)
    b.k_cache.copy_(_raw_to_device(kc))
    b.v_cache.copy_(_raw_to_device(vc))
    bt = r["block_tables"].copy()
    bt[1, 35 // 16] = 10 ** 6                               # the page of seq 1's new tokens
    b.block_tables.copy_(torch.from_numpy(bt.astype(np.int32)))
    with tu.make_plan(b) as plan:
        tu.append_kv(plan, b, _raw_to_device(k_new), _raw_to_device(v_new))
        torch.cuda.synchronize()
        assert plan.last_device_error() == ua.UA_ERR_BOUNDS
    # sequence 0 was written exactly; nothing of sequence 1 landed anywhere
    k_ref, _ = oracle.append_kv(k_new[:4], v_new[:4], kc, vc, [0, 4], r["kv_lens"][:1],
                                r["block_tables"][:1], 16)
    assert np.array_equal(_to_raw(b.k_cache), k_ref)


def test_append_then_attention_matches_the_oracle():
    case = W.make_case("app_attn", [1, 60, 1, 300], [500, 260, 2000, 300], 32, 8, 128, 16,
                       seed=330)
    r, k_new, v_new, kc, vc = _split_new_tokens(case)
    b = tu.to_device(case)
    b.k_cache.copy_(_raw_to_device(kc))
    b.v_cache.copy_(_raw_to_device(vc))
    with tu.make_plan(b) as plan:
        tu.append_kv(plan, b, _raw_to_device(k_new), _raw_to_device(v_new))
        out = tu.forward(plan, b)
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert_close(as_f64(out), oracle_full(case), case.kv_dtype, case.name)


def test_full_size_mixed_append_bit_exact():
    """The mixed serving step (8 prefill + 120 decode sequences): every new
    token of the step appended, the whole cache compared."""
    case = W.config3_mixed()
    r, k_new, v_new, kc, vc = _split_new_tokens(case)
    b = tu.to_device(case)
    b.k_cache.copy_(_raw_to_device(kc))
    b.v_cache.copy_(_raw_to_device(vc))
    with tu.make_plan(b) as plan:
        tu.append_kv(plan, b, _raw_to_device(k_new), _raw_to_device(v_new))
        torch.cuda.synchronize()
        assert plan.last_device_error() == 0
    assert np.array_equal(_to_raw(b.k_cache), r["k_cache"])
    assert np.array_equal(_to_raw(b.v_cache), r["v_cache"])
