"""Pins of the append oracle (oracle/append.py) to things other than itself:
the e4m3 format's own code table, torch's e4m3 cast where the two readings
coincide, the nearest-value property, and caches built directly by the input
generator (which writes every token's K/V at its page slot)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from oracle import append as A


def _finite_codes():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_e4m3(codes)
    keep = ~np.isnan(vals)
    return codes[keep], vals[keep]


def test_encode_inverts_decode_on_every_finite_code():
    codes, vals = _finite_codes()
    assert len(codes) == 254
    assert np.array_equal(oracle.encode_e4m3(vals), codes)


def test_encode_matches_torch_cast_below_overflow():
    """torch rounds to nearest even and overflows to NaN; below the overflow
    threshold (464 = midway between 448 and the next step) the two agree."""
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(4000) * 50.0,
        rng.standard_normal(2000) * 2.0 ** -7,          # subnormal range
        rng.uniform(-463.9, 463.9, 2000),
    ]).astype(np.float32)
    # exact midpoints between consecutive finite codes (ties)
    _, vals = _finite_codes()
    pos = np.unique(vals[vals >= 0])
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids, pos.astype(np.float32)])
    ours = oracle.encode_e4m3(x)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, theirs)


def test_saturation_and_nan():
    x = np.array([464.0, 465.0, 500.0, 1e30, np.inf, -464.0, -1e30, -np.inf, np.nan])
    assert oracle.encode_e4m3(x).tolist() == [0x7E] * 5 + [0xFE] * 3 + [0x7F]


def test_nearest_and_monotone():
    _, vals = _finite_codes()
    grid = np.unique(vals)
    rng = np.random.default_rng(6)
    x = np.sort(rng.uniform(-448.0, 448.0, 5000))
    dec = oracle.decode_e4m3(oracle.encode_e4m3(x))
    # no grid value is strictly closer than the chosen one
    best = np.min(np.abs(grid[None, :] - x[:, None]), axis=1)
    assert np.all(np.abs(dec - x) <= best + 0.0)
    assert np.all(np.diff(dec) >= 0)


def test_quantize_divides_in_binary32():
    rng = np.random.default_rng(7)
    f = rng.standard_normal(3000).astype(np.float32)
    bits = (torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    scale = np.float32(3.0 / 448.0)
    codes = oracle.quantize_e4m3(bits, float(scale))
    x = oracle.decode_bf16(bits).astype(np.float32) / scale      # binary32 quotient
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inrange = np.abs(x) < 464
    assert np.array_equal(codes[inrange], ref[inrange])
    assert np.all(codes[~inrange] & 0x7F == 0x7E)


def _split_new_tokens(case):
    """The generator's cache holds every token; take the new tokens' rows out of
    it (by the page table) and blank their slots, giving (k_new, v_new, cache
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
            k_new[cu[s] + i] = kc[blk, slot]
            v_new[cu[s] + i] = vc[blk, slot]
            kc[blk, slot] = blank
            vc[blk, slot] = blank
    return r, k_new, v_new, kc, vc


@pytest.mark.parametrize("bs", [16, 32])
def test_append_rebuilds_the_generator_cache(bs):
    case = W.make_case("app", [1, 7, 40, 1], [33, 70, 40, 200], 8, 2, 64, bs, seed=11)
    r, k_new, v_new, kc, vc = _split_new_tokens(case)
    k2, v2 = oracle.append_kv(k_new, v_new, kc, vc, r["cu_query_lens"], r["kv_lens"],
                              r["block_tables"], bs)
    assert np.array_equal(k2, r["k_cache"]) and np.array_equal(v2, r["v_cache"])


def test_append_fp8_writes_quantized_rows_and_nothing_else():
    case = W.make_case("app8", [3, 1, 17], [50, 9, 17], 4, 4, 64, 16, seed=12)
    r = case.raw()
    rng = np.random.default_rng(13)
    T = int(r["cu_query_lens"][-1])
    f = (rng.standard_normal((T, 4, 64)) * 2.0).astype(np.float32)
    bits = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    kc = np.full((64, 16, 4, 64), 0x7F, dtype=np.uint8)
    vc = kc.copy()
    bt = r["block_tables"]
    k2, v2 = oracle.append_kv(bits, bits, kc, vc, r["cu_query_lens"], r["kv_lens"], bt, 16,
                              kv_dtype="fp8_e4m3", k_scale=0.01, v_scale=0.02)
    written = np.zeros(kc.shape[:2], dtype=bool)
    cu, kvl = r["cu_query_lens"], r["kv_lens"]
    for s in range(3):
        ql = int(cu[s + 1] - cu[s])
        t = np.arange(int(kvl[s]) - ql, int(kvl[s]))
        # read back through the attention oracle's own page addressing
        blk, slot = oracle.attention.page_address(bt, s, t, 16)
        assert np.array_equal(k2[blk, slot], oracle.quantize_e4m3(bits[cu[s]:cu[s + 1]], 0.01))
        assert np.array_equal(v2[blk, slot], oracle.quantize_e4m3(bits[cu[s]:cu[s + 1]], 0.02))
        for p in t:
            written[bt[s, p // 16], p % 16] = True
    assert np.all(k2[~written] == 0x7F) and np.all(v2[~written] == 0x7F)


def test_mutations_are_caught(monkeypatch):
    """A planted mistake in the oracle must fail a pin."""
    codes, vals = _finite_codes()
    # 1. truncation instead of round-to-nearest-even
    real = A._encode_one

    def trunc(x):
        if np.isnan(x) or np.isinf(x) or abs(x) < 2.0 ** -6:
            return real(x)
        sign = 0x80 if np.signbit(x) else 0
        _, e2 = np.frexp(abs(x))
        e = int(e2) - 1
        q = np.floor(abs(x) / 2.0 ** (e - 3))
        return sign | ((e + 7) << 3) | int(q - 8) if e + 7 <= 15 else sign | 0x7E

    monkeypatch.setattr(A, "_encode_one", trunc)
    mids = np.array([1.0625, 3.3, 100.0 + 1.0], dtype=np.float32)
    theirs = torch.from_numpy(mids).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert not np.array_equal(oracle.encode_e4m3(mids), theirs)
    monkeypatch.setattr(A, "_encode_one", real)
    # 2. multiplying by the scale instead of dividing
    real_q = A.quantize_e4m3

    def times(bits, scale):
        x = oracle.decode_bf16(bits).astype(np.float32)
        return A.encode_e4m3((x * np.float32(scale)).astype(np.float32))

    monkeypatch.setattr(A, "quantize_e4m3", times)
    bits = np.array([0x3F80, 0x4000, 0xC040], dtype=np.uint16)    # 1, 2, -3
    x = oracle.decode_bf16(bits).astype(np.float32) / np.float32(0.25)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert not np.array_equal(A.quantize_e4m3(bits, 0.25), ref)
    monkeypatch.setattr(A, "quantize_e4m3", real_q)
    assert np.array_equal(A.quantize_e4m3(bits, 0.25), ref)
    # 3. rows placed one token off: the rebuilt cache differs from the generator's
    case = W.make_case("app_mut", [5], [21], 2, 2, 64, 16, seed=14)
    r, k_new, v_new, kc, vc = _split_new_tokens(case)
    shifted = np.concatenate([k_new[1:], k_new[:1]])
    k2, _ = oracle.append_kv(shifted, v_new, kc, vc, r["cu_query_lens"], r["kv_lens"],
                             r["block_tables"], 16)
    assert not np.array_equal(k2, r["k_cache"])
