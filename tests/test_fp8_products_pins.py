"""Pins of the fp8-products oracle (oracle/fp8_products.py) to things other
than itself: the e4m3 codec and torch's e4m3 cast, closed forms for one key,
two keys and identical keys, and the exact (unquantised) oracle on inputs
whose every quantisation step is exact."""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8_products as F


def _bf16_bits(x):
    """float values that bf16 holds exactly -> bf16 words."""
    v = np.asarray(x, dtype=np.float32)
    bits = v.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "not bf16-exact"
    return (bits >> 16).astype(np.uint16)


def _problem(q_rows, k_vals, v_vals, cu, kv, hq, hkv, bs=16):
    """Raw arrays of one batch: q_rows [Tq, hq, d] floats (bf16-exact), k_vals /
    v_vals [B][kv_s, hkv, d] e4m3-exact values, an identity block table."""
    d = q_rows.shape[2]
    pages = [(-(-n // bs)) for n in kv]
    nblk = sum(pages)
    kc = np.zeros((nblk, bs, hkv, d), dtype=np.uint8)
    vc = np.zeros((nblk, bs, hkv, d), dtype=np.uint8)
    bt = np.zeros((len(kv), max(pages)), dtype=np.int32)
    nxt = 0
    for s, n in enumerate(kv):
        for i in range(pages[s]):
            bt[s, i] = nxt + i
        for t in range(n):
            kc[nxt + t // bs, t % bs] = oracle.encode_e4m3(k_vals[s][t])
            vc[nxt + t // bs, t % bs] = oracle.encode_e4m3(v_vals[s][t])
        nxt += pages[s]
    return (_bf16_bits(q_rows), kc, vc, np.asarray(cu, np.int32), np.asarray(kv, np.int32), bt)


def _vals(rng, shape, top=126):
    """Random finite e4m3 values: codes below `top` (<= 126 keeps clear of the
    NaN code 127), either sign."""
    codes = rng.integers(0, top, size=shape, dtype=np.uint8)
    codes |= (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7)
    return oracle.decode_e4m3(codes)


def test_round_e4m3_matches_the_codec_and_torch():
    rng = np.random.default_rng(11)
    codes = np.arange(256, dtype=np.uint8)
    grid = oracle.decode_e4m3(codes)
    grid = np.unique(grid[~np.isnan(grid)])
    mids = (grid[:-1] + grid[1:]) / 2
    x = np.concatenate([rng.standard_normal(5000) * 40.0, rng.standard_normal(2000) * 2.0 ** -7,
                        grid, mids, rng.uniform(-463.0, 463.0, 2000)]).astype(np.float32)
    ours = F.round_e4m3(x)
    codec = oracle.decode_e4m3(oracle.encode_e4m3(x))
    assert np.array_equal(ours, codec)
    theirs = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ours, theirs)
    big = np.array([470.0, 1e9, np.inf, -1e9])
    assert F.round_e4m3(big).tolist() == [448.0, 448.0, 448.0, -448.0]
    assert np.isnan(F.round_e4m3(np.array([np.nan])))[0]


def test_query_row_quantisation_closed_form():
    # amax 1 -> inv 448: 0.296875 * 448 = 133 -> 128 (steps of 16 in [128, 256));
    # -0.5 * 448 = -224 (on the grid); 2^-12 * 448 = 0.109375 -> 0.109375 (on the
    # grid, steps of 2^-6 in [2^-4, 2^-3))
    row = np.array([1.0, 0.296875, -0.5, 2.0 ** -12, 0.0], dtype=np.float32)
    q8, inv = F.quantize_q_rows(_bf16_bits(row[None, :]))
    assert inv.dtype == np.float32 and inv[0] == np.float32(448.0)
    assert q8[0].tolist() == [448.0, 128.0, -224.0, 0.109375, 0.0]
    # a zero row keeps inv = 1 and quantises to zeros
    q8, inv = F.quantize_q_rows(np.zeros((1, 5), dtype=np.uint16))
    assert inv[0] == 1.0 and not q8.any()


def test_single_visible_key_returns_its_value_row():
    d, hq, hkv = 16, 4, 2
    rng = np.random.default_rng(12)
    q = rng.choice([-1.0, 0.5, 0.25, 1.5], size=(1, hq, d)).astype(np.float32)
    kvals = [_vals(rng, (1, hkv, d), 120)]
    vvals = [_vals(rng, (1, hkv, d))]
    raw = _problem(q, kvals, vvals, [0, 1], [1], hq, hkv)
    out = F.paged_attention_fp8_products(*raw, block_size=16, scale=0.3, k_scale=0.7,
                                         v_scale=1.25)
    for h in range(hq):
        assert np.array_equal(out[0, h], vvals[0][0, h // (hq // hkv)] * 1.25)


def test_identical_keys_give_the_mean_of_the_values():
    """Equal scores: p = 1 for every key of every block, so the output is the
    plain mean of the visible values, across block boundaries."""
    d, hq, hkv, kv = 8, 2, 1, 300
    rng = np.random.default_rng(13)
    q = rng.choice([-1.0, 0.75, 2.0], size=(1, hq, d)).astype(np.float32)
    krow = _vals(rng, (hkv, d), 110)
    kvals = [np.broadcast_to(krow, (kv, hkv, d)).copy()]
    vvals = [_vals(rng, (kv, hkv, d))]
    raw = _problem(q, kvals, vvals, [0, 1], [kv], hq, hkv)
    out = F.paged_attention_fp8_products(*raw, block_size=16, scale=0.2, v_scale=0.5)
    expect = vvals[0][:, 0].mean(axis=0) * 0.5
    for h in range(hq):
        assert np.allclose(out[0, h], expect, rtol=0, atol=1e-12)


def test_two_keys_closed_form():
    """Scores x0 and x0 + ln 0.3: p = (1, 0.3), P rounds to (1, 0.3125), l is
    the sum of the unrounded p (1.3): out = (v0 + 0.3125 v1) / 1.3 * v_scale."""
    d = 4
    q = np.zeros((1, 1, d), dtype=np.float32)
    q[0, 0, 0] = 448.0                              # inv = 1, q8 = q
    k = np.zeros((2, 1, d))
    k[0, 0, 0] = 1.0
    v = np.array([[[1.0, 2.0, -4.0, 0.5]], [[8.0, -1.0, 0.25, 3.0]]])
    scale = -math.log(0.3) / 448.0                   # s0 - s1 = -ln 0.3
    raw = _problem(q, [k], [v], [0, 1], [2], 1, 1)
    out = F.paged_attention_fp8_products(*raw, block_size=16, scale=scale, v_scale=2.0,
                                         causal=False)
    expect = (v[0, 0] + 0.3125 * v[1, 0]) / 1.3 * 2.0
    assert np.allclose(out[0, 0], expect, rtol=1e-14, atol=1e-14)


def _grid_problem(seed, kv_list, hq, hkv, d=16):
    """Every quantisation step exact: q rows 448 e_0 (inv = 1), key values at
    dimension 0 on a grid of 1/8 and scale with 448 * scale = 8 ln 2, so every
    score is a multiple of ln 2 (8 k in log2 units). Keys 0..127 score 0..3,
    later keys 4..12, and the key at 130 scores 12: the reference moves once,
    at the second block (12 > 3 + 8), and every p relative to it is 2^-j with
    0 <= j <= 8 (all e4m3 values)."""
    rng = np.random.default_rng(seed)
    tq = len(kv_list)
    q = np.zeros((tq, hq, d), dtype=np.float32)
    q[:, :, 0] = 448.0
    kvals, vvals = [], []
    for n in kv_list:
        k = np.zeros((n, hkv, d))
        first = min(n, 128)
        k[:first, :, 0] = rng.integers(0, 4, size=(first, hkv)) / 8.0
        if n > 128:
            k[128:, :, 0] = rng.integers(4, 13, size=(n - 128, hkv)) / 8.0
        if n > 130:
            k[130, :, 0] = 12.0 / 8.0
        k[:, :, 1:] = _vals(rng, (n, hkv, d - 1), 120)
        kvals.append(k)
        vvals.append(_vals(rng, (n, hkv, d)))
    cu = list(range(tq + 1))
    return _problem(q, kvals, vvals, cu, kv_list, hq, hkv), 8.0 * math.log(2.0) / 448.0


@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 200)])
def test_exact_grid_equals_the_unquantised_oracle(causal, window):
    """On the exact grid the fp8-products path computes the plain softmax:
    it must equal the exact oracle (oracle.paged_attention) to rounding, over
    many blocks, with a reference that moves (alpha != 1)."""
    (q, kc, vc, cu, kv, bt), scale = _grid_problem(14, [700, 129, 1, 300], 4, 2)
    got = F.paged_attention_fp8_products(q, kc, vc, cu, kv, bt, 16, scale, k_scale=1.0,
                                         v_scale=0.75, causal=causal, window=window)
    exp, _ = oracle.paged_attention(q, kc, vc, cu, kv, bt, 16, scale, kv_dtype="fp8_e4m3",
                                    k_scale=1.0, v_scale=0.75, causal=causal, window=window)
    assert np.allclose(got, exp, rtol=0, atol=1e-12)


def test_lagging_reference_keeps_p_up_to_256():
    """Scores 0 and 8 ln 2 in two blocks: the second block's max exceeds the
    reference by exactly 2^8, which does not move it, so that key's p is 256
    (an e4m3 value) and the output is (v0 + 256 v1) / 257."""
    d = 4
    q = np.zeros((1, 1, d), dtype=np.float32)
    q[0, 0, 0] = 448.0
    n = 129
    k = np.zeros((n, 1, d))
    k[128, 0, 0] = 1.0
    v = np.zeros((n, 1, d))
    v[0, 0] = [1.0, 2.0, -4.0, 0.5]
    v[128, 0] = [8.0, -1.0, 0.25, 3.0]
    # keys 1..127 score like key 0 but carry zero values
    raw = _problem(q, [k], [v], [0, 1], [n], 1, 1)
    out = F.paged_attention_fp8_products(*raw, block_size=16, scale=8 * math.log(2) / 448.0,
                                         causal=False)
    expect = (v[0, 0] * 0 + 256.0 * v[128, 0]) / (128 + 256.0)
    assert np.allclose(out[0, 0], expect + v[0, 0] / 384.0, rtol=1e-13, atol=1e-13)


def test_mutation_unrounded_p_is_caught(monkeypatch):
    monkeypatch.setattr(F, "round_e4m3", lambda x: np.asarray(x, dtype=np.float64))
    with pytest.raises(AssertionError):
        test_two_keys_closed_form()


def test_mutation_stale_alpha_is_caught(monkeypatch):
    real_exp = np.exp

    def attend_without_rescale(q8, inv, K8, V8, keys, vis, scale, k_scale, v_scale, block_n=128):
        # the recurrence with alpha forced to 1 (the running max moves, but
        # earlier blocks are not rescaled)
        n, d = q8.shape
        S = (q8 @ K8.T) * (scale * k_scale) / inv.astype(np.float64)[:, None]
        m = np.full(n, -np.inf)
        l = np.zeros(n)
        acc = np.zeros((n, d))
        for b0 in range(0, int(keys[-1]) + 1, block_n):
            cols = (keys >= b0) & (keys < b0 + block_n)
            mask = vis[:, cols]
            sb = np.where(mask, S[:, cols], -np.inf)
            bm = np.max(sb, axis=1)
            with np.errstate(invalid="ignore"):
                m = np.where(~np.isfinite(m) | (bm > m + F.LAG), np.maximum(m, bm), m)
            p = np.where(mask, real_exp(sb - np.where(np.isfinite(m), m, 0)[:, None]), 0.0)
            l = l + p.sum(axis=1)
            acc = acc + F.round_e4m3(p) @ V8[cols]
        return np.where(l[:, None] > 0, acc * v_scale / l[:, None], 0.0)

    monkeypatch.setattr(F, "attend_fp8_blocks", attend_without_rescale)
    with pytest.raises(AssertionError):
        test_exact_grid_equals_the_unquantised_oracle(True, 0)
