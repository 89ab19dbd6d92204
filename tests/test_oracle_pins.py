"""Pins for the fp64 oracle against things other than itself (CPU only).

Each check below would fail for a plausible mistake in the oracle: a wrong
GQA mapping, an off-by-one causal bound, a wrong page address, a dropped
scale, a wrong e4m3 bias, a wrong combine weight. The mutation tests at the
end plant such mistakes in the oracle and confirm that a pin catches each one.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import oracle.attention as OA
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


# ---------------------------------------------------------------------------
# Independent dense re-materialisation + torch SDPA (a library routine)
# ---------------------------------------------------------------------------

def _dense_kv_by_loops(cache, bt, s, kv, bs):
    """Dense [kv, Hkv, d] float64 rows of one sequence, gathered with plain
    Python loops over the page table (no oracle helper involved)."""
    rows = []
    for t in range(kv):
        page = int(bt[s, t // bs])
        slot = t - (t // bs) * bs
        rows.append(cache[page, slot].to(torch.float64))
    return torch.stack(rows) if rows else torch.zeros((0,) + tuple(cache.shape[2:]), dtype=torch.float64)


def sdpa_reference(case: W.Case):
    """Expected output [Tq, Hq, d] via torch.nn.functional.scaled_dot_product_attention
    in float64 on a dense copy of the cache, with the mask built by torch.tril."""
    cu = case.cu_query_lens.tolist()
    kvl = case.kv_lens.tolist()
    qpk = case.num_q_heads // case.num_kv_heads
    out = torch.zeros(case.q.shape, dtype=torch.float64)
    kc = case.k_cache.to(torch.float64) * (case.k_scale if case.kv_dtype == W.FP8 else 1.0)
    vc = case.v_cache.to(torch.float64) * (case.v_scale if case.kv_dtype == W.FP8 else 1.0)
    for s in range(case.num_seqs):
        q0, q1, kv = cu[s], cu[s + 1], kvl[s]
        ql = q1 - q0
        if ql == 0:
            continue
        K = _dense_kv_by_loops(kc, case.block_tables, s, kv, case.block_size)  # [kv, Hkv, d]
        V = _dense_kv_by_loops(vc, case.block_tables, s, kv, case.block_size)
        K = K.repeat_interleave(qpk, dim=1).permute(1, 0, 2)                   # [Hq, kv, d]
        V = V.repeat_interleave(qpk, dim=1).permute(1, 0, 2)
        Q = case.q[q0:q1].to(torch.float64).permute(1, 0, 2)                   # [Hq, ql, d]
        ctx = kv - ql
        ones = torch.ones(ql, kv, dtype=torch.bool)
        mask = ones.tril(diagonal=ctx) if case.causal else ones.clone()
        if case.window > 0:
            mask &= ~ones.tril(diagonal=ctx - case.window)
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                             scale=case.scale)
        out[q0:q1] = o.permute(1, 0, 2)
    return out.numpy()


def run_oracle(case: W.Case):
    r = case.raw()
    return oracle.paged_attention(r["q"], r["k_cache"], r["v_cache"], r["cu_query_lens"],
                                  r["kv_lens"], r["block_tables"], case.block_size, case.scale,
                                  kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                                  v_scale=case.v_scale, causal=case.causal, window=case.window)


def _small_cases():
    cases = [W.config1_tiny_mixed()]
    for seed in range(4):
        cases.append(W.random_small_case(seed, head_dim=32, num_q_heads=6, num_kv_heads=2,
                                         max_kv=90, max_seqs=4))
    cases.append(W.random_small_case(7, head_dim=16, num_q_heads=4, num_kv_heads=4,
                                     block_size=32, max_kv=120, max_seqs=3))
    cases.append(W.random_small_case(8, kv_dtype=W.FP8, head_dim=32, num_q_heads=8,
                                     num_kv_heads=2, max_kv=80, max_seqs=3))
    cases.append(W.random_small_case(9, head_dim=16, num_q_heads=4, num_kv_heads=1,
                                     max_kv=60, max_seqs=3, window=5))
    cases.append(W.random_small_case(10, head_dim=16, num_q_heads=2, num_kv_heads=1,
                                     max_kv=60, max_seqs=3, causal=False))
    return cases


@pytest.mark.parametrize("case", _small_cases(), ids=lambda c: c.name)
def test_oracle_matches_sdpa_on_dense_copy(case):
    got, _ = run_oracle(case)
    exp = sdpa_reference(case)
    assert np.max(np.abs(got - exp)) <= 1e-12


def test_dense_special_case_is_causal_sdpa():
    """Identity page table and q_len == kv_len: plain dense causal attention."""
    case = W.make_case("dense_small", [48, 48], [48, 48], 2, 2, 32, 16, table="identity")
    got, _ = run_oracle(case)
    for s in range(2):
        q = case.q[48 * s:48 * (s + 1)].to(torch.float64).permute(1, 0, 2)
        k = case.k_cache[3 * s:3 * (s + 1)].reshape(48, 2, 32).to(torch.float64).permute(1, 0, 2)
        v = case.v_cache[3 * s:3 * (s + 1)].reshape(48, 2, 32).to(torch.float64).permute(1, 0, 2)
        exp = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                               scale=case.scale)
        assert np.max(np.abs(got[48 * s:48 * (s + 1)] - exp.permute(1, 0, 2).numpy())) <= 1e-12


# ---------------------------------------------------------------------------
# Hand-derived worked examples (tests/golden)
# ---------------------------------------------------------------------------

def _golden_case(c):
    d, hkv, bs = c["head_dim"], c["num_kv_heads"], c["block_size"]
    q = torch.tensor(c["q"], dtype=torch.float64).to(torch.bfloat16)
    nb = c["num_blocks"]
    tdt = torch.bfloat16 if c["kv_dtype"] == "bf16" else torch.float8_e4m3fn
    kc = torch.zeros((nb, bs, hkv, d), dtype=torch.float32)
    vc = torch.zeros((nb, bs, hkv, d), dtype=torch.float32)
    bt = torch.tensor(c["block_tables"], dtype=torch.int32)
    for s, kv in enumerate(c["kv_lens"]):
        for t in range(kv):
            kc[int(bt[s, t // bs]), t % bs] = torch.tensor(c["k"][s][t])
            vc[int(bt[s, t // bs]), t % bs] = torch.tensor(c["v"][s][t])
    cu = [0]
    for ql in c["query_lens"]:
        cu.append(cu[-1] + ql)
    return W.Case(name=c["name"], q=q, k_cache=kc.to(tdt), v_cache=vc.to(tdt),
                  cu_query_lens=torch.tensor(cu, dtype=torch.int32),
                  kv_lens=torch.tensor(c["kv_lens"], dtype=torch.int32), block_tables=bt,
                  num_q_heads=c["num_q_heads"], num_kv_heads=hkv, head_dim=d, block_size=bs,
                  kv_dtype=c["kv_dtype"], scale=0.5493061443340549, k_scale=c["k_scale"],
                  v_scale=c["v_scale"], causal=c["causal"], window=c["window"])


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("c", _golden(), ids=lambda c: c["name"])
def test_worked_examples(c):
    case = _golden_case(c)
    assert abs(math.log(3.0) / 2 - case.scale) < 1e-16
    out, lse = run_oracle(case)
    assert np.max(np.abs(out - np.array(c["out"]))) <= 1e-15
    assert np.max(np.abs(lse - np.array(c["lse"]))) <= 1e-15


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def test_single_visible_key_returns_its_value_row():
    """window = 1 leaves exactly the key at pos, and query 0 of a fresh prefill
    (ctx = 0) sees key 0 alone: the output is that V row, exactly."""
    case = W.make_case("w1", [7, 1, 20], [7, 33, 50], 4, 2, 32, 16, window=1, seed=3)
    out, lse = run_oracle(case)
    cu = case.cu_query_lens.tolist()
    kvl = case.kv_lens.tolist()
    for s in range(3):
        ql = cu[s + 1] - cu[s]
        for i in range(ql):
            pos = kvl[s] - ql + i
            page = int(case.block_tables[s, pos // 16])
            for h in range(4):
                v = case.v_cache[page, pos % 16, h // 2].to(torch.float64).numpy()
                assert np.array_equal(out[cu[s] + i, h], v)
    case0 = W.make_case("fresh", [30], [30], 2, 2, 16, 16, seed=4)
    out0, _ = run_oracle(case0)
    page0 = int(case0.block_tables[0, 0])
    for h in range(2):
        assert np.array_equal(out0[0, h], case0.v_cache[page0, 0, h].to(torch.float64).numpy())


def test_identical_keys_give_mean_of_visible_values():
    case = W.make_case("same_k", [5, 1], [40, 70], 4, 2, 32, 16, seed=5)
    case.k_cache[:] = case.k_cache[0, 0, 0]
    out, _ = run_oracle(case)
    cu = case.cu_query_lens.tolist()
    kvl = case.kv_lens.tolist()
    for s in range(2):
        ql = cu[s + 1] - cu[s]
        V = _dense_kv_by_loops(case.v_cache.to(torch.float64), case.block_tables, s, kvl[s], 16)
        for i in range(ql):
            pos = kvl[s] - ql + i
            for h in range(4):
                exp = V[:pos + 1, h // 2].mean(0).numpy()
                assert np.max(np.abs(out[cu[s] + i, h] - exp)) <= 1e-13


def test_rows_are_probability_distributions():
    case = W.random_small_case(11, head_dim=32, num_q_heads=4, num_kv_heads=2, max_kv=100)
    r = case.raw()
    rows = [(t, h) for t in range(case.q.shape[0]) for h in range(4)]
    _, _, probs = oracle.paged_attention_rows(r["q"], r["k_cache"], r["v_cache"],
                                              r["cu_query_lens"], r["kv_lens"], r["block_tables"],
                                              16, case.scale, rows, with_probs=True)
    for keys, p in probs:
        assert abs(np.sum(p) - 1.0) <= 1e-12
        assert np.all(p >= 0)
        assert len(keys) == len(p) and len(p) >= 1


def test_lse_matches_scipy_logsumexp():
    case = W.random_small_case(12, head_dim=32, num_q_heads=4, num_kv_heads=2, max_kv=100)
    r = case.raw()
    _, lse = run_oracle(case)
    cu = case.cu_query_lens.tolist()
    kvl = case.kv_lens.tolist()
    for s in range(case.num_seqs):
        ql = cu[s + 1] - cu[s]
        K = _dense_kv_by_loops(case.k_cache.to(torch.float64), case.block_tables, s, kvl[s], 16)
        for i in range(ql):
            pos = kvl[s] - ql + i
            for h in range(4):
                x = case.scale * (K[:pos + 1, h // 2] @ case.q[cu[s] + i, h].to(torch.float64))
                assert abs(lse[cu[s] + i, h] - scipy.special.logsumexp(x.numpy())) <= 1e-12


def test_rows_api_agrees_with_batch_api():
    case = W.random_small_case(13, head_dim=32, num_q_heads=8, num_kv_heads=2, max_kv=200)
    r = case.raw()
    full, lse = run_oracle(case)
    rng = np.random.default_rng(0)
    rows = [(int(rng.integers(case.q.shape[0])), int(rng.integers(8))) for _ in range(20)]
    o, l = oracle.paged_attention_rows(r["q"], r["k_cache"], r["v_cache"], r["cu_query_lens"],
                                       r["kv_lens"], r["block_tables"], 16, case.scale, rows)
    for n, (t, h) in enumerate(rows):
        assert np.max(np.abs(o[n] - full[t, h])) <= 1e-13
        assert abs(l[n] - lse[t, h]) <= 1e-13


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def test_block_permutation_invariance():
    case = W.random_small_case(14, head_dim=32, num_q_heads=4, num_kv_heads=2, max_kv=150)
    out, lse = run_oracle(case)
    nb = case.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(77))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(nb)
    # physical block b moves to slot inv[b]
    k2 = torch.empty_like(case.k_cache)
    v2 = torch.empty_like(case.v_cache)
    k2[inv] = case.k_cache
    v2[inv] = case.v_cache
    bt2 = inv[case.block_tables.long()].to(torch.int32)
    case2 = W.Case(**{**case.__dict__, "k_cache": k2, "v_cache": v2, "block_tables": bt2})
    out2, lse2 = run_oracle(case2)
    assert np.max(np.abs(out - out2)) <= 1e-12
    assert np.max(np.abs(lse - lse2)) <= 1e-12


@pytest.mark.parametrize("nsplit", [1, 2, 3, 16, 128])
def test_split_combine_equals_unsplit(nsplit):
    rng = np.random.default_rng(nsplit)
    n, d = 300, 32
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    q = rng.standard_normal(d)
    keys = np.sort(rng.choice(n, size=250, replace=False))
    o_ref, l_ref, _ = oracle.attend(q, K[keys], V[keys], 0.3)
    bounds = np.linspace(0, n, nsplit + 1).round().astype(int)
    outs, lses = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, l = oracle.partial_attention(q, K, V, 0.3, keys, int(a), int(b))
        outs.append(o)
        lses.append(l)
    # empty chunks are tolerated with weight zero
    outs.append(np.full(d, 123.0))
    lses.append(-np.inf)
    o, l = oracle.combine_partials(outs, lses)
    assert np.max(np.abs(o - o_ref)) <= 1e-12
    assert abs(l - l_ref) <= 1e-12


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def test_e4m3_all_codes_match_torch_conversion():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert nan.sum() == 2  # 0x7F and 0xFF


def test_e4m3_format_landmarks():
    d = oracle.decode_e4m3(np.array([0x7E, 0x01, 0x08, 0x38, 0xB8, 0x00, 0x80, 0x07], np.uint8))
    assert list(d[:5]) == [448.0, 2.0 ** -9, 2.0 ** -6, 1.0, -1.0]
    assert d[5] == 0.0 and d[6] == 0.0 and np.signbit(d[6])
    assert d[7] == 7 * 2.0 ** -9


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(1)
    bits = torch.randint(0, 65536, (20000,), generator=g, dtype=torch.int32).to(torch.int16)
    x = bits.view(torch.bfloat16).to(torch.float64).numpy()
    ours = oracle.decode_bf16(bits.numpy().view(np.uint16))
    nan = np.isnan(x)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], x[~nan])


# ---------------------------------------------------------------------------
# Mutation checks: a planted mistake in the oracle must fail a pin above.
# ---------------------------------------------------------------------------

def _pin_fails(case):
    got, _ = run_oracle(case)
    exp = sdpa_reference(case)
    return not (np.max(np.abs(got - exp)) <= 1e-12)


GQA_CASE = lambda: W.random_small_case(21, head_dim=16, num_q_heads=6, num_kv_heads=3,
                                       max_kv=70, max_seqs=3)


def test_mutation_interleaved_gqa_is_caught(monkeypatch):
    monkeypatch.setattr(OA, "kv_head_of", lambda h, hq, hkv: h % hkv)
    assert _pin_fails(GQA_CASE())


def test_mutation_causal_off_by_one_is_caught(monkeypatch):
    orig = OA.visible_keys

    def wrong(kv, ql, i, causal, window):
        k = orig(kv, ql, i, causal, window)
        return k[:-1] if len(k) > 1 else k
    monkeypatch.setattr(OA, "visible_keys", wrong)
    assert _pin_fails(GQA_CASE())


def test_mutation_top_left_causal_is_caught(monkeypatch):
    orig = OA.visible_keys
    monkeypatch.setattr(OA, "visible_keys", lambda kv, ql, i, c, w: orig(kv, kv, i, c, w))
    assert _pin_fails(GQA_CASE())


def test_mutation_page_slot_is_caught(monkeypatch):
    def wrong(bt, s, t, bs):
        t = np.asarray(t, dtype=np.int64)
        return bt[s, t // bs].astype(np.int64), (t + 1) % bs
    monkeypatch.setattr(OA, "page_address", wrong)
    assert _pin_fails(GQA_CASE())


def test_mutation_page_table_row_is_caught(monkeypatch):
    def wrong(bt, s, t, bs):
        t = np.asarray(t, dtype=np.int64)
        return bt[0, t // bs].astype(np.int64), t % bs
    monkeypatch.setattr(OA, "page_address", wrong)
    assert _pin_fails(W.make_case("three_seqs", [3, 1, 5], [40, 50, 33], 2, 1, 16, 16, seed=22))


def test_mutation_dropped_fp8_scale_is_caught(monkeypatch):
    orig = OA.gather_kv
    monkeypatch.setattr(OA, "gather_kv", lambda c, bt, s, t, g, bs, fmt, sc:
                        orig(c, bt, s, t, g, bs, fmt, 1.0))
    assert _pin_fails(W.random_small_case(23, kv_dtype=W.FP8, head_dim=16, num_q_heads=2,
                                          num_kv_heads=1, max_kv=70, max_seqs=3))


def test_mutation_e4m3_bias_is_caught(monkeypatch):
    orig = OA.decode_e4m3
    monkeypatch.setattr(OA, "decode_e4m3", lambda c: orig(c) * 2.0)
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = OA.decode_e4m3(codes)
    ok = ~np.isnan(ref)
    assert not np.array_equal(ours[ok], ref[ok])


def test_mutation_combine_weight_is_caught(monkeypatch):
    rng = np.random.default_rng(5)
    K, V, q = rng.standard_normal((64, 8)), rng.standard_normal((64, 8)), rng.standard_normal(8)
    keys = np.arange(64)
    o_ref, _, _ = oracle.attend(q, K, V, 0.5)
    parts = [oracle.partial_attention(q, K, V, 0.5, keys, a, a + 16) for a in range(0, 64, 16)]
    outs, lses = zip(*parts)
    wrong_out = sum(outs) / len(outs)   # forgetting the lse weights
    assert np.max(np.abs(wrong_out - o_ref)) > 1e-6
    o, _ = oracle.combine_partials(outs, lses)
    assert np.max(np.abs(o - o_ref)) <= 1e-12


def test_pooled_oracle_equals_the_whole_batch_oracle():
    """oracle.pool cuts a batch into (sequence, KV head) units run in spawned
    processes; the assembled result is the whole-batch definition (GQA groups,
    windows, non-causal masks and fp8 scales included)."""
    from oracle import pool
    cases = [W.config1_tiny_mixed(),
             W.random_small_case(3, kv_dtype=W.FP8, num_q_heads=16, num_kv_heads=4, window=50),
             W.random_small_case(7, causal=False, num_q_heads=6, num_kv_heads=2)]
    for case in cases:
        r = case.raw()
        kw = dict(kv_dtype=case.kv_dtype, k_scale=case.k_scale, v_scale=case.v_scale,
                  causal=case.causal, window=case.window)
        a, la = oracle.paged_attention(r["q"], r["k_cache"], r["v_cache"], r["cu_query_lens"],
                                       r["kv_lens"], r["block_tables"], case.block_size,
                                       case.scale, **kw)
        b, lb = pool.paged_attention_parallel(r, case.block_size, case.scale, workers=3, **kw)
        np.testing.assert_allclose(b, a, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lb, la, rtol=0, atol=1e-12)
    per_round, n = pool.time_units(cases[0].raw(), 16, 0.125, 0.2, workers=2, rounds=2)
    assert n == 2 and len(per_round) == 2
    for done, wall in per_round:
        assert wall > 0 and len(done) >= 1
        assert set(done) <= set(pool.units_of(cases[0].cu_query_lens.numpy(), 4))
