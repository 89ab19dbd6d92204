"""C-ABI library checks that need no GPU: exports, validation, the scheduler.

The scheduler's tile lists are compared with a brute-force enumeration of
which rows exist and which keys each row can see (exact integer equality).
"""
import os
import re

import numpy as np
import pytest

import paged_kv_attention_unified_gb300 as ua

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_kv_attention_unified_gb300 import build
    build.build()


def _header_functions():
    txt = open(os.path.join(ROOT, "include", "ua.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^(?:ua_status|const char\*)\s+(ua_\w+)\s*\(", txt, flags=re.M)))


def test_library_exports_every_declared_symbol():
    names = _header_functions()
    assert len(names) >= 10
    assert sorted(ua.EXPORTS) == names
    lib = ua.lib()
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings():
    for code in range(-6, 1):
        s = ua.ua_status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in ua.ua_status_string(-99)


BAD = [
    dict(cu=[0, 1], kv=[0]),                         # kv_len < q_len
    dict(cu=[1, 2], kv=[5]),                         # cu[0] != 0
    dict(cu=[0, 3, 2], kv=[5, 5]),                   # negative q_len
    dict(cu=[0, 1], kv=[5], hq=6, hkv=4),            # Hq % Hkv != 0
    dict(cu=[0, 1], kv=[500], max_blocks=2),          # page table too short
    dict(cu=[0, 1], kv=[5], num_splits=129),          # too many splits
    dict(cu=[0, 1], kv=[5], dtype=7),                 # unknown dtype
    dict(cu=[0, 1], kv=[-1]),                         # negative kv_len
]


@pytest.mark.parametrize("bad", BAD)
def test_invalid_problems_are_rejected(bad):
    with pytest.raises(ua.UAError) as e:
        ua.ua_schedule(bad["cu"], bad["kv"], bad.get("hq", 4), bad.get("hkv", 4), 128, 16,
                       bad.get("max_blocks", 64), kv_dtype=bad.get("dtype", 0),
                       num_splits=bad.get("num_splits", 0))
    assert e.value.status == ua.UA_ERR_INVALID_ARG


@pytest.mark.parametrize("d,bs", [(80, 16), (128, 8), (512, 16), (16, 16), (288, 16), (64, 24)])
def test_unsupported_shapes(d, bs):
    with pytest.raises(ua.UAError) as e:
        ua.ua_schedule([0, 1], [5], 4, 4, d, bs, 64)
    assert e.value.status == ua.UA_ERR_UNSUPPORTED


def test_empty_batch_schedules_nothing():
    info, pre, dec, grp = ua.ua_schedule([0], [], 4, 4, 128, 16, 1)
    assert (info.num_prefill_tiles, info.num_decode_tiles, info.num_combine_groups) == (0, 0, 0)
    info, pre, dec, grp = ua.ua_schedule([0, 0, 0], [0, 7], 4, 4, 128, 16, 1)
    assert info.num_decode_tiles == 0 and info.num_prefill_tiles == 0


def _visible(kv, ql, i, causal, window):
    """Every key position, tested one by one (vectorised with numpy)."""
    pos = kv - ql + i
    t = np.arange(kv)
    keep = np.ones(kv, dtype=bool)
    if causal:
        keep &= ~(t > pos)
    if window > 0:
        keep &= ~(t <= pos - window)
    return t[keep]


def _check_schedule(cu, kv, hq, hkv, causal=1, window=0, num_splits=0, num_sms=152,
                    decode_rows_max=-1, d=128):
    info, pre, dec, grp = ua.ua_schedule(cu, kv, hq, hkv, d, 16, 1 + max(kv) // 16 + 1,
                                         causal=causal, window=window, num_splits=num_splits,
                                         num_sms=num_sms, decode_rows_max=decode_rows_max)
    qpk = hq // hkv
    # the prefill kernels take bf16 caches with qpk dividing 128 (block size 16
    # here) at head_dim 64, 128, 192 and 256
    prefill_ok = 128 % qpk == 0 and d in (64, 128, 192, 256)
    rows_max = (2 ** 63) if not prefill_ok else (32 if decode_rows_max < 0 else decode_rows_max)
    seen = {}
    for kind, tiles, rows_per in (("pre", pre, ua.UA_PREFILL_ROWS), ("dec", dec, 8)):
        for t in tiles:
            assert 1 <= t["nrows"] <= rows_per
            for r in range(t["row0"], t["row0"] + t["nrows"]):
                key = (t["seq"], t["kv_head"], r)
                seen.setdefault(key, []).append((kind, t))
    # every (seq, kv head, row) exists exactly once (split pieces share a row)
    expected = set()
    for s in range(len(kv)):
        ql = cu[s + 1] - cu[s]
        for g in range(hkv):
            for r in range(ql * qpk):
                expected.add((s, g, r))
    assert set(seen) == expected
    bounds = {}
    for (s, g, r), owners in seen.items():
        ql = cu[s + 1] - cu[s]
        kind = owners[0][0]
        assert all(k == kind for k, _ in owners)
        assert kind == ("dec" if ql * qpk <= rows_max else "pre")
        pieces = sorted((t["kv_lo"], t["kv_hi"]) for _, t in owners)
        # pieces are contiguous and disjoint
        for (a0, a1), (b0, b1) in zip(pieces, pieces[1:]):
            assert a1 == b0
        lo, hi = pieces[0][0], pieces[-1][1]
        # the tile's range is exactly the floor-16 of the lowest and one past the
        # highest key visible to any of its rows
        t0 = owners[0][1]
        bkey = (s, t0["row0"], t0["nrows"])
        if bkey not in bounds:
            vmin, vmax = None, None
            for i in sorted({rr // qpk for rr in range(t0["row0"], t0["row0"] + t0["nrows"])}):
                v = _visible(kv[s], ql, i, causal, window)
                vmin = v.min() if vmin is None else min(vmin, v.min())
                vmax = v.max() if vmax is None else max(vmax, v.max())
            bounds[bkey] = (vmin, vmax)
        vmin, vmax = bounds[bkey]
        assert hi == vmax + 1
        align = 16 if kind == "dec" else 128
        assert lo == (vmin // align) * align
        assert lo % 16 == 0 and all(p[0] % 16 == 0 for p in pieces)
        assert hi <= kv[s]
        if len(owners) > 1:
            assert len(owners) <= 128
            gids = {t["group"] for _, t in owners}
            assert len(gids) == 1
            gg = grp[gids.pop()]
            assert gg["nsplits"] == len(owners)
            assert sorted(t["slot"] for _, t in owners) == list(
                range(gg["slot0"], gg["slot0"] + gg["nsplits"]))
            if num_splits > 0:
                assert len(owners) <= num_splits
        else:
            assert owners[0][1]["slot"] == -1 and owners[0][1]["group"] == -1
    # slots are used once each
    slots = [t["slot"] for t in dec if t["slot"] >= 0]
    assert sorted(slots) == list(range(info.num_slots))
    # longest-first order
    work = [(t["kv_hi"] - t["kv_lo"]) * t["nrows"] for t in dec]
    assert work == sorted(work, reverse=True)
    # equal work keeps (sequence, KV head, row, key) order
    key = lambda t: (t["seq"], t["kv_head"], t["row0"], t["kv_lo"])
    for a, b, wa, wb in zip(dec, dec[1:], work, work[1:]):
        if wa == wb:
            assert key(a) < key(b)
    if not dec:
        assert info.num_prefill_ctas == min(num_sms, len(pre))
    else:
        assert 1 <= info.num_prefill_ctas <= min(num_sms, len(pre)) or not pre
    return info, pre, dec, grp


def test_schedule_tiny_mixed():
    _check_schedule([0, 1, 6, 23], [40, 130, 300], 4, 4)


def test_schedule_tiny_mixed_with_prefill_kernel():
    _check_schedule([0, 1, 6, 23], [40, 130, 300], 4, 4, decode_rows_max=16)


@pytest.mark.parametrize("ns", [1, 2, 3, 16, 128])
def test_schedule_forced_splits(ns):
    _check_schedule([0, 1, 2, 4], [3000, 17, 900], 32, 8, num_splits=ns)


def test_schedule_window_and_noncausal():
    _check_schedule([0, 3, 4, 40], [100, 1000, 70], 8, 2, window=37)
    _check_schedule([0, 3, 4, 40], [100, 1000, 70], 8, 2, causal=0)
    _check_schedule([0, 3, 4, 40], [100, 1000, 70], 8, 2, causal=0, window=5,
                    decode_rows_max=8)


def test_schedule_auto_splits_long_decode():
    info, _, dec, grp = _check_schedule([0] + list(range(1, 9)), [131072] * 8, 64, 8)
    # every (sequence, KV head) is cut; each sequence gets >= 16 split pieces
    assert info.num_combine_groups == 64
    for s in range(8):
        assert sum(g["nsplits"] for g in grp if g["seq"] == s) >= 16
    assert info.workspace_bytes == info.num_slots * 8 * 129 * 4


def test_schedule_random_brute_force():
    import random
    rng = random.Random(0)
    for it in range(30):
        B = rng.randint(1, 6)
        hkv = rng.choice([1, 2, 4])
        hq = hkv * rng.choice([1, 2, 4, 8, 16])
        cu, kv = [0], []
        for _ in range(B):
            k = rng.randint(0, 600)
            q = rng.choice([0, 1, rng.randint(0, k), k]) if k else 0
            q = min(q, k)
            cu.append(cu[-1] + q)
            kv.append(k)
        if max(kv) == 0:
            kv[0] = 1
        _check_schedule(cu, kv, hq, hkv, causal=rng.choice([0, 1]), window=rng.choice([0, 0, 9]),
                        num_splits=rng.choice([0, 0, 1, 3, 7]), num_sms=rng.choice([2, 152]),
                        decode_rows_max=rng.choice([-1, 8, 32]))


def _prefill_cost(t, cu, kv, qpk, causal=1):
    """128 x 128 query-key blocks of one prefill tile (both 128-row query tiles)."""
    s = t["seq"]
    ql = cu[s + 1] - cu[s]
    ctx = kv[s] - ql
    cost = 0
    for r0 in range(t["row0"], t["row0"] + t["nrows"], 128):
        rows = min(128, t["row0"] + t["nrows"] - r0)
        hi = min(kv[s], ctx + (r0 + rows - 1) // qpk + 1) if causal else kv[s]
        cost += max(0, -(-(hi - t["kv_lo"]) // 128))
    return cost


@pytest.mark.parametrize("case", ["dense", "mixed"])
def test_prefill_list_ends_with_shortest_tiles(case):
    """The persistent prefill CTAs take tiles in list order: the shortest tiles,
    up to 1/16 of the work, come last and longest first; the rest keeps the
    (sequence, KV head) grouping."""
    if case == "dense":
        cu, kv, hq, hkv = [0, 4096, 8192, 12288, 16384], [4096] * 4, 32, 32
    else:
        rng = np.random.default_rng(3)
        ql = [int(x) for x in rng.integers(512, 2049, 8)] + [1] * 20
        kv = [q + int(c) for q, c in zip(ql[:8], rng.integers(0, 1025, 8))] + \
             [int(x) for x in rng.integers(1024, 8193, 20)]
        cu = [0] + list(np.cumsum(ql))
        hq, hkv = 32, 8
    cu = [int(x) for x in cu]
    info, pre, dec, grp = ua.ua_schedule(cu, kv, hq, hkv, 128, 16, max(kv) // 16 + 2)
    qpk = hq // hkv
    cost = [_prefill_cost(t, cu, kv, qpk) for t in pre]
    total = sum(cost)
    # size of the tail: the shortest tiles whose cost adds up to at most 1/16
    m, acc = 0, 0
    for c in sorted(cost):
        if acc + c > total / 16:
            break
        acc += c
        m += 1
    assert 0 < m < len(pre)
    tail, bulk = cost[len(pre) - m:], cost[:len(pre) - m]
    assert tail == sorted(tail, reverse=True)
    assert max(tail) <= min(bulk)
    assert sum(tail) <= total / 16
    # the bulk keeps each (sequence, KV head) group contiguous
    seen, prev = set(), None
    for t in pre[:len(pre) - m]:
        key = (t["seq"], t["kv_head"])
        if key != prev:
            assert key not in seen
            seen.add(key)
            prev = key
    if case == "dense":
        assert info.num_prefill_ctas == min(152, len(pre))
    else:   # mixed: some SMs are left to the decode kernel
        assert 1 <= info.num_prefill_ctas < min(152, len(pre))


def _mixed_ctas(n_prefill_seqs, prefill_q, n_decode, decode_kv):
    ql = [prefill_q] * n_prefill_seqs + [1] * n_decode
    kv = [prefill_q] * n_prefill_seqs + [decode_kv] * n_decode
    cu = [0] + [int(x) for x in np.cumsum(ql)]
    info, pre, dec, _ = ua.ua_schedule(cu, kv, 32, 8, 128, 16, max(kv) // 16 + 1)
    return info.num_prefill_ctas, len(pre)


def test_mixed_prefill_cta_count_follows_the_work_balance():
    """With decode work in the batch the prefill kernel gets fewer SMs: more as
    its share of the work grows, all of them (up to its tile count) when there
    is no decode work, and at least one."""
    alone, tiles = _mixed_ctas(4, 2048, 0, 0)
    assert alone == min(152, tiles)
    counts = [_mixed_ctas(4, 2048, nd, 8192)[0] for nd in (8, 64, 256, 1024)]
    assert all(a >= b for a, b in zip(counts, counts[1:])), counts   # more decode -> fewer
    assert counts[-1] >= 1 and counts[0] <= 152
    grow = [_mixed_ctas(ns, 2048, 128, 4096)[0] for ns in (1, 4, 16)]
    assert all(a <= b for a, b in zip(grow, grow[1:])), grow       # more prefill -> more


def _piece_lengths(dec):
    return [t["kv_hi"] - t["kv_lo"] for t in dec]


def _waves(n, slots):
    return -(-n // slots)


def test_uniform_decode_splits_fill_whole_waves():
    """64 (sequence, KV head) tiles of 131072 keys on 152 x 3 CTA slots: the
    average-load piece (18400 keys) would give 8 pieces per tile, 512 CTAs,
    whose last 56 hold only the 12 % tails; 7 equal pieces (448 CTAs) run in
    one wave."""
    info, _, dec, grp = _check_schedule([0] + list(range(1, 9)), [131072] * 8, 64, 8)
    assert len(dec) == 448 and _waves(len(dec), 456) == 1
    lens = _piece_lengths(dec)
    assert max(lens) - min(lens) <= 16 * 7
    assert all(g["nsplits"] == 7 for g in grp)
    # 128 tiles of 16384 keys (too few to fill HBM unsplit): the chosen cut
    # beats both the average-load chunk (4608 keys: 4 pieces, 512 CTAs, 2
    # waves) and no split (16384 keys)
    info, _, dec, grp = _check_schedule(list(range(17)), [16384] * 16, 32, 8)
    lens = _piece_lengths(dec)
    per_tile = len(dec) // 128
    assert per_tile > 1
    assert _waves(len(dec), 456) * (max(lens) + 128) < min(2 * (4608 + 128), 16384 + 128)
    assert all(g["nsplits"] == per_tile for g in grp)


def test_uniform_bf16_batches_that_fill_hbm_stay_unsplit():
    """256 tiles of 8192 keys (bf16, d128): one CTA each, 1.7 per SM, already
    stream at the copy peak, so they stay unsplit; the same batch over an
    e4m3 cache (whose CTAs are slower) and a 255-tile batch are split."""
    info, _, dec, _ = _check_schedule(list(range(33)), [8192] * 32, 32, 8)
    assert len(dec) == 256 and info.num_combine_groups == 0 and info.split_tokens == 0
    info, _, dec, _ = ua.ua_schedule(list(range(33)), [8192] * 32, 32, 8, 128, 16, 513,
                                     kv_dtype=ua.UA_KV_FP8_E4M3)
    assert len(dec) > 256
    # 255 tiles: fewer than the saturating count, so split into whole waves
    info, _, dec, _ = ua.ua_schedule(list(range(256)), [8192] * 255, 8, 1, 128, 16, 513)
    assert len(dec) > 255


def test_nonuniform_decode_keeps_the_average_load_chunk():
    """Lengths that differ by more than 1/16 keep the chunk of about one CTA
    slot's average load (longest-first order balances the rest)."""
    import random
    rng = random.Random(3)
    kv = [rng.randint(512, 4096) for _ in range(64)]
    info, _, dec, _ = _check_schedule(list(range(65)), kv, 32, 8)
    total = 8 * sum(kv)
    chunk = max(256, -(-total // 456))
    chunk = -(-chunk // 16) * 16
    assert info.split_tokens == chunk
    assert max(_piece_lengths(dec)) == chunk


def test_short_tiles_overfilling_one_wave_split_only_their_tail():
    """512 unsplit window tiles (about 1024 keys) on 456 CTA slots: the 56
    tiles that start last in longest-first order are cut into pieces of at
    least 256 keys (at most 456 // 56 = 8 each), ordered after every whole
    tile; the other 456 stay whole. Batches that overfill by more than half a
    wave keep their tiles whole."""
    import random
    rng = random.Random(0)
    kv = [rng.randint(512, 4096) for _ in range(64)]
    info, _, dec, grp = _check_schedule(list(range(65)), kv, 32, 8, window=1024)
    assert info.split_tokens == 0
    whole = [t for t in dec if t["group"] < 0]
    pieces = [t for t in dec if t["group"] >= 0]
    assert len(whole) == 456 and len(grp) == 56
    assert all(2 <= g["nsplits"] <= 8 for g in grp)
    assert min(_piece_lengths(pieces)) >= 256 - 16
    # every piece is scheduled after every whole tile, and the split tiles are
    # the shortest ones
    first_piece = min(i for i, t in enumerate(dec) if t["group"] >= 0)
    assert all(t["group"] < 0 for t in dec[:first_piece]) and first_piece == 456
    tile_len = {}
    for t in dec:
        key = (t["seq"], t["kv_head"])
        tile_len[key] = tile_len.get(key, 0) + t["kv_hi"] - t["kv_lo"]
    split = {(g["seq"], g["kv_head"]) for g in grp}
    assert max(tile_len[k] for k in split) <= min(v for k, v in tile_len.items() if k not in split)
    # 64 more sequences: 1024 tiles, more than half a wave late -> no split
    kv2 = kv + kv
    info, _, dec, grp = _check_schedule(list(range(129)), kv2, 32, 8, window=1024)
    assert len(grp) == 0 and len(dec) == 1024


def test_head_dim_256_splits_for_one_cta_per_sm():
    """At head_dim 256 the decode kernel holds one CTA per SM: uniform pieces
    are sized for 152 slots (whole waves of 152 CTAs)."""
    info, _, dec, _ = _check_schedule([0] + list(range(1, 9)), [131072] * 8, 64, 8, d=256)
    assert len(dec) % 152 == 0 or len(dec) < 152


def test_unified_max_rejects_a_null_plan_without_touching_cuda():
    lib = ua.lib()
    assert lib.ua_plan_set_unified_max(None, 1, 2.0) == ua.UA_ERR_INVALID_ARG
    assert lib.ua_plan_set_unified_max(None, 0, 0.0) == ua.UA_ERR_INVALID_ARG


def test_append_rejects_a_null_plan_without_touching_cuda():
    lib = ua.lib()
    st = lib.ua_append_kv(None, 16, 16, 16, 16, 16, 1, 1.0, 1.0, None)
    assert st == ua.UA_ERR_INVALID_ARG


def test_head_dim_256_prefills_go_to_the_wide_prefill_kernel():
    """head_dim 256: long prefills run in the wide (one 128-row query tile,
    64-key tiles) prefill kernel, single tokens in the decode kernel; block
    sizes that do not divide or are not divided by 64 keep everything in the
    decode kernel. Every row lands in exactly one tile."""
    info, pre, dec, grp = ua.ua_schedule([0, 1, 301], [500, 800], 8, 2, 256, 16, 64)
    assert info.num_prefill_tiles > 0 and info.num_decode_tiles > 0
    assert {t["seq"] for t in pre} == {1} and {t["seq"] for t in dec} == {0}
    rows = {(t["seq"], t["kv_head"], r) for t in pre + dec
            for r in range(t["row0"], t["row0"] + t["nrows"])}
    assert len(rows) == (1 + 300) * 4 * 2
    info, pre, dec, _ = ua.ua_schedule([0, 1, 301], [500, 800], 8, 2, 256, 48, 17)
    assert info.num_prefill_tiles == 0 and info.num_decode_tiles > 0

def test_fp8_products_setter_rejects_a_null_plan_without_touching_cuda():
    lib = ua.lib()
    assert lib.ua_plan_set_fp8_products(None, 1) == ua.UA_ERR_INVALID_ARG
    assert lib.ua_plan_set_fp8_products(None, 0) == ua.UA_ERR_INVALID_ARG
