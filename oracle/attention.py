"""fp64 reference for unified paged-KV attention (test infrastructure only).

See the package docstring for the definition and the pages it follows. Each
helper below is one step of that definition, kept separate so that tests can
check (and deliberately break) it step by step.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np

BF16 = "bf16"
FP8 = "fp8_e4m3"


# ---------------------------------------------------------------------------
# Number formats
# ---------------------------------------------------------------------------

def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 word -> float64, exactly.

    bf16 is by definition the upper 16 bits of an IEEE-754 binary32 value, so
    the word shifted left by 16 and reinterpreted as binary32 is its value.
    """
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 code -> float64, from the format definition.

    The e4m3 kernels are named on "flashatten takeaways EP2 工程" (the
    flash_fwd_hdim*_e4m3_sm90 files); the format itself: 1 sign bit, 4
    exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal
    (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN; there are no infinities,
    so the largest finite value is 1.75 * 2^8 = 448.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    val = np.where(e == 0, sub, normal)
    val = np.where((e == 15) & ((c & 0x7) == 7), np.nan, val)
    return sign * val


def widen(raw: np.ndarray, fmt: str) -> np.ndarray:
    if fmt == BF16:
        return decode_bf16(raw)
    if fmt == FP8:
        return decode_e4m3(raw)
    raise ValueError(f"unknown format {fmt}")


# ---------------------------------------------------------------------------
# Steps of the definition
# ---------------------------------------------------------------------------

def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """Query head h reads KV head h // (Hq/Hkv): contiguous GQA groups
    ("vllm_triton_unified_attention_notes", num_queries_per_kv and the
    query_offset_1 bound in the Q-load section)."""
    return h // (num_q_heads // num_kv_heads)


def visible_keys(kv_len: int, q_len: int, i: int, causal: bool, window: int) -> np.ndarray:
    """Key positions visible to query i of a sequence.

    context_len = kv_len - q_len tokens precede the first query
    ("vllm_triton_unified_attention_notes", the M/L/acc/context_len section),
    so query i sits at absolute position pos = context_len + i and, when causal,
    sees keys 0..pos. A positive window keeps only keys with t > pos - window.
    """
    pos = (kv_len - q_len) + i
    t = np.arange(kv_len, dtype=np.int64)
    keep = np.ones(kv_len, dtype=bool)
    if causal:
        keep &= t <= pos
    if window > 0:
        keep &= t > pos - window
    return t[keep]


def page_address(block_tables: np.ndarray, s: int, t: np.ndarray, block_size: int):
    """Logical token t of sequence s -> (physical block, slot in block)
    ("vllm_triton_unified_attention_notes", the paged K/V load section)."""
    t = np.asarray(t, dtype=np.int64)
    return block_tables[s, t // block_size].astype(np.int64), t % block_size


def gather_kv(cache: np.ndarray, block_tables: np.ndarray, s: int, t: np.ndarray,
              g: int, block_size: int, fmt: str, kv_scale: float) -> np.ndarray:
    """Rows K[bt[s, t//bs], t%bs, g, :] widened to fp64 (and dequantised by
    the per-tensor scale for fp8). Returns [len(t), d]."""
    blk, slot = page_address(block_tables, s, t, block_size)
    rows = widen(cache[blk, slot, g, :], fmt)
    if fmt == FP8:
        rows = rows * float(kv_scale)
    return rows


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """softmax(scale * q K^T) V for one query row over the given key rows.

    Returns (out [d], lse (natural log), p [n]). Max subtraction is only the
    usual overflow guard; the result is the plain softmax.
    """
    x = scale * (K @ q)
    if x.size == 0:
        return np.zeros(V.shape[1]), -np.inf, x
    m = np.max(x)
    e = np.exp(x - m)
    z = np.sum(e)
    p = e / z
    return p @ V, m + np.log(z), p


# ---------------------------------------------------------------------------
# Whole batch
# ---------------------------------------------------------------------------

def _seq_of_tokens(cu: np.ndarray) -> np.ndarray:
    B = len(cu) - 1
    out = np.empty(int(cu[-1]), dtype=np.int64)
    for s in range(B):
        out[cu[s]:cu[s + 1]] = s
    return out


def paged_attention_rows(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                         cu_query_lens: np.ndarray, kv_lens: np.ndarray,
                         block_tables: np.ndarray, block_size: int, scale: float,
                         rows: Iterable[Tuple[int, int]], kv_dtype: str = BF16,
                         k_scale: float = 1.0, v_scale: float = 1.0, causal: bool = True,
                         window: int = 0, with_probs: bool = False):
    """Attention output for selected (query token index, query head) rows.

    Returns (out [n, d] fp64, lse [n] natural log[, list of (keys, probs)]).
    Rows of one (sequence, KV head) share one gather of K and V.
    """
    cu = np.asarray(cu_query_lens, dtype=np.int64)
    kvl = np.asarray(kv_lens, dtype=np.int64)
    bt = np.asarray(block_tables, dtype=np.int64)
    Hq = q_bits.shape[1]
    Hkv = k_cache.shape[2]
    d = q_bits.shape[2]
    rows = list(rows)
    seq_of = _seq_of_tokens(cu)
    groups: Dict[Tuple[int, int], List[int]] = {}
    for n, (tok, h) in enumerate(rows):
        s = int(seq_of[tok])
        groups.setdefault((s, kv_head_of(h, Hq, Hkv)), []).append(n)
    out = np.zeros((len(rows), d))
    lse = np.full(len(rows), -np.inf)
    probs = [None] * len(rows)
    for (s, g), idx in groups.items():
        qlen = int(cu[s + 1] - cu[s])
        kv = int(kvl[s])
        t_all = np.arange(kv, dtype=np.int64)
        K = gather_kv(k_cache, bt, s, t_all, g, block_size, kv_dtype, k_scale)
        V = gather_kv(v_cache, bt, s, t_all, g, block_size, kv_dtype, v_scale)
        for n in idx:
            tok, h = rows[n]
            i = tok - int(cu[s])
            vis = visible_keys(kv, qlen, i, causal, window)
            qv = decode_bf16(q_bits[tok, h, :])
            o, l, p = attend(qv, K[vis], V[vis], scale)
            out[n] = o
            lse[n] = l
            if with_probs:
                probs[n] = (vis, p)
    if with_probs:
        return out, lse, probs
    return out, lse


def paged_attention(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                    cu_query_lens: np.ndarray, kv_lens: np.ndarray, block_tables: np.ndarray,
                    block_size: int, scale: float, kv_dtype: str = BF16, k_scale: float = 1.0,
                    v_scale: float = 1.0, causal: bool = True, window: int = 0):
    """Whole-batch output [Tq, Hq, d] and lse [Tq, Hq] (natural log), fp64.

    Same definition as paged_attention_rows; per (sequence, KV head) the
    scores of all its query rows are formed with one matrix product (a library
    primitive) and masked row by row with visible_keys.
    """
    cu = np.asarray(cu_query_lens, dtype=np.int64)
    kvl = np.asarray(kv_lens, dtype=np.int64)
    bt = np.asarray(block_tables, dtype=np.int64)
    Tq, Hq, d = q_bits.shape
    Hkv = k_cache.shape[2]
    out = np.zeros((Tq, Hq, d))
    lse = np.full((Tq, Hq), -np.inf)
    B = len(kvl)
    for s in range(B):
        q0, q1 = int(cu[s]), int(cu[s + 1])
        qlen, kv = q1 - q0, int(kvl[s])
        if qlen == 0:
            continue
        t_all = np.arange(kv, dtype=np.int64)
        masks = np.zeros((qlen, kv), dtype=bool)
        for i in range(qlen):
            masks[i, visible_keys(kv, qlen, i, causal, window)] = True
        for g in range(Hkv):
            K = gather_kv(k_cache, bt, s, t_all, g, block_size, kv_dtype, k_scale)
            V = gather_kv(v_cache, bt, s, t_all, g, block_size, kv_dtype, v_scale)
            for h in range(Hq):
                if kv_head_of(h, Hq, Hkv) != g:
                    continue
                Q = decode_bf16(q_bits[q0:q1, h, :])          # [qlen, d]
                X = scale * (Q @ K.T)                          # [qlen, kv]
                X = np.where(masks, X, -np.inf)
                m = np.max(X, axis=1, keepdims=True)
                E = np.where(masks, np.exp(X - m), 0.0)
                Z = np.sum(E, axis=1, keepdims=True)
                out[q0:q1, h, :] = (E / Z) @ V
                lse[q0:q1, h] = (m + np.log(Z))[:, 0]
    return out, lse


# ---------------------------------------------------------------------------
# Split-KV and its log-sum-exp combine
# ---------------------------------------------------------------------------

def partial_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                      keys: np.ndarray, t0: int, t1: int):
    """Attention of one query row over the visible keys that fall in [t0, t1).

    This is FlashDecoding's per-chunk step ("Fused Attention" notes,
    FlashDecoding section: split K/V into chunks and attend to each): the
    normalised partial output and its lse. An empty chunk gives lse = -inf
    and a zero output, which carries zero weight in the combine.
    """
    sel = keys[(keys >= t0) & (keys < t1)]
    o, l, _ = attend(q, K[sel], V[sel], scale)
    return o, l


def combine_partials(outs: Sequence[np.ndarray], lses: Sequence[float]):
    """Global reduction of per-chunk results by their log-sum-exp
    ("flashatten takeaways EP2 工程", the split-KV combine step):
    lse* = log sum_s exp(lse_s); out = sum_s exp(lse_s - lse*) out_s."""
    lses = np.asarray(lses, dtype=np.float64)
    finite = np.isfinite(lses)
    if not finite.any():
        return np.zeros_like(np.asarray(outs[0])), -np.inf
    m = np.max(lses[finite])
    w = np.where(finite, np.exp(np.where(finite, lses, 0.0) - m), 0.0)
    z = np.sum(w)
    lse_star = m + np.log(z)
    out = np.zeros_like(np.asarray(outs[0], dtype=np.float64))
    for ws, o in zip(w / z, outs):
        if ws != 0.0:
            out = out + ws * np.asarray(o, dtype=np.float64)
    return out, lse_star
