"""Reference for attention with fp8 tensor-core products over an fp8 cache
(test infrastructure only; see the package docstring).

What it computes: the low-precision variant of the fused attention forward.
The "Fused Attention" notes run Q.K^T on fp8 operands and cast P to the input
type before P.V (the FP8 path of their _attn_fwd_inner / bench_flash_attention:
q, k, v converted to an 8-bit float, `p = p.to(dtype)` ahead of the second
dot), and their FlashAttention-3 summary names the block-quantised FP8 path of
Hopper. Over a paged e4m3 cache with per-tensor scales k_scale, v_scale:

  1. each query row (one token, one head) is quantised to e4m3 with its own
     scale: amax = max |q|, inv = 448 / amax (binary32 division; 1 for a zero
     row), q8 = e4m3(q * inv) (product in binary32, rounded to nearest even,
     saturating). The row's value is q8 / inv.
  2. scores s = scale * (q8 . k8) * k_scale / inv, over the visible keys
     (k8 the cache's e4m3 values), exactly as in the bf16 definition
     otherwise (causal / window / key range).
  3. online softmax over key blocks of BLOCK_N = 128 keys aligned to multiples
     of 128 (the blocks of the tutorial's inner loop), against a reference
     m_b that follows the running max lazily: m_b = max(m_{b-1}, max s over
     the block) when that exceeds m_{b-1} by more than 8 ln 2 (or m_{b-1} is
     -inf), else m_b = m_{b-1}; alpha = exp(m_{b-1} - m_b), p = exp(s - m_b)
     over the block (so p <= 2^8), l = l * alpha + sum p (from p before the
     cast, as the tutorial sums p ahead of `p.to(dtype)`), and
     acc = acc * alpha + e4m3(p) . v8 (p rounded to e4m3, nearest even).
  4. out = acc * v_scale / l (rows with no visible key: 0).

Readings (where the pages leave the step open): one quantisation scale per
query row (the finest "block" of the block quantisation, and exact for the
largest element of every row); P cast to e4m3 as it stands (the tutorial
casts p as it stands), against a reference that moves only when the row max
has grown by more than 2^8: the exact-max recurrence of the tutorial gives
the same softmax, and a lagging reference keeps p within [0, 2^8], inside
e4m3's range (448), while weights down to 2^-10 of the reference survive
the cast (e4m3 keeps values down to 2^-9); l from the unrounded p (the
tutorial's l_ij is the sum of p before the cast).

Everything is in binary64 except the two quantisation decisions, which take
the binary32 values the GPU path also rounds.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

from .attention import FP8, decode_bf16, gather_kv, kv_head_of, visible_keys

BLOCK_N = 128
E4M3_MAX = 448.0
# The reference max moves when the block max exceeds it by more than this
# (natural-log units; 8 in log2 units).
LAG = 8.0 * np.log(2.0)


def round_e4m3(x: np.ndarray) -> np.ndarray:
    """Values rounded to the OCP E4M3 grid (nearest, ties to even), saturating
    to +-448; NaN stays NaN. Vectorised form of the format's definition: steps
    of 2^-9 below 2^-6 (subnormals), steps of 2^(E-3) in the binade
    [2^E, 2^(E+1)) above."""
    v = np.asarray(x, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore", invalid="ignore"):
        _, e2 = np.frexp(a)                    # a = f * 2^e2, f in [0.5, 1)
        e = np.maximum(e2.astype(np.int64) - 1, -6)   # binade exponent, subnormals share -6
        step = np.exp2((e - 3).astype(np.float64))
        r = np.rint(a / step) * step
    r = np.minimum(r, E4M3_MAX)
    r = np.where(np.isnan(v), np.nan, r)
    return np.copysign(r, v)


def quantize_q_rows(q_bits: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Step 1: bf16 query rows [..., d] -> (e4m3 values [..., d] as binary64,
    inv [...] as binary32): q8 = e4m3(q * inv), inv = 448 / max |q|."""
    q = decode_bf16(q_bits).astype(np.float32)
    amax = np.max(np.abs(q), axis=-1)
    with np.errstate(divide="ignore"):
        inv = np.where(amax > 0, np.float32(E4M3_MAX) / amax, np.float32(1.0)).astype(np.float32)
    y = (q * inv[..., None]).astype(np.float32)
    return round_e4m3(y.astype(np.float64)), inv


def attend_fp8_blocks(q8: np.ndarray, inv: np.ndarray, K8: np.ndarray, V8: np.ndarray,
                      keys: np.ndarray, vis: np.ndarray, scale: float, k_scale: float,
                      v_scale: float, block_n: int = BLOCK_N) -> np.ndarray:
    """Steps 2-4 for the query rows of one (sequence, head).

    q8 [n, d], inv [n]: quantised rows; K8, V8 [kv, d]: e4m3 cache values of
    the sequence's keys; keys [kv] their positions; vis [n, kv] the visibility
    mask. Returns out [n, d] (binary64).
    """
    n, d = q8.shape
    S = (q8 @ K8.T) * (float(scale) * float(k_scale)) / inv.astype(np.float64)[:, None]
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    acc = np.zeros((n, d))
    kv = K8.shape[0]
    if kv == 0:
        return acc
    for b0 in range(0, int(keys[-1]) + 1, block_n):
        cols = (keys >= b0) & (keys < b0 + block_n)
        if not cols.any():
            continue
        mask = vis[:, cols]
        sb = np.where(mask, S[:, cols], -np.inf)
        bmax = np.max(sb, axis=1)
        m_max = np.maximum(m, bmax)
        with np.errstate(invalid="ignore"):
            grow = ~np.isfinite(m) | (m_max > m + LAG)
        m_new = np.where(grow, m_max, m)
        live = np.isfinite(m_new)
        with np.errstate(invalid="ignore"):
            alpha = np.where(live & np.isfinite(m), np.exp(m - m_new), 0.0)
            p = np.where(mask & live[:, None], np.exp(sb - np.where(live, m_new, 0.0)[:, None]),
                         0.0)
        l = l * alpha + np.sum(p, axis=1)
        acc = acc * alpha[:, None] + round_e4m3(p) @ V8[cols]
        m = np.where(live, m_new, m)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(l[:, None] > 0, acc * float(v_scale) / l[:, None], 0.0)
    return out


def paged_attention_fp8_products(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                                 cu_query_lens: np.ndarray, kv_lens: np.ndarray,
                                 block_tables: np.ndarray, block_size: int, scale: float,
                                 k_scale: float = 1.0, v_scale: float = 1.0, causal: bool = True,
                                 window: int = 0, block_n: int = BLOCK_N) -> np.ndarray:
    """Whole-batch output [Tq, Hq, d] (binary64) of the fp8-products path over
    an e4m3 cache (k_cache / v_cache hold e4m3 codes)."""
    cu = np.asarray(cu_query_lens, dtype=np.int64)
    kvl = np.asarray(kv_lens, dtype=np.int64)
    bt = np.asarray(block_tables, dtype=np.int64)
    Tq, Hq, d = q_bits.shape
    Hkv = k_cache.shape[2]
    out = np.zeros((Tq, Hq, d))
    q8_all, inv_all = quantize_q_rows(q_bits)
    for s in range(len(kvl)):
        q0, q1 = int(cu[s]), int(cu[s + 1])
        qlen, kv = q1 - q0, int(kvl[s])
        if qlen == 0:
            continue
        keys = np.arange(kv, dtype=np.int64)
        vis = np.zeros((qlen, kv), dtype=bool)
        for i in range(qlen):
            vis[i, visible_keys(kv, qlen, i, causal, window)] = True
        for g in range(Hkv):
            # the cache's e4m3 values, not yet scaled (the scales enter steps 2 and 4)
            K8 = gather_kv(k_cache, bt, s, keys, g, block_size, FP8, 1.0)
            V8 = gather_kv(v_cache, bt, s, keys, g, block_size, FP8, 1.0)
            for h in range(Hq):
                if kv_head_of(h, Hq, Hkv) != g:
                    continue
                out[q0:q1, h, :] = attend_fp8_blocks(
                    q8_all[q0:q1, h, :], inv_all[q0:q1, h], K8, V8, keys, vis, scale,
                    k_scale, v_scale, block_n)
    return out
