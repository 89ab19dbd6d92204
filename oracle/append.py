"""Reference for appending a step's new K/V to the paged cache (test
infrastructure only; see the package docstring).

What it computes ("flashatten takeaways EP2 工程", the split-KV launcher's
Append_KV path: the new keys and values are written into the cache at each
sequence's offset before attention reads it; the paged layout and the
"quantization" path of "vllm_triton_unified_attention_notes", test section):

  for sequence s, new token i < qlen_s (its rows are q's rows cu[s] + i):
    pos = (kv_len_s - qlen_s) + i            kv_len counts the new tokens
    blk = block_tables[s, pos // bs], slot = pos % bs
    K[blk, slot, :, :] = k_new[cu[s] + i, :, :]   (V likewise)
  bf16 cache: the bf16 words are copied.
  fp8 cache:  code = e4m3(k_new / k_scale), the quotient taken in binary32
              (round to nearest), then rounded to e4m3 to nearest, ties to
              even, saturating at +-448; NaN stays NaN.

Readings (the pages name the path, not its arithmetic): the division and its
binary32 precision are the plainest form of "x / scale" with a per-tensor
scale; saturation (instead of an overflow to NaN) keeps a cache entry finite
whatever the scale; both sides take the rounding decision on the same
binary32 quotient, so codes are compared bit for bit.
"""
from __future__ import annotations

import numpy as np

from .attention import decode_bf16

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def encode_e4m3(x: np.ndarray) -> np.ndarray:
    """binary32/binary64 values -> OCP E4M3 codes, round to nearest even,
    saturating to +-448 (infinities too); NaN -> 0x7F.

    From the format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
    exponent field 0 holds the subnormals m/8 * 2^-6 (steps of 2^-9); normal
    values are (1 + m/8) * 2^(e-7); the field pair e = 15, m = 7 is NaN, so
    1.75 * 2^8 = 448 is the largest finite value. A value is rounded on the
    grid of its binade: steps of 2^-9 below 2^-6, steps of 2^(E-3) in
    [2^E, 2^(E+1)).
    """
    v = np.asarray(x, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint8)
    flat_v = v.reshape(-1)
    flat_o = out.reshape(-1)
    for n in range(flat_v.size):
        flat_o[n] = _encode_one(float(flat_v[n]))
    return out


def _encode_one(x: float) -> int:
    if np.isnan(x):
        return E4M3_NAN
    sign = 0x80 if np.signbit(x) else 0x00
    a = abs(x)
    if np.isinf(a):
        return sign | 0x7E           # saturate at 448
    if a >= 2.0 ** -6:
        _, exp2 = np.frexp(a)        # a = f * 2^exp2 with f in [0.5, 1)
        e = int(exp2) - 1            # binade: 2^e <= a < 2^(e+1)
        q = float(np.rint(a / 2.0 ** (e - 3)))   # 8 <= q <= 16, ties to even
        if q == 16.0:
            e, q = e + 1, 8.0
        field = e + 7
        if field > 15 or (field == 15 and q - 8 > 6):
            return sign | 0x7E       # saturate at 448
        return sign | (field << 3) | int(q - 8)
    m = int(np.rint(a / 2.0 ** -9))  # subnormal steps; m = 8 is the first normal
    return sign | m


def quantize_e4m3(bits_bf16: np.ndarray, scale: float) -> np.ndarray:
    """bf16 words -> e4m3 codes of value / scale, the quotient in binary32."""
    x = decode_bf16(bits_bf16).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        qt = (x / np.float32(scale)).astype(np.float32)
    return encode_e4m3(qt)


def append_kv(k_new: np.ndarray, v_new: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
              cu_query_lens, kv_lens, block_tables: np.ndarray, block_size: int,
              kv_dtype: str = "bf16", k_scale: float = 1.0, v_scale: float = 1.0):
    """Copies of k_cache / v_cache with every new token written at its slot.

    k_new, v_new: bf16 words [total_tokens, Hkv, d] (uint16).
    k_cache, v_cache: [num_blocks, block_size, Hkv, d], bf16 words (uint16) or
    e4m3 codes (uint8).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    cu = [int(c) for c in cu_query_lens]
    for s in range(len(cu) - 1):
        ql = cu[s + 1] - cu[s]
        ctx = int(kv_lens[s]) - ql
        for i in range(ql):
            pos = ctx + i
            blk = int(block_tables[s, pos // block_size])
            slot = pos % block_size
            row = cu[s] + i
            if kv_dtype == "bf16":
                kc[blk, slot] = k_new[row]
                vc[blk, slot] = v_new[row]
            else:
                kc[blk, slot] = quantize_e4m3(k_new[row], k_scale)
                vc[blk, slot] = quantize_e4m3(v_new[row], v_scale)
    return kc, vc
