"""Plain fp64 CPU oracle for unified paged-KV attention (test infrastructure).

This package is test infrastructure only. The tests, the smoke check and the
benchmark's CPU-baseline leg use it to produce expected values; the product
library never imports, links or runs it, and it shares no code with the CUDA
path. It is written for a reader checking it against the pages by eye: no
tiling, no online softmax, no exp2 -- the textbook definition.

Definition (softmax(q K^T / sqrt(d)) V over the visible prefix), from
"flashatten takeaways EP2 工程" (kv cache section, the boxed O_{t+1} equation),
with the paged layout, GQA grouping and context length of
"vllm_triton_unified_attention_notes" (unified_attention and
kernel_unified_attention_2d sections):

  for sequence s, query i < qlen_s, query head h:
    g   = h // (Hq // Hkv)                      contiguous GQA groups
    pos = (kv_len_s - qlen_s) + i               context_len + i, bottom-right causal
    visible t: 0 <= t < kv_len_s, (not causal or t <= pos),
               (window <= 0 or t > pos - window)
    k_t = K[bt[s, t // bs], t % bs, g, :] * k_scale     (k_scale only for fp8)
    x_t = scale * <q[cu[s] + i, h, :], k_t>
    out = sum_t exp(x_t - max x) v_t / sum_t exp(x_t - max x)
    lse = max x + log sum_t exp(x_t - max x)            (natural log)

Inputs are raw bit patterns (bf16 words as uint16, e4m3 codes as uint8) and
are widened to fp64 exactly from their format definitions.

The append step (writing a step's new K/V into the paged cache, with the
e4m3 quantisation of the fp8 cache) is in oracle/append.py.

The fp8-products variant (fp8 Q.K^T and fp8 P, the FP8 path of the "Fused
Attention" notes) is in oracle/fp8_products.py. There the key blocks and the
running max are part of what the method computes -- P is rounded to e4m3
relative to the running max of its block -- so that oracle follows the
blockwise recurrence, still in binary64.

Parity pins live in tests/test_oracle_pins.py, tests/test_append_pins.py and
tests/test_fp8_products_pins.py; every function is pinned there (none is
"parity unpinned").
"""
from .attention import (  # noqa: F401
    decode_bf16,
    decode_e4m3,
    kv_head_of,
    visible_keys,
    gather_kv,
    attend,
    paged_attention,
    paged_attention_rows,
    partial_attention,
    combine_partials,
)
from .append import encode_e4m3, quantize_e4m3, append_kv  # noqa: F401
from .fp8_products import (  # noqa: F401
    round_e4m3,
    quantize_q_rows,
    attend_fp8_blocks,
    paged_attention_fp8_products,
)
