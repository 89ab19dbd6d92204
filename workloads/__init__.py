"""Seeded synthetic inputs for unified paged-KV attention.

This module only draws random numbers and lays them out in the paged-cache
format; it holds none of the attention arithmetic. Both the CUDA path (through
its Python binding) and the CPU oracle consume what it returns, so the two see
identical bytes.

Layouts follow "vllm_triton_unified_attention_notes" (the test section):
  q            [total_q_tokens, num_q_heads, head_dim]              bf16
  k_cache/v    [num_blocks, block_size, num_kv_heads, head_dim]     bf16 or fp8 e4m3
  cu_query_lens[num_seqs + 1] int32, leading 0, prefix sums of query lengths
  kv_lens      [num_seqs] int32, kv_len counts the new query tokens too
  block_tables [num_seqs, max_blocks_per_seq] int32 physical block ids

Draw order with one torch CPU generator: lengths, block permutation, Q, K, V.
fp8 caches are drawn N(0,1) in fp32, scaled per tensor by amax/448 and
rounded with torch's float8_e4m3fn conversion (input preparation, not part of
the attention path).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

BF16 = "bf16"
FP8 = "fp8_e4m3"
E4M3_MAX = 448.0


@dataclasses.dataclass
class Case:
    name: str
    q: torch.Tensor              # bf16 [Tq, Hq, d]
    k_cache: torch.Tensor        # bf16 or float8_e4m3fn [NB, bs, Hkv, d]
    v_cache: torch.Tensor
    cu_query_lens: torch.Tensor  # int32 [B+1]
    kv_lens: torch.Tensor        # int32 [B]
    block_tables: torch.Tensor   # int32 [B, max_blocks]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str
    scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    causal: bool = True
    window: int = 0

    @property
    def num_seqs(self) -> int:
        return int(self.kv_lens.numel())

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def query_lens(self) -> List[int]:
        cu = self.cu_query_lens.tolist()
        return [cu[i + 1] - cu[i] for i in range(len(cu) - 1)]

    @property
    def max_q(self) -> int:
        return max(self.query_lens) if self.num_seqs else 0

    @property
    def max_kv(self) -> int:
        return int(self.kv_lens.max()) if self.num_seqs else 0

    def raw(self):
        """Raw bit patterns as numpy arrays (uint16 bf16 words, uint8 e4m3 codes)."""
        q = self.q.contiguous().view(torch.int16).numpy().view(np.uint16)
        if self.kv_dtype == BF16:
            k = self.k_cache.contiguous().view(torch.int16).numpy().view(np.uint16)
            v = self.v_cache.contiguous().view(torch.int16).numpy().view(np.uint16)
        else:
            k = self.k_cache.contiguous().view(torch.uint8).numpy()
            v = self.v_cache.contiguous().view(torch.uint8).numpy()
        return dict(q=q, k_cache=k, v_cache=v,
                    cu_query_lens=self.cu_query_lens.numpy().astype(np.int64),
                    kv_lens=self.kv_lens.numpy().astype(np.int64),
                    block_tables=self.block_tables.numpy().astype(np.int64))


def _normal(gen: torch.Generator, shape, std: float = 1.0) -> torch.Tensor:
    return torch.randn(*shape, generator=gen, dtype=torch.float32) * std


def _fill_cache(gen, shape, kv_dtype, std, chunk_blocks=4096):
    """Draw a cache block-chunk by block-chunk (bounded host memory).

    For fp8 the per-tensor scale needs the whole tensor's amax, so the
    generator state is saved, the tensor is drawn once for amax, then the
    state is restored and the tensor drawn again for quantisation.
    """
    nb = shape[0]
    if kv_dtype == BF16:
        out = torch.empty(shape, dtype=torch.bfloat16)
        for b0 in range(0, nb, chunk_blocks):
            b1 = min(nb, b0 + chunk_blocks)
            out[b0:b1] = _normal(gen, (b1 - b0,) + tuple(shape[1:]), std).to(torch.bfloat16)
        return out, 1.0
    state = gen.get_state()
    amax = 0.0
    for b0 in range(0, nb, chunk_blocks):
        b1 = min(nb, b0 + chunk_blocks)
        amax = max(amax, float(_normal(gen, (b1 - b0,) + tuple(shape[1:]), std).abs().max()))
    gen.set_state(state)
    s = amax / E4M3_MAX if amax > 0 else 1.0
    out = torch.empty(shape, dtype=torch.float8_e4m3fn)
    for b0 in range(0, nb, chunk_blocks):
        b1 = min(nb, b0 + chunk_blocks)
        x = _normal(gen, (b1 - b0,) + tuple(shape[1:]), std)
        out[b0:b1] = (x / s).to(torch.float8_e4m3fn)
    return out, s


def make_case(name: str,
              query_lens: Sequence[int],
              kv_lens: Sequence[int],
              num_q_heads: int,
              num_kv_heads: int,
              head_dim: int,
              block_size: int,
              kv_dtype: str = BF16,
              num_blocks: Optional[int] = None,
              table: str = "random",
              seed: int = 0,
              gen: Optional[torch.Generator] = None,
              scale: Optional[float] = None,
              causal: bool = True,
              window: int = 0,
              std: float = 1.0,
              poison: bool = False,
              extra_table_cols: int = 0) -> Case:
    """Build one seeded case.

    table: "random" deals a random permutation of physical block ids to the
    sequences in order (distinct ids); "identity" gives sequence s the ids
    s*max_blocks .. s*max_blocks+n-1.
    poison: unused blocks, tail slots past kv_len in each sequence's last block
    and block-table padding entries all hold NaN (bf16 NaN or e4m3 0x7F).
    """
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    qlens = [int(x) for x in query_lens]
    kvls = [int(x) for x in kv_lens]
    B = len(qlens)
    need = [-(-kv // block_size) for kv in kvls]
    max_blocks = max(need) if B else 1
    max_blocks = max(max_blocks, 1) + extra_table_cols
    total_need = sum(need)
    if num_blocks is None:
        num_blocks = total_need + (1 if poison else 0)
        if table == "identity":
            num_blocks = max(num_blocks, B * max_blocks)
    if table == "identity":
        assert num_blocks >= B * max_blocks
    assert num_blocks >= total_need + (1 if poison else 0)

    # block ids: a random permutation of [0, num_blocks), dealt in order
    perm = torch.randperm(num_blocks, generator=gen)
    bt = torch.zeros((B, max_blocks), dtype=torch.int32)
    used = torch.zeros(num_blocks, dtype=torch.bool)
    pos = 0
    for s in range(B):
        for j in range(need[s]):
            if table == "identity":
                bid = s * max_blocks + j
            else:
                bid = int(perm[pos])
                pos += 1
            bt[s, j] = bid
            used[bid] = True
    unused = torch.nonzero(~used).flatten()
    pad_id = int(unused[0]) if (poison and unused.numel()) else 0
    for s in range(B):
        bt[s, need[s]:] = pad_id

    Tq = sum(qlens)
    q = _normal(gen, (Tq, num_q_heads, head_dim), std).to(torch.bfloat16)
    shape = (num_blocks, block_size, num_kv_heads, head_dim)
    k_cache, k_scale = _fill_cache(gen, shape, kv_dtype, std)
    v_cache, v_scale = _fill_cache(gen, shape, kv_dtype, std)
    if poison:
        _poison(k_cache, v_cache, used, bt, kvls, block_size, kv_dtype)
    cu = torch.zeros(B + 1, dtype=torch.int32)
    if B:
        cu[1:] = torch.cumsum(torch.tensor(qlens, dtype=torch.int64), 0).to(torch.int32)
    return Case(name=name, q=q, k_cache=k_cache, v_cache=v_cache,
                cu_query_lens=cu, kv_lens=torch.tensor(kvls, dtype=torch.int32),
                block_tables=bt, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, block_size=block_size, kv_dtype=kv_dtype,
                scale=(1.0 / math.sqrt(head_dim)) if scale is None else float(scale),
                k_scale=float(k_scale), v_scale=float(v_scale), causal=causal, window=window)


def _poison(k_cache, v_cache, used, bt, kvls, bs, kv_dtype):
    if kv_dtype == BF16:
        def put(t, idx):
            t[idx] = float("nan")
    else:
        def put(t, idx):
            t.view(torch.uint8)[idx] = 0x7F
    for t in (k_cache, v_cache):
        put(t, ~used)
        for s, kv in enumerate(kvls):
            if kv % bs:
                last = int(bt[s, (kv - 1) // bs])
                put(t, (last, slice(kv % bs, None)))


# --------------------------------------------------------------------------
# The five synthetic workloads (sizes from the benchmark description).
# --------------------------------------------------------------------------

def config1_tiny_mixed(seed: int = 0, poison: bool = False) -> Case:
    """3 sequences, query_lens [1,5,17], kv_lens [40,130,300], 4/4 heads,
    d 64, block_size 16, 256 physical blocks, ids drawn without replacement."""
    return make_case("tiny_mixed_b3_h4_d64", [1, 5, 17], [40, 130, 300], 4, 4, 64, 16,
                     num_blocks=256, seed=seed, scale=1.0 / 8.0, poison=poison)


def config2_pure_decode(seed: int = 0, poison: bool = False) -> Case:
    """64 decode sequences, kv_len ~ U[512, 4096], 32 q / 8 kv heads, d 128, bf16."""
    gen = torch.Generator().manual_seed(seed)
    kv = torch.randint(512, 4097, (64,), generator=gen).tolist()
    return make_case("pure_decode_b64_kv512-4096_h32-8_d128_bf16", [1] * 64, kv, 32, 8, 128, 16,
                     gen=gen, poison=poison)


def config3_mixed(seed: int = 0, poison: bool = False) -> Case:
    """8 prefill sequences (query_len U[512,2048], prior context U[0,1024]) then
    120 decode sequences (kv_len U[1024,8192]); 32/8 heads, d 128, bf16, causal."""
    gen = torch.Generator().manual_seed(seed)
    pq = torch.randint(512, 2049, (8,), generator=gen).tolist()
    pc = torch.randint(0, 1025, (8,), generator=gen).tolist()
    dk = torch.randint(1024, 8193, (120,), generator=gen).tolist()
    qlens = pq + [1] * 120
    kvls = [c + q for c, q in zip(pc, pq)] + dk
    return make_case("mixed_8prefill_120decode_h32-8_d128_bf16", qlens, kvls, 32, 8, 128, 16,
                     gen=gen, poison=poison)


def config4_dense_prefill(seed: int = 0, poison: bool = False) -> Case:
    """Batch 4, 32 heads (MHA), q = kv = 4096, d 128, block_size 128, identity table."""
    return make_case("dense_causal_prefill_b4_h32_l4096_d128", [4096] * 4, [4096] * 4, 32, 32, 128,
                     128, table="identity", seed=seed, poison=poison)


def config5_long_fp8_decode(seed: int = 0, poison: bool = False) -> Case:
    """8 decode sequences at kv_len 131072, 64 q / 8 kv heads, d 128, fp8 e4m3 KV."""
    return make_case("long_decode_fp8_b8_kv131072_h64-8_d128", [1] * 8, [131072] * 8, 64, 8, 128, 16,
                     kv_dtype=FP8, seed=seed, poison=poison)


def config6_dense_prefill_fp8(seed: int = 0, poison: bool = False) -> Case:
    """Config 4's prefill over a paged fp8 e4m3 cache: batch 4, 32 heads (MHA),
    q = kv = 4096, d 128, block_size 16, random table (not one of the five
    benchmark configurations: it measures the fp8 prefill path)."""
    return make_case("dense_causal_prefill_fp8_b4_h32_l4096_d128_bs16", [4096] * 4, [4096] * 4,
                     32, 32, 128, 16, kv_dtype=FP8, seed=seed, poison=poison)


def config7_uniform_decode(seed: int = 0, poison: bool = False) -> Case:
    """32 decode sequences of exactly 8192 keys, 32 q / 8 kv heads, d 128,
    bf16 (not one of the five benchmark configurations: it measures how the
    automatic split sizing handles a batch of equal lengths)."""
    return make_case("uniform_decode_b32_kv8192_h32-8_d128_bf16", [1] * 32, [8192] * 32, 32, 8,
                     128, 16, seed=seed, poison=poison)


def config8_pure_decode_d256(seed: int = 0, poison: bool = False) -> Case:
    """Config 2's batch at head_dim 256: 64 decode sequences, kv_len ~
    U[512, 4096], 32 q / 8 kv heads, bf16 (not one of the five benchmark
    configurations: it measures the head_dim 256 decode path)."""
    gen = torch.Generator().manual_seed(seed)
    kv = torch.randint(512, 4097, (64,), generator=gen).tolist()
    return make_case("pure_decode_b64_kv512-4096_h32-8_d256_bf16", [1] * 64, kv, 32, 8, 256, 16,
                     gen=gen, poison=poison)


def config9_dense_prefill_d256(seed: int = 0, poison: bool = False) -> Case:
    """Config 4's dense causal prefill at head_dim 256: batch 4, 32 heads
    (MHA), q = kv = 4096, bf16, block_size 128, identity table (not one of the
    five benchmark configurations: it measures the head_dim 256 prefill
    kernel)."""
    return make_case("dense_causal_prefill_b4_h32_l4096_d256", [4096] * 4, [4096] * 4, 32, 32,
                     256, 128, table="identity", seed=seed, poison=poison)


def config10_pure_decode_d96(seed: int = 0, poison: bool = False) -> Case:
    """Config 2's batch at head_dim 96 (rows of 192 bytes: not whole 128-byte
    panels): 64 decode sequences, kv_len ~ U[512, 4096], 32 q / 8 kv heads,
    bf16 (not one of the five benchmark configurations: it measures the
    decode kernel at a head dim that is not a power of two)."""
    gen = torch.Generator().manual_seed(seed)
    kv = torch.randint(512, 4097, (64,), generator=gen).tolist()
    return make_case("pure_decode_b64_kv512-4096_h32-8_d96_bf16", [1] * 64, kv, 32, 8, 96, 16,
                     gen=gen, poison=poison)


def config11_dense_prefill_d192(seed: int = 0, poison: bool = False) -> Case:
    """Config 4's dense causal prefill at head_dim 192: batch 4, 32 heads
    (MHA), q = kv = 4096, bf16, block_size 128, identity table (not one of the
    five benchmark configurations: it measures the wide prefill kernel at
    head_dim 192)."""
    return make_case("dense_causal_prefill_b4_h32_l4096_d192", [4096] * 4, [4096] * 4, 32, 32,
                     192, 128, table="identity", seed=seed, poison=poison)


CONFIGS = {
    1: config1_tiny_mixed,
    2: config2_pure_decode,
    3: config3_mixed,
    4: config4_dense_prefill,
    5: config5_long_fp8_decode,
    6: config6_dense_prefill_fp8,
    7: config7_uniform_decode,
    8: config8_pure_decode_d256,
    9: config9_dense_prefill_d256,
    10: config10_pure_decode_d96,
    11: config11_dense_prefill_d192,
}


def random_small_case(seed: int, kv_dtype: str = BF16, head_dim: int = 128,
                      num_q_heads: int = 8, num_kv_heads: int = 2, block_size: int = 16,
                      max_seqs: int = 6, max_kv: int = 700, causal: bool = True,
                      window: int = 0, poison: bool = False) -> Case:
    """A ragged mix of decode, short and long prefill sequences, sized so the
    oracle finishes in well under a second."""
    gen = torch.Generator().manual_seed(1000 + seed)
    B = int(torch.randint(1, max_seqs + 1, (1,), generator=gen))
    qlens, kvls = [], []
    for _ in range(B):
        kind = int(torch.randint(0, 4, (1,), generator=gen))
        kv = int(torch.randint(1, max_kv + 1, (1,), generator=gen))
        if kind == 0:
            q = 1
        elif kind == 1:
            q = int(torch.randint(1, min(kv, 9) + 1, (1,), generator=gen))
        elif kind == 2:
            q = int(torch.randint(1, kv + 1, (1,), generator=gen))
        else:
            q = kv
        qlens.append(q)
        kvls.append(kv)
    return make_case(f"random_small_{seed}", qlens, kvls, num_q_heads, num_kv_heads, head_dim,
                     block_size, kv_dtype=kv_dtype, gen=gen, causal=causal, window=window,
                     poison=poison)
