"""PyTorch conveniences around the C ABI: device copies and one-call runs.

PyTorch only provides device memory and streams here; the attention itself
runs in libua.so's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch

from . import (UA_KV_BF16, UA_KV_FP8_E4M3, Plan, ua_append_kv, ua_forward)


@dataclasses.dataclass
class DeviceBatch:
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    cu_query_lens: torch.Tensor
    kv_lens: torch.Tensor
    block_tables: torch.Tensor
    cu_host: Sequence[int]
    kv_host: Sequence[int]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: int
    scale: float
    k_scale: float
    v_scale: float
    causal: int
    window: int

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_q(self) -> int:
        return max([b - a for a, b in zip(self.cu_host[:-1], self.cu_host[1:])] or [0])

    @property
    def max_kv(self) -> int:
        return max(list(self.kv_host) or [0])

    def new_out(self) -> torch.Tensor:
        return torch.empty(self.q.shape, dtype=torch.bfloat16, device=self.q.device)


def to_device(case, device="cuda") -> DeviceBatch:
    """Copy a host case (an object with the workloads.Case fields) to `device`.
    fp8 caches travel as raw e4m3 bytes."""
    kv_dtype = UA_KV_FP8_E4M3 if case.kv_dtype == "fp8_e4m3" else UA_KV_BF16
    k = case.k_cache.view(torch.uint8) if kv_dtype == UA_KV_FP8_E4M3 else case.k_cache
    v = case.v_cache.view(torch.uint8) if kv_dtype == UA_KV_FP8_E4M3 else case.v_cache
    return DeviceBatch(
        q=case.q.to(device).contiguous(), k_cache=k.to(device).contiguous(),
        v_cache=v.to(device).contiguous(),
        cu_query_lens=case.cu_query_lens.to(device=device, dtype=torch.int32).contiguous(),
        kv_lens=case.kv_lens.to(device=device, dtype=torch.int32).contiguous(),
        block_tables=case.block_tables.to(device=device, dtype=torch.int32).contiguous(),
        cu_host=case.cu_query_lens.tolist(), kv_host=case.kv_lens.tolist(),
        num_q_heads=case.num_q_heads, num_kv_heads=case.num_kv_heads, head_dim=case.head_dim,
        block_size=case.block_size, kv_dtype=kv_dtype, scale=case.scale, k_scale=case.k_scale,
        v_scale=case.v_scale, causal=int(case.causal), window=int(case.window))


def make_plan(b: DeviceBatch, num_splits: int = 0, decode_rows_max: int = -1,
              stream=None) -> Plan:
    return Plan(b.cu_host, b.kv_host, b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size,
                int(b.block_tables.shape[1]), kv_dtype=b.kv_dtype, causal=b.causal,
                window=b.window, num_splits=num_splits, decode_rows_max=decode_rows_max,
                stream=stream)


def forward(plan: Plan, b: DeviceBatch, out: Optional[torch.Tensor] = None,
            stream=None) -> torch.Tensor:
    if out is None:
        out = b.new_out()
    ua_forward(plan.handle, b.q, b.k_cache, b.v_cache, out, b.cu_query_lens, b.kv_lens,
               b.block_tables, b.num_blocks, b.max_q, b.max_kv, b.scale, b.k_scale, b.v_scale,
               stream=stream)
    return out


def append_kv(plan: Plan, b: DeviceBatch, k_new: torch.Tensor, v_new: torch.Tensor,
              stream=None) -> None:
    """Write new K/V rows [total_q, Hkv, d] (bf16, device) into b's caches."""
    ua_append_kv(plan.handle, k_new, v_new, b.k_cache, b.v_cache, b.block_tables, b.num_blocks,
                 b.k_scale, b.v_scale, stream)


def run(case, num_splits: int = 0, decode_rows_max: int = -1, device="cuda") -> torch.Tensor:
    """One forward of a host case on `device`; returns the bf16 output on the host."""
    b = to_device(case, device)
    with make_plan(b, num_splits, decode_rows_max) as plan:
        out = forward(plan, b)
        torch.cuda.synchronize()
        err = plan.last_device_error()
    if err != 0:
        raise RuntimeError(f"device error word {err}")
    return out.cpu()
