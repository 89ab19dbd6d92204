"""Shared helpers for the GPU parity tests (CUDA path vs the fp64 oracle)."""
import numpy as np
import torch

import oracle
import workloads as W

# Tolerances on the bf16 output against the fp64 oracle.
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
FP8_MAX_ABS = 6e-2


def oracle_full(case):
    r = case.raw()
    out, _ = oracle.paged_attention(r["q"], r["k_cache"], r["v_cache"], r["cu_query_lens"],
                                    r["kv_lens"], r["block_tables"], case.block_size, case.scale,
                                    kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                                    v_scale=case.v_scale, causal=case.causal, window=case.window)
    return out


def oracle_rows(case, rows):
    r = case.raw()
    out, _ = oracle.paged_attention_rows(r["q"], r["k_cache"], r["v_cache"], r["cu_query_lens"],
                                         r["kv_lens"], r["block_tables"], case.block_size,
                                         case.scale, rows, kv_dtype=case.kv_dtype,
                                         k_scale=case.k_scale, v_scale=case.v_scale,
                                         causal=case.causal, window=case.window)
    return out


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).cpu().numpy()


def assert_close(got: np.ndarray, exp: np.ndarray, kv_dtype: str, what: str = ""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - exp)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if kv_dtype == W.FP8:
        assert mx <= FP8_MAX_ABS, f"{what}: max-abs {mx:.3e} > {FP8_MAX_ABS}"
    else:
        assert mx <= BF16_MAX_ABS, f"{what}: max-abs {mx:.3e} > {BF16_MAX_ABS}"
        assert mean <= BF16_MEAN_ABS, f"{what}: mean-abs {mean:.3e} > {BF16_MEAN_ABS}"
    return mx, mean


def sample_rows(case, n, seed=0):
    """n (token, head) rows spread over every sequence, including first and last tokens."""
    rng = np.random.default_rng(seed)
    cu = case.cu_query_lens.tolist()
    rows = []
    B = case.num_seqs
    for k in range(n):
        s = k % B if k < 2 * B else int(rng.integers(B))
        ql = cu[s + 1] - cu[s]
        if ql == 0:
            continue
        i = [0, ql - 1][k % 2] if k < 2 * B else int(rng.integers(ql))
        rows.append((cu[s] + i, int(rng.integers(case.num_q_heads))))
    return rows
