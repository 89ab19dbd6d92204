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


def oracle_full_parallel(case):
    """The whole-batch oracle output, computed (sequence, KV head) unit by unit
    on every host core (oracle.pool): for the full-size workloads."""
    from oracle import pool
    r = case.raw()
    out, _ = pool.paged_attention_parallel(r, case.block_size, case.scale,
                                           kv_dtype=case.kv_dtype, k_scale=case.k_scale,
                                           v_scale=case.v_scale, causal=case.causal,
                                           window=case.window)
    return out


def as_f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).cpu().numpy()


# (what, elements compared, max-abs, mean-abs) of every comparison flagged
# for the report; tests/conftest.py prints them at the end of the run.
PARITY_REPORT = []


def assert_close(got: np.ndarray, exp: np.ndarray, kv_dtype: str, what: str = "",
                 report: bool = False):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert got.shape == exp.shape, f"{what}: shape {got.shape} vs {exp.shape}"
    err = np.abs(got - exp)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    if report:
        PARITY_REPORT.append((what, int(err.size), mx, mean))
    if kv_dtype == W.FP8:
        assert mx <= FP8_MAX_ABS, f"{what}: max-abs {mx:.3e} > {FP8_MAX_ABS}"
    else:
        assert mx <= BF16_MAX_ABS, f"{what}: max-abs {mx:.3e} > {BF16_MAX_ABS}"
        assert mean <= BF16_MEAN_ABS, f"{what}: mean-abs {mean:.3e} > {BF16_MEAN_ABS}"
    return mx, mean


def oracle_fp8_products(case):
    """The fp8-products oracle (e4m3 Q rows, e4m3 P) of an fp8-cache case."""
    from oracle import fp8_products as F
    r = case.raw()
    return F.paged_attention_fp8_products(r["q"], r["k_cache"], r["v_cache"], r["cu_query_lens"],
                                          r["kv_lens"], r["block_tables"], case.block_size,
                                          case.scale, k_scale=case.k_scale, v_scale=case.v_scale,
                                          causal=case.causal, window=case.window)
