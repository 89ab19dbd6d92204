"""Unified paged-KV attention forward for GB300 (sm_103a): Python binding.

A thin ctypes layer over the C ABI in include/ua.h (libua.so, built in-tree by
build.py). The functions below carry the C names and only marshal arguments;
every step of the attention runs in the library's CUDA kernels. Importing
succeeds without the library; the first call raises if libua.so was not
built -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libua.so")

UA_OK = 0
UA_ERR_INVALID_ARG = -1
UA_ERR_UNSUPPORTED = -2
UA_ERR_CUDA = -3
UA_ERR_WORKSPACE = -4
UA_ERR_DEVICE_TIMEOUT = -5
UA_ERR_BOUNDS = -6
UA_KV_BF16 = 0
UA_KV_FP8_E4M3 = 1
UA_MAX_SPLITS = 128
UA_DECODE_ROWS = 8
UA_PREFILL_ROWS = 256

# Every symbol include/ua.h declares.
EXPORTS = (
    "ua_schedule", "ua_plan_create", "ua_plan_create_ex", "ua_forward", "ua_forward_oneshot",
    "ua_plan_get_info", "ua_last_device_error", "ua_plan_destroy", "ua_status_string",
    "ua_gather_kv_debug", "ua_plan_set_profiling", "ua_plan_kernel_times",
    "ua_forward_static_scratch", "ua_plan_set_debug", "ua_append_kv",
    "ua_plan_set_unified_max", "ua_plan_set_prefill_ctas", "ua_plan_set_fp8_products", "ua_forward_host",
)


class ua_tile(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("seq", "kv_head", "row0", "nrows", "kv_lo", "kv_hi", "slot", "group")]


class ua_combine_group(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("seq", "kv_head", "row0", "nrows", "slot0", "nsplits", "pad0", "pad1")]


class ua_plan_info(ctypes.Structure):
    _fields_ = [("num_prefill_tiles", ctypes.c_int64), ("num_decode_tiles", ctypes.c_int64),
                ("num_combine_groups", ctypes.c_int64), ("num_slots", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("split_tokens", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("num_prefill_ctas", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class UAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {ua_status_string(status)} ({status})")


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
_I32P = ctypes.POINTER(ctypes.c_int32)

_SIGS = {
    "ua_status_string": (ctypes.c_char_p, [_I32]),
    "ua_schedule": (_I32, [_I32P, _I32P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                           _I32, _I32, _I32, ctypes.POINTER(ua_plan_info),
                           ctypes.POINTER(ua_tile), _I64, ctypes.POINTER(ua_tile), _I64,
                           ctypes.POINTER(ua_combine_group), _I64]),
    "ua_plan_create": (_I32, [ctypes.POINTER(_P), _I32P, _I32P, _I32, _I32, _I32, _I32, _I32,
                              _I32, _I32, _I32, _I32, _I32, _P]),
    "ua_plan_create_ex": (_I32, [ctypes.POINTER(_P), _I32P, _I32P, _I32, _I32, _I32, _I32, _I32,
                                 _I32, _I32, _I32, _I32, _I32, _I32, _P]),
    "ua_forward": (_I32, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I32, _I32, _F, _F, _F, _P]),
    "ua_append_kv": (_I32, [_P, _P, _P, _P, _P, _P, _I64, _F, _F, _P]),
    "ua_forward_oneshot": (_I32, [_P, _P, _P, _P, _I32P, _I32P, _P, _P, _P, _I32, _I32, _I32,
                                  _I32, _I32, _I32, _I64, _I32, _I32, _I32, _F, _I32, _I32, _F,
                                  _F, _I32, _P]),
    "ua_forward_host": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32,
                               _I32, _I64, _I32, _F, _I32, _I32, _F, _F, _I32, _I32P, _P]),
    "ua_plan_get_info": (_I32, [_P, ctypes.POINTER(ua_plan_info)]),
    "ua_last_device_error": (_I32, [_P, _I32P]),
    "ua_plan_destroy": (_I32, [_P]),
    "ua_gather_kv_debug": (_I32, [_P, _P, _P, _P, _P, _I64, _P, _P, _I64, _P]),
    "ua_plan_set_profiling": (_I32, [_P, _I32]),
    "ua_plan_set_debug": (_I32, [_P, _I32, _I64]),
    "ua_plan_set_unified_max": (_I32, [_P, _I32, _F]),
    "ua_plan_set_prefill_ctas": (_I32, [_P, _I32]),
    "ua_plan_set_fp8_products": (_I32, [_P, _I32]),
    "ua_forward_static_scratch": (_I32, [_P, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32,
                                         _I32, _I32, _I64, _I32, _I32, _I32, _F, _I32, _I32, _F,
                                         _F, _I32, _P, _P]),
    "ua_plan_kernel_times": (_I32, [_P, ctypes.POINTER(ctypes.c_float),
                                    ctypes.POINTER(ctypes.c_int64)]),
}


def lib() -> ctypes.CDLL:
    """The loaded libua.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _check(status: int, where: str):
    if status != UA_OK:
        raise UAError(status, where)


def _i32_array(values):
    vals = [int(v) for v in values]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def ua_status_string(status: int) -> str:
    return lib().ua_status_string(int(status)).decode()


def ua_schedule(cu_query_lens, kv_lens, num_q_heads, num_kv_heads, head_dim, block_size,
                max_blocks_per_seq, kv_dtype=UA_KV_BF16, causal=1, window=0, num_splits=0,
                num_sms=152, decode_rows_max=-1):
    """Run the CPU scheduler alone; returns (info, prefill, decode, groups) as
    lists of dicts. Raises UAError on a rejected problem."""
    cu, kv = _i32_array(cu_query_lens), _i32_array(kv_lens)
    n = len(list(kv_lens))
    info = ua_plan_info()
    args = (cu, kv, n, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
            kv_dtype, causal, window, num_splits, num_sms, decode_rows_max)
    _check(lib().ua_schedule(*args, ctypes.byref(info), None, 0, None, 0, None, 0), "ua_schedule")
    pre = (ua_tile * max(1, info.num_prefill_tiles))()
    dec = (ua_tile * max(1, info.num_decode_tiles))()
    grp = (ua_combine_group * max(1, info.num_combine_groups))()
    _check(lib().ua_schedule(*args, ctypes.byref(info), pre, info.num_prefill_tiles, dec,
                             info.num_decode_tiles, grp, info.num_combine_groups), "ua_schedule")

    def rows(arr, n, cls):
        return [{f: getattr(arr[i], f) for f, _ in cls._fields_} for i in range(n)]
    return (info, rows(pre, info.num_prefill_tiles, ua_tile),
            rows(dec, info.num_decode_tiles, ua_tile),
            rows(grp, info.num_combine_groups, ua_combine_group))


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return int(getattr(stream, "cuda_stream", stream))


def ua_plan_create(cu_query_lens, kv_lens, num_q_heads, num_kv_heads, head_dim, block_size,
                   max_blocks_per_seq, kv_dtype=UA_KV_BF16, causal=1, window=0, num_splits=0,
                   decode_rows_max=-1, stream=None) -> int:
    """Create a plan from host lengths; returns the opaque plan handle."""
    cu, kv = _i32_array(cu_query_lens), _i32_array(kv_lens)
    n = len(list(kv_lens))
    h = ctypes.c_void_p()
    _check(lib().ua_plan_create_ex(ctypes.byref(h), cu, kv, n, num_q_heads, num_kv_heads,
                                   head_dim, block_size, max_blocks_per_seq, kv_dtype, causal,
                                   window, num_splits, decode_rows_max, _stream_handle(stream)),
           "ua_plan_create")
    return h.value


def ua_plan_get_info(plan: int) -> ua_plan_info:
    info = ua_plan_info()
    _check(lib().ua_plan_get_info(plan, ctypes.byref(info)), "ua_plan_get_info")
    return info


def ua_forward(plan, q, k_cache, v_cache, out, cu_query_lens, kv_lens, block_tables, num_blocks,
               max_q, max_kv, scale, k_scale=1.0, v_scale=1.0, stream=None):
    """Launch the forward on `stream` (default: torch's current stream).
    Tensor arguments are CUDA tensors (or raw device pointers)."""
    ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
    _check(lib().ua_forward(plan, ptr(q), ptr(k_cache), ptr(v_cache), ptr(out),
                            ptr(cu_query_lens), ptr(kv_lens), ptr(block_tables), int(num_blocks),
                            int(max_q), int(max_kv), float(scale), float(k_scale),
                            float(v_scale), _stream_handle(stream)), "ua_forward")


def ua_append_kv(plan, k_new, v_new, k_cache, v_cache, block_tables, num_blocks, k_scale=1.0,
                 v_scale=1.0, stream=None):
    """Write the step's new K/V rows into the paged cache on `stream` (positions
    from the plan's lengths). Tensor arguments are CUDA tensors (or raw device
    pointers)."""
    ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
    _check(lib().ua_append_kv(plan, ptr(k_new), ptr(v_new), ptr(k_cache), ptr(v_cache),
                              ptr(block_tables), int(num_blocks), float(k_scale),
                              float(v_scale), _stream_handle(stream)), "ua_append_kv")


def ua_forward_oneshot(q, k_cache, v_cache, out, cu_query_lens_host, kv_lens_host,
                       cu_query_lens, kv_lens, block_tables, num_q_heads, num_kv_heads,
                       head_dim, block_size, max_blocks_per_seq, num_blocks, kv_dtype, max_q,
                       max_kv, scale, causal=1, window=0, k_scale=1.0, v_scale=1.0,
                       num_splits=0, stream=None):
    ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
    n = len(list(kv_lens_host))
    _check(lib().ua_forward_oneshot(ptr(q), ptr(k_cache), ptr(v_cache), ptr(out),
                                    _i32_array(cu_query_lens_host), _i32_array(kv_lens_host),
                                    ptr(cu_query_lens), ptr(kv_lens), ptr(block_tables), n,
                                    num_q_heads, num_kv_heads, head_dim, block_size,
                                    max_blocks_per_seq, int(num_blocks), kv_dtype, int(max_q),
                                    int(max_kv), float(scale), causal, window, float(k_scale),
                                    float(v_scale), num_splits, _stream_handle(stream)),
           "ua_forward_oneshot")


def ua_forward_host(q_host, out_host, cu_query_lens_host, kv_lens_host, block_tables_host,
                    k_cache, v_cache, num_q_heads, num_kv_heads, head_dim, block_size,
                    num_blocks, kv_dtype, scale, causal=1, window=0, k_scale=1.0, v_scale=1.0,
                    num_splits=0, stream=None) -> int:
    """One step from host buffers (q/out/lengths/page tables on the host, the
    cache on the device); returns the device error word. Host tensors:
    contiguous CPU tensors (bf16 q / out, int32 lengths and page tables),
    pinned for asynchronous copies."""
    n = int(kv_lens_host.shape[0])
    err = ctypes.c_int32(0)
    _check(lib().ua_forward_host(
        q_host.data_ptr(), out_host.data_ptr(), cu_query_lens_host.data_ptr(),
        kv_lens_host.data_ptr(), block_tables_host.data_ptr(), k_cache.data_ptr(),
        v_cache.data_ptr(), n, num_q_heads, num_kv_heads, head_dim, block_size,
        int(block_tables_host.shape[1]) if n else 0, num_blocks, kv_dtype, scale, causal, window,
        k_scale, v_scale, num_splits, ctypes.byref(err), _stream_handle(stream)),
        "ua_forward_host")
    return err.value


def ua_last_device_error(plan: int) -> int:
    code = ctypes.c_int32(0)
    _check(lib().ua_last_device_error(plan, ctypes.byref(code)), "ua_last_device_error")
    return code.value


def ua_plan_destroy(plan: int):
    _check(lib().ua_plan_destroy(plan), "ua_plan_destroy")


def ua_gather_kv_debug(plan, k_cache, v_cache, kv_lens, block_tables, num_blocks, k_out, v_out,
                       rows_cap, stream=None):
    ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
    _check(lib().ua_gather_kv_debug(plan, ptr(k_cache), ptr(v_cache), ptr(kv_lens),
                                    ptr(block_tables), int(num_blocks), ptr(k_out), ptr(v_out),
                                    int(rows_cap), _stream_handle(stream)), "ua_gather_kv_debug")


def ua_plan_set_profiling(plan: int, enable: bool):
    _check(lib().ua_plan_set_profiling(plan, 1 if enable else 0), "ua_plan_set_profiling")


def ua_plan_set_debug(plan: int, flags: int, wait_timeout_ns: int = 0):
    """Test aid: flags bit 0 idles the prefill producer (bounded waits run out)."""
    _check(lib().ua_plan_set_debug(plan, int(flags), int(wait_timeout_ns)), "ua_plan_set_debug")


def ua_plan_set_prefill_ctas(plan: int, num_ctas: int = 0):
    """Prefill CTAs of later forwards on this plan (0: the scheduler's count)."""
    _check(lib().ua_plan_set_prefill_ctas(plan, int(num_ctas)), "ua_plan_set_prefill_ctas")


def ua_plan_set_fp8_products(plan: int, enable: bool = True):
    """fp8 tensor-core products for the prefill tiles of an e4m3 cache (later
    forwards on this plan); enable=False restores the staged bf16 path."""
    _check(lib().ua_plan_set_fp8_products(plan, 1 if enable else 0), "ua_plan_set_fp8_products")


def ua_plan_set_unified_max(plan: int, phi=None):
    """Unified max for decode rows (None: off): phi in units of the scaled
    score; rows whose first maximum lies outside its range fall back to the
    running maximum."""
    on = phi is not None
    _check(lib().ua_plan_set_unified_max(plan, int(on), float(phi) if on else 0.0),
           "ua_plan_set_unified_max")


KERNEL_KINDS = ("prefill", "decode", "combine", "append", "stage")


def ua_plan_kernel_times(plan: int):
    """{kind: (milliseconds, launches)} since the last read (synchronises)."""
    ms = (ctypes.c_float * len(KERNEL_KINDS))()
    n = (ctypes.c_int64 * len(KERNEL_KINDS))()
    _check(lib().ua_plan_kernel_times(plan, ms, n), "ua_plan_kernel_times")
    return {k: (ms[i], n[i]) for i, k in enumerate(KERNEL_KINDS)}


def ua_forward_static_scratch(q, k_cache, v_cache, out, cu_query_lens, kv_lens, block_tables,
                              num_q_heads, num_kv_heads, head_dim, block_size,
                              max_blocks_per_seq, num_blocks, kv_dtype, max_q, max_kv, scale,
                              causal=1, window=0, k_scale=1.0, v_scale=1.0, num_splits=0,
                              device_error=None, stream=None):
    """The forward without any device allocation (scratch in a static device
    array inside libua.so); for callers that may not allocate device memory."""
    ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
    n = int(kv_lens.numel()) if hasattr(kv_lens, "numel") else int(len(kv_lens))
    _check(lib().ua_forward_static_scratch(
        ptr(q), ptr(k_cache), ptr(v_cache), ptr(out), ptr(cu_query_lens), ptr(kv_lens),
        ptr(block_tables), n, num_q_heads, num_kv_heads, head_dim, block_size,
        max_blocks_per_seq, int(num_blocks), kv_dtype, int(max_q), int(max_kv), float(scale),
        causal, window, float(k_scale), float(v_scale), num_splits,
        None if device_error is None else ptr(device_error), _stream_handle(stream)),
        "ua_forward_static_scratch")


class Plan:
    """RAII wrapper around a plan handle."""

    def __init__(self, *args, **kwargs):
        self.handle = ua_plan_create(*args, **kwargs)

    @property
    def info(self) -> ua_plan_info:
        return ua_plan_get_info(self.handle)

    def forward(self, *args, **kwargs):
        ua_forward(self.handle, *args, **kwargs)

    def append_kv(self, *args, **kwargs):
        ua_append_kv(self.handle, *args, **kwargs)

    def last_device_error(self) -> int:
        return ua_last_device_error(self.handle)

    def set_unified_max(self, phi=None):
        ua_plan_set_unified_max(self.handle, phi)

    def close(self):
        if self.handle:
            ua_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
