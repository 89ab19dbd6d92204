"""Run the fp64 oracle over a large batch on every host core (test infrastructure).

Test infrastructure only, like the rest of this package: the tests and the
benchmark's CPU-baseline leg use it; the product library never does.

Nothing here computes attention. The definition (softmax(scale * q K^T) V over
the visible keys of KV head h // (Hq/Hkv), "vllm_triton_unified_attention_notes",
unified_attention and kernel_unified_attention_2d sections) is independent for
every (sequence, query head), and the query heads of one KV head read only that
head's keys and values. So the batch is cut into units of one sequence and one
KV head, and each unit is one call of `paged_attention` on that restriction of
the inputs: the unit's query rows, the cache's one KV head, the sequence's page
table row. The calls run in spawned worker processes (one thread each) that map
the inputs read-only from .npy files; their outputs land in a shared result
file. The result is the whole-batch `paged_attention` output, computed unit by
unit.
"""
from __future__ import annotations

import os
import shutil
import tempfile
import time
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS",
                "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS")
_ARRAYS = ("q", "k_cache", "v_cache", "cu_query_lens", "kv_lens", "block_tables")


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux
        return os.cpu_count() or 1


def units_of(cu_query_lens, num_kv_heads: int) -> List[Tuple[int, int]]:
    """(sequence, KV head) pairs of every sequence with at least one query."""
    cu = np.asarray(cu_query_lens, dtype=np.int64)
    return [(s, g) for s in range(len(cu) - 1) if cu[s + 1] > cu[s]
            for g in range(num_kv_heads)]


def _scratch_dir(need_bytes: int) -> str:
    """A directory for the shared input/output files: /dev/shm when it has room."""
    for base in ("/dev/shm", tempfile.gettempdir()):
        try:
            if os.path.isdir(base) and shutil.disk_usage(base).free > 1.25 * need_bytes + (1 << 28):
                return tempfile.mkdtemp(prefix="ua_oracle_", dir=base)
        except OSError:
            continue
    return tempfile.mkdtemp(prefix="ua_oracle_")


def _unit(arr: Dict[str, np.ndarray], params: dict, s: int, g: int):
    """paged_attention restricted to sequence s and KV head g.

    Returns (out [q_len, qpk, d], lse [q_len, qpk])."""
    from .attention import paged_attention
    cu = arr["cu_query_lens"]
    q0, q1 = int(cu[s]), int(cu[s + 1])
    qpk = params["qpk"]
    return paged_attention(
        arr["q"][q0:q1, g * qpk:(g + 1) * qpk, :], arr["k_cache"][:, :, g:g + 1, :],
        arr["v_cache"][:, :, g:g + 1, :], [0, q1 - q0], arr["kv_lens"][s:s + 1],
        arr["block_tables"][s:s + 1], params["block_size"], params["scale"],
        kv_dtype=params["kv_dtype"], k_scale=params["k_scale"], v_scale=params["v_scale"],
        causal=params["causal"], window=params["window"])


def _worker(dirpath, params, units, mode, budget_s, rounds, counter, barrier, results):
    """Spawned process: claim units from the shared counter and run them.

    mode "parity": every unit once, outputs written into the shared files.
    mode "timing": `rounds` windows, each starting at a common barrier; in each
    the worker takes units in a cycle until budget_s of wall time has passed
    since the window opened. Reports, per window, the claimed units and the
    (start, end) times."""
    try:
        arr = {n: np.load(os.path.join(dirpath, n + ".npy"), mmap_mode="r") for n in _ARRAYS}
        out = lse = None
        if mode == "parity":
            out = np.lib.format.open_memmap(os.path.join(dirpath, "out.npy"), mode="r+")
            lse = np.lib.format.open_memmap(os.path.join(dirpath, "lse.npy"), mode="r+")
            rounds = 1
        cu = arr["cu_query_lens"]
        qpk = params["qpk"]
        report = []
        for _ in range(rounds):
            done: List[int] = []
            barrier.wait(timeout=600)
            t0 = time.monotonic()
            while True:
                with counter.get_lock():
                    k = counter.value
                    counter.value += 1
                if mode == "parity":
                    if k >= len(units):
                        break
                elif time.monotonic() - t0 >= budget_s:
                    break
                s, g = units[k % len(units)]
                o, l = _unit(arr, params, s, g)
                if mode == "parity":
                    out[cu[s]:cu[s + 1], g * qpk:(g + 1) * qpk, :] = o
                    lse[cu[s]:cu[s + 1], g * qpk:(g + 1) * qpk] = l
                done.append(k % len(units))
            report.append((done, t0, time.monotonic()))
        if out is not None:
            out.flush()
            lse.flush()
        results.put(("ok", report))
    except BaseException as e:  # reported to the parent, which raises
        barrier.abort()            # the other workers stop waiting at once
        results.put(("error", repr(e)))


def _run(raw: dict, params: dict, mode: str, workers: Optional[int], budget_s: float,
         units: Optional[Sequence[Tuple[int, int]]] = None, rounds: int = 1):
    import multiprocessing as mp
    q = np.asarray(raw["q"])
    Tq, Hq, d = q.shape
    Hkv = int(np.asarray(raw["k_cache"]).shape[2])
    params = dict(params, qpk=Hq // Hkv)
    units = list(units) if units is not None else units_of(raw["cu_query_lens"], Hkv)
    n = max(1, min(workers or host_cores(), len(units) if mode == "parity" else 1 << 30))
    need = sum(np.asarray(raw[k]).nbytes for k in _ARRAYS) + (Tq * Hq * (d + 1) * 8
                                                              if mode == "parity" else 0)
    dirpath = _scratch_dir(need)
    saved = {v: os.environ.get(v) for v in _THREAD_VARS}
    try:
        for name in _ARRAYS:
            np.save(os.path.join(dirpath, name + ".npy"), np.ascontiguousarray(raw[name]))
        if mode == "parity":
            np.lib.format.open_memmap(os.path.join(dirpath, "out.npy"), mode="w+",
                                      dtype=np.float64, shape=(Tq, Hq, d))[...] = 0.0
            np.lib.format.open_memmap(os.path.join(dirpath, "lse.npy"), mode="w+",
                                      dtype=np.float64, shape=(Tq, Hq))[...] = -np.inf
        ctx = mp.get_context("spawn")
        counter = ctx.Value("q", 0)
        barrier = ctx.Barrier(n)
        results = ctx.Queue()
        for v in _THREAD_VARS:           # one BLAS thread per worker process
            os.environ[v] = "1"
        procs = [ctx.Process(target=_worker, args=(dirpath, params, units, mode, budget_s,
                                                   rounds, counter, barrier, results),
                             daemon=True)
                 for _ in range(n)]
        for p in procs:
            p.start()
        got = []
        import queue as _queue
        while len(got) < n:
            try:
                got.append(results.get(timeout=5.0))
            except _queue.Empty:
                if sum(p.is_alive() for p in procs) < n - len(got):
                    try:   # a worker may have exited just after posting its result
                        got.append(results.get(timeout=10.0))
                    except _queue.Empty:
                        raise RuntimeError("an oracle worker process died without a result")
        for p in procs:
            p.join()
        errs = [g[1] for g in got if g[0] != "ok"]
        if errs:
            raise RuntimeError(f"oracle worker failed: {errs[0]}")
        if mode == "parity":
            out = np.array(np.load(os.path.join(dirpath, "out.npy"), mmap_mode="r"))
            lse = np.array(np.load(os.path.join(dirpath, "lse.npy"), mmap_mode="r"))
            return out, lse
        per_round = []
        for r in range(rounds):
            done = [units[k] for g in got for k in g[1][r][0]]
            wall = max(g[1][r][2] for g in got) - min(g[1][r][1] for g in got)
            per_round.append((done, wall))
        return per_round, n
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
        shutil.rmtree(dirpath, ignore_errors=True)


def paged_attention_parallel(raw: dict, block_size: int, scale: float, kv_dtype: str = "bf16",
                             k_scale: float = 1.0, v_scale: float = 1.0, causal: bool = True,
                             window: int = 0, workers: Optional[int] = None):
    """Whole-batch (out [Tq, Hq, d], lse [Tq, Hq]) as `paged_attention` gives,
    computed unit by unit on `workers` processes (default: every host core).
    raw: the arrays of `paged_attention` (q, k_cache, v_cache, cu_query_lens,
    kv_lens, block_tables)."""
    params = dict(block_size=int(block_size), scale=float(scale), kv_dtype=kv_dtype,
                  k_scale=float(k_scale), v_scale=float(v_scale), causal=bool(causal),
                  window=int(window))
    return _run(raw, params, "parity", workers, 0.0)


def time_units(raw: dict, block_size: int, scale: float, budget_s: float,
               kv_dtype: str = "bf16", k_scale: float = 1.0, v_scale: float = 1.0,
               causal: bool = True, window: int = 0, workers: Optional[int] = None,
               units: Optional[Sequence[Tuple[int, int]]] = None, rounds: int = 1):
    """Throughput of the oracle on `workers` processes (default: every host
    core). In each of `rounds` windows, after a common start, every worker
    takes (sequence, KV head) units in the given order (default: sequence
    by sequence), cycling over the batch, until budget_s of wall time has
    passed. Returns ([(units done in the window, with repeats; its wall
    seconds)] per window, worker count)."""
    params = dict(block_size=int(block_size), scale=float(scale), kv_dtype=kv_dtype,
                  k_scale=float(k_scale), v_scale=float(v_scale), causal=bool(causal),
                  window=int(window))
    return _run(raw, params, "timing", workers, float(budget_s), units, int(rounds))
