"""The host-buffer entry point on batches large enough for its pipelined path
(the sequences cut into runs whose query and output copies overlap the
forward of the neighbouring runs), against the planned path and the fp64
oracle."""
import pytest
import torch

import paged_kv_attention_unified_gb300 as ua
from paged_kv_attention_unified_gb300 import torch_utils as tu
import workloads as W

from _helpers import as_f64, assert_close, oracle_full_parallel

pytestmark = pytest.mark.gpu

PIPELINE_MIN_BYTES = 32 << 20   # q bytes from which ua_forward_host cuts the batch


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_attention_unified_gb300 import build
    build.build()


def _host_forward(case, b, pinned=True, block_tables=None):
    q_h = case.q.contiguous()
    out_h = torch.full_like(q_h, float("nan"))
    cu_h, kv_h = case.cu_query_lens.to(torch.int32), case.kv_lens.to(torch.int32)
    bt_h = (case.block_tables if block_tables is None else block_tables).to(torch.int32).contiguous()
    if pinned:
        q_h, out_h, cu_h, kv_h, bt_h = (t.pin_memory() for t in (q_h, out_h, cu_h, kv_h, bt_h))
    err = ua.ua_forward_host(q_h, out_h, cu_h, kv_h, bt_h, b.k_cache, b.v_cache,
                             b.num_q_heads, b.num_kv_heads, b.head_dim, b.block_size,
                             b.num_blocks, b.kv_dtype, b.scale, causal=b.causal,
                             window=b.window, k_scale=b.k_scale, v_scale=b.v_scale)
    return err, out_h


def _prefill_case(causal=True, window=0):
    # 6300 query tokens of 32 heads x 128 dims: 51.6 MB of q in three runs
    # of 2100 tokens. Both cuts fall in the 5000-token sequence, longer than
    # a run, so where the mask allows it they fall inside it on whole
    # prefill tiles (64 tokens of 4-head rows): runs [0, 2048),
    # [2048, 4160), [4160, 6300), the last holding an empty query too; else
    # on the next boundary: [0, 5000), [5000, 6300)
    case = W.make_case("host_runs_prefill", [5000, 0, 1300], [5600, 300, 1300], 32, 8, 128, 16,
                       seed=91, causal=causal, window=window)
    assert case.q.numel() * 2 >= PIPELINE_MIN_BYTES
    return case


@pytest.mark.parametrize("causal,window,pinned", [(True, 0, True), (True, 0, False),
                                                  (False, 0, True), (True, 700, True),
                                                  (False, 700, True)])
def test_runs_of_a_prefill_batch_match_the_planned_path_bit_for_bit(causal, window, pinned):
    """Every row of a prefill tile takes the same arithmetic whatever tiles
    surround it, and a cut inside a sequence keeps the row positions (causal:
    the keys up to the run's last row; no mask: all keys; a window without
    the causal mask cuts only between sequences): the runs change no bit."""
    case = _prefill_case(causal, window)
    b = tu.to_device(case)
    ref = tu.run(case)
    err, out_h = _host_forward(case, b, pinned)
    assert err == 0
    assert torch.equal(out_h.view(torch.int16), ref.view(torch.int16))


def test_one_long_prefill_runs_in_pieces_bit_for_bit():
    """A single causal sequence of 6300 new tokens over 600 tokens of context
    (51.6 MB of q): three runs of its rows, each over the keys up to its last
    row, give the one-plan output bit for bit."""
    case = W.make_case("host_runs_one_seq", [6300], [6900], 32, 8, 128, 16, seed=92)
    assert case.q.numel() * 2 >= PIPELINE_MIN_BYTES
    b = tu.to_device(case)
    ref = tu.run(case)
    err, out_h = _host_forward(case, b)
    assert err == 0
    assert torch.equal(out_h.view(torch.int16), ref.view(torch.int16))


def test_runs_of_the_dense_prefill_workload_match_bit_for_bit():
    """The dense-prefill benchmark workload (4 x 4096 tokens, 134 MB of q in
    four runs of one sequence each) bit for bit."""
    case = W.CONFIGS[4]()
    b = tu.to_device(case)
    ref = tu.run(case)
    err, out_h = _host_forward(case, b)
    assert err == 0
    assert torch.equal(out_h.view(torch.int16), ref.view(torch.int16))


def test_runs_of_the_mixed_workload_match_the_oracle():
    """The mixed benchmark workload (8 prefill + 120 decode sequences, 68 MB
    of q) through the host path: every element against the fp64 oracle (the
    decode splits are chosen per run, so the bits may differ from the
    whole-batch plan)."""
    case = W.CONFIGS[3]()
    assert case.q.numel() * 2 >= PIPELINE_MIN_BYTES
    b = tu.to_device(case)
    err, out_h = _host_forward(case, b)
    assert err == 0
    del b
    torch.cuda.empty_cache()
    assert_close(as_f64(out_h), oracle_full_parallel(case), case.kv_dtype,
                 f"workload 3 via the host runs ({case.name})", report=True)


def test_a_bad_page_is_reported_through_the_one_plan_host_path():
    """Below the pipelining threshold the error word comes back through a
    pinned block: a bad page id still reaches the caller's word, and a clean
    call after it reads UA_OK."""
    case = W.make_case("host_bad_page_small", [1, 1, 40], [100, 64, 300], 8, 2, 128, 16, seed=93)
    assert case.q.numel() * 2 < PIPELINE_MIN_BYTES
    b = tu.to_device(case)
    bt = case.block_tables.clone()
    bt[0, 2] = case.num_blocks + 5
    err, _ = _host_forward(case, b, block_tables=bt)
    assert err == ua.UA_ERR_BOUNDS
    err, out_h = _host_forward(case, b)
    assert err == 0
    assert torch.equal(out_h.view(torch.int16), tu.run(case).view(torch.int16))


def test_a_bad_page_in_the_last_run_is_reported():
    case = _prefill_case()
    b = tu.to_device(case)
    bt = case.block_tables.clone()
    bt[2, 3] = case.num_blocks + 7          # never dereferenced, reported instead
    err, _ = _host_forward(case, b, block_tables=bt)
    assert err == ua.UA_ERR_BOUNDS
