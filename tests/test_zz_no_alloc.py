"""fi_prefill_noalloc, the prefill entry point that allocates no memory, through
the C ABI: every call is checked against the fp64 oracle and against the
regular plan + run path on the same inputs.

Some callers cannot allocate while they run: a serving engine that reserves
all device memory for its KV cache up front and forbids allocation while it
serves, or a plugin whose enqueue callback must not allocate because the host
framework owns memory.  The no-allocation entry point keeps its scratch (the
indptr copies and the work list) in a fixed device array inside the library.
This file runs last so that a run stopping at the first failure has already run
every other test; it passes alone in a fresh process and after the others.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from gpu_util import (OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS, assert_within_tolerance,
                      compare_attention, device_inputs, fi, gpu_cache, oracle_attention,
                      oracle_cache, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _append(m, d):
    cache = gpu_cache(d)
    ctx = m.fi_context_create()
    m.fi_nvfp4_append(ctx, d["k"], d["v"], cache.k_scale, cache.v_scale, d["slot_mapping"], cache)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    return cache


def _regular(m, d, cache):
    sp = d["spec"]
    ctx = m.fi_context_create()
    plan = m.fi_plan_create(ctx)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                      sm_scale=d["sm_scale"])
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    m.fi_prefill_run(plan, d["q"], cache, out, lse)
    assert m.fi_device_status(ctx) == 0
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)
    return out, lse


def _noalloc(m, d, cache, with_status=True):
    """Calls the C entry point directly (ctypes), with caller-owned outputs and
    a caller-owned status word (or none: the bits are then discarded)."""
    sp = d["spec"]
    qo = np.ascontiguousarray(d["host"]["qo_indptr"].numpy(), dtype=np.int32)
    kv = np.ascontiguousarray(d["host"]["kv_indptr"].numpy(), dtype=np.int32)
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cc = cache.c()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = m.lib.fi_prefill_noalloc(qo.ctypes.data, kv.ctypes.data, qo.size - 1,
                                  d["page_table"].data_ptr(), d["page_table"].stride(0),
                                  sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                                  float(d["sm_scale"]), d["q"].data_ptr(), C.byref(cc),
                                  out.data_ptr(), lse.data_ptr(),
                                  status.data_ptr() if with_status else None, stream)
    assert rc == m.FI_OK, m.lib.fi_status_string(rc).decode()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


def _close(a, b, la, lb):
    err = (a.float() - b.float()).abs()
    assert float(err.max()) <= OUT_MAX_ABS and float(err.mean()) <= OUT_MEAN_ABS
    assert float((la - lb).abs().max()) <= LSE_MAX_ABS


def test_noalloc_matches_oracle_and_plan_and_run_on_calls_in_a_row():
    """Consecutive calls with different batches (ragged, uniform, then newest
    tokens over a longer cache with a sequence that has no query rows): no call
    may see anything an earlier one left in the shared scratch."""
    m = fi()
    for name in ("ragged_small", "uniform_small", "offset_small"):
        d = device_inputs(name)
        cache = _append(m, d)
        out, lse = _noalloc(m, d, cache)
        ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
        assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))
        reg_out, reg_lse = _regular(m, d, cache)
        _close(out, reg_out, lse, reg_lse)


def test_noalloc_many_units_without_a_status_word():
    """2160 ragged (sequence, q-tile) list entries: the list is staged to the
    scratch in pieces of 1024 entries (two full pieces and a tail, at growing
    offsets).  The first call passes no status word (the bits go to the scratch
    and are discarded), the second one does; both agree with plan + run on
    every row and with the oracle on sampled rows."""
    m = fi()
    d = device_inputs("many_units")
    qo = d["host"]["qo_indptr"].numpy()
    items = sum(-(-int(qo[b + 1] - qo[b]) // 128) for b in range(len(qo) - 1))
    assert items > 2 * 1024
    cache = _append(m, d)
    reg_out, reg_lse = _regular(m, d, cache)
    rows = sample_rows(d, 2000, seed=11)
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d), rows=rows)
    for with_status in (False, True):
        out, lse = _noalloc(m, d, cache, with_status=with_status)
        _close(out, reg_out, lse, reg_lse)
        assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse, rows=rows))


def test_noalloc_rejects_batches_beyond_its_scratch():
    m = fi()
    d = device_inputs("ragged_small")
    sp = d["spec"]
    cache = gpu_cache(d)
    # 300000 one-token sequences: 2 * 300001 indptr words exceed the scratch
    n = 300000
    qo = np.arange(n + 1, dtype=np.int32)
    pt = torch.zeros((n, 1), dtype=torch.int32, device="cuda")
    q = torch.zeros((n, sp.num_qo_heads, sp.head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    cc = cache.c()
    rc = m.lib.fi_prefill_noalloc(qo.ctypes.data, qo.ctypes.data, n, pt.data_ptr(), 1,
                                  sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                                  0.0, q.data_ptr(), C.byref(cc), out.data_ptr(), None, None,
                                  C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == m.FI_ERR_SCRATCH_TOO_SMALL
