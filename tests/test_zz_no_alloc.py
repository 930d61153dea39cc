"""fi_prefill_noalloc, the prefill entry point that allocates no memory, checked
against the regular plan + run path through the C ABI.

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

from gpu_util import (OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS, device_inputs, fi, gpu_cache)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


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


def _noalloc(m, d, cache):
    """Calls the C entry point directly (ctypes), with caller-owned outputs and
    a caller-owned status word."""
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
                                  out.data_ptr(), lse.data_ptr(), status.data_ptr(), stream)
    assert rc == m.FI_OK, m.lib.fi_status_string(rc).decode()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out, lse


def _close(a, b, la, lb):
    err = (a.float() - b.float()).abs()
    assert float(err.max()) <= OUT_MAX_ABS and float(err.mean()) <= OUT_MEAN_ABS
    assert float((la - lb).abs().max()) <= LSE_MAX_ABS


def test_noalloc_matches_plan_and_run_on_two_calls_in_a_row():
    """Two consecutive calls with different batches (ragged, then uniform):
    the second call must not see anything the first left in the shared scratch."""
    m = fi()
    for name in ("ragged_small", "uniform_small"):
        d = device_inputs(name)
        cache = gpu_cache(d)
        ctx = m.fi_context_create()
        m.fi_nvfp4_append(ctx, d["k"], d["v"], cache.k_scale, cache.v_scale,
                          d["slot_mapping"], cache)
        assert m.fi_device_status(ctx) == 0
        m.fi_context_destroy(ctx)
        ref_out, ref_lse = _regular(m, d, cache)
        out, lse = _noalloc(m, d, cache)
        _close(out, ref_out, lse, ref_lse)


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
