"""Programmatic dependent launches: the append and prefill kernels start while
the previous grid of the stream finishes and wait for it (griddepcontrol.wait)
before touching memory.  Kernels adjacent in one stream, eagerly and in a CUDA
graph, must give the same bytes as the same calls separated by a host sync,
including a prefill followed by an append that overwrites the cache the
prefill reads."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import (assert_within_tolerance, compare_attention, device_inputs, fi, gpu_cache,
                      oracle_attention, oracle_cache)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _plan(m, ctx, d):
    sp = d["spec"]
    plan = m.fi_plan_create(ctx)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                      sm_scale=d["sm_scale"])
    return plan


@pytest.mark.parametrize("name", ["ragged_small", "gqa3_small"])
def test_adjacent_append_and_prefill_equal_synced_calls(name):
    m = fi()
    d = device_inputs(name)
    ctx = m.fi_context_create()
    plan = _plan(m, ctx, d)
    torch.cuda.synchronize()
    # reference: each call followed by a host sync
    c_ref = gpu_cache(d)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c_ref.k_scale, c_ref.v_scale, d["slot_mapping"], c_ref)
    torch.cuda.synchronize()
    ref = torch.empty_like(d["q"])
    m.fi_prefill_run(plan, d["q"], c_ref, ref)
    torch.cuda.synchronize()
    # append -> prefill -> append (same cache, new values) -> prefill, no syncs
    c = gpu_cache(d)
    out1 = torch.empty_like(d["q"])
    out2 = torch.empty_like(d["q"])
    k2, v2 = (d["k"] * 0.5).contiguous(), (-d["v"]).contiguous()
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    m.fi_prefill_run(plan, d["q"], c, out1)
    m.fi_nvfp4_append(ctx, k2, v2, c.k_scale, c.v_scale, d["slot_mapping"], c)
    m.fi_prefill_run(plan, d["q"], c, out2)
    torch.cuda.synchronize()
    assert torch.equal(out1, ref)
    # the second prefill reads the rewritten cache: equal to a synced run on it
    c2 = gpu_cache(d)
    m.fi_nvfp4_append(ctx, k2, v2, c2.k_scale, c2.v_scale, d["slot_mapping"], c2)
    torch.cuda.synchronize()
    ref2 = torch.empty_like(d["q"])
    m.fi_prefill_run(plan, d["q"], c2, ref2)
    torch.cuda.synchronize()
    assert torch.equal(out2, ref2)
    for name_t in ("k_data", "v_data", "k_sf", "v_sf"):
        assert torch.equal(getattr(c, name_t), getattr(c2, name_t))
    # and both prefills against the oracle: the first on the cache of the
    # first append, the second on the cache both appends leave
    h = d["host"]
    host = oracle_cache(d)
    ref_out, _ = oracle_attention(d, host)
    assert_within_tolerance(compare_attention(out1, None, ref_out, None))
    assert O.append(W.bits(k2), W.bits(v2), d["k_scale"], d["v_scale"],
                    h["slot_mapping"].numpy(), host) == 0
    for name_t in ("k_data", "v_data", "k_sf", "v_sf"):
        assert np.array_equal(getattr(c, name_t).cpu().numpy(), host[name_t]), name_t
    ref_out2, _ = oracle_attention(d, host)
    assert_within_tolerance(compare_attention(out2, None, ref_out2, None))
    assert m.fi_device_status(ctx) == 0
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


def test_adjacent_calls_in_a_graph():
    m = fi()
    d = device_inputs("ragged_small")
    ctx = m.fi_context_create()
    plan = _plan(m, ctx, d)
    c_ref = gpu_cache(d)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c_ref.k_scale, c_ref.v_scale, d["slot_mapping"], c_ref)
    torch.cuda.synchronize()
    ref = torch.empty_like(d["q"])
    m.fi_prefill_run(plan, d["q"], c_ref, ref)
    torch.cuda.synchronize()
    c = gpu_cache(d)
    out = torch.zeros_like(d["q"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for _ in range(3):  # repeated appends of the same tokens, then the prefill
                m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c,
                                  stream=s)
            m.fi_prefill_run(plan, d["q"], c, out, None, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert m.fi_device_status(ctx) == 0
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)
