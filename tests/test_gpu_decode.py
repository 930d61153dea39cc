"""Decode through the C ABI vs the oracle: the newest 1..8 tokens of each
sequence attend to its whole NVFP4 cache (query row t sees keys
j <= t + kv_len - qo_len), the keys split evenly over the kernel's warps and
pairs cut into several pieces merged, within the same tolerances as the
prefill."""
import numpy as np
import pytest
import torch

from gpu_util import (assert_within_tolerance, compare_attention, device_inputs, fi, gpu_cache,
                      oracle_attention, oracle_attention_subset, oracle_cache)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _run_decode(d):
    m = fi()
    sp = d["spec"]
    ctx = m.fi_context_create()
    c = gpu_cache(d)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    plan = m.fi_plan_create(ctx)
    m.fi_decode_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                     sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                     sm_scale=d["sm_scale"])
    info = m.fi_plan_get_info(plan)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    m.fi_decode_run(plan, d["q"], c, out, lse)
    status = m.fi_device_status(ctx)
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)
    return out, lse, c, status, info


@pytest.mark.parametrize("name", ["decode_small", "decode_spec_small", "decode_d64", "decode_g8",
                                  "decode_g6_d64", "decode_mixed", "decode_ps128",
                                  "decode_spec_d64"])
def test_decode_matches_oracle(name):
    d = device_inputs(name)
    out, lse, c, status, info = _run_decode(d)
    assert status == 0
    sp = d["spec"]
    assert info["max_qo_len"] == max(sp.qo_lens) and info["max_kv_len"] == max(sp.seq_lens)
    host = oracle_cache(d)
    ref_out, ref_lse = oracle_attention(d, host)
    res = compare_attention(out, lse, ref_out, ref_lse)
    print(name, info["num_units"], res)
    assert_within_tolerance(res)


def test_decode_splits_long_sequences_into_merged_pieces():
    """decode_small has a 5000-key sequence: cut into pieces over several
    warps, merged; its rows must agree with the oracle like the others."""
    d = device_inputs("decode_small")
    out, lse, _, status, info = _run_decode(d)
    assert status == 0
    sp = d["spec"]
    # 404 steps of 32 keys over 51 warps: more pieces than (sequence, head) pairs
    assert info["num_units"] > sp.num_kv_heads * len(sp.seq_lens)
    host = oracle_cache(d)
    ref_out, ref_lse = oracle_attention(d, host)
    last = int(d["host"]["qo_indptr"][-1]) - 1   # the 5000-key sequence's query row
    rows = np.array([(last, h) for h in range(sp.num_qo_heads)], np.int64)
    sel = rows[:, 0] * sp.num_qo_heads + rows[:, 1]
    res = compare_attention(out, lse, ref_out[sel], ref_lse[sel], rows=rows)
    assert_within_tolerance(res)


def test_decode_repeated_runs_merge_every_time():
    """Three runs of one plan with split pairs (output cleared in between, the
    partial slots reused) must each match the oracle."""
    m = fi()
    d = device_inputs("decode_small")
    sp = d["spec"]
    ctx = m.fi_context_create()
    c = gpu_cache(d)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    plan = m.fi_plan_create(ctx)
    m.fi_decode_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                     sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                     sm_scale=d["sm_scale"])
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    for _ in range(3):
        out = torch.full_like(d["q"], float("nan"))
        lse = torch.full(d["q"].shape[:2], float("nan"), dtype=torch.float32, device="cuda")
        m.fi_decode_run(plan, d["q"], c, out, lse)
        assert m.fi_device_status(ctx) == 0
        assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


def test_decode_step_captured_in_a_cuda_graph():
    """The append of the newest tokens, the decode and its merge captured in
    one CUDA graph on a side stream: two replays give the bytes of the eager
    calls, and the oracle's result."""
    m = fi()
    d = device_inputs("decode_mixed")
    sp = d["spec"]
    ctx = m.fi_context_create()
    c = gpu_cache(d)
    plan = m.fi_plan_create(ctx)
    m.fi_decode_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                     sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                     sm_scale=d["sm_scale"])
    assert m.fi_plan_get_info(plan)["num_units"] > sp.batch * sp.num_kv_heads  # pairs merged

    def step(stream=None):
        m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c,
                          stream=stream)
        m.fi_decode_run(plan, d["q"], c, out, lse, stream=stream)

    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    step()
    torch.cuda.synchronize()
    eager_out, eager_lse = out.clone(), lse.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(stream=s)
    for _ in range(2):
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager_out) and torch.equal(lse, eager_lse)
    assert m.fi_device_status(ctx) == 0
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


def test_decode_plan_limits_and_plan_kinds():
    m = fi()
    d = device_inputs("decode_small")
    sp = d["spec"]
    ctx = m.fi_context_create()
    plan = m.fi_plan_create(ctx)
    qo = np.array([0, 9], np.int32)           # 9 query tokens: more than a decode plan takes
    kv = np.array([0, 40], np.int32)
    with pytest.raises(m.FiError):
        m.fi_decode_plan(plan, qo, kv, d["page_table"][:1], sp.num_qo_heads, sp.num_kv_heads,
                         sp.head_dim, sp.page_size)
    m.fi_decode_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                     sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size)
    c = gpu_cache(d)
    out = torch.empty_like(d["q"])
    with pytest.raises(m.FiError):
        m.fi_prefill_run(plan, d["q"], c, out)     # a decode plan is not a prefill plan
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size)
    with pytest.raises(m.FiError):
        m.fi_decode_run(plan, d["q"], c, out)      # and the other way round
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


def test_decode_equals_prefill_path_on_the_same_inputs():
    """The prefill path also serves decode shapes; both must agree closely."""
    m = fi()
    d = device_inputs("decode_spec_small")
    sp = d["spec"]
    out_d, lse_d, c, status, _ = _run_decode(d)
    assert status == 0
    ctx = m.fi_context_create()
    plan = m.fi_plan_create(ctx)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                      sm_scale=d["sm_scale"])
    out_p = torch.empty_like(d["q"])
    lse_p = torch.empty_like(lse_d)
    m.fi_prefill_run(plan, d["q"], c, out_p, lse_p)
    assert m.fi_device_status(ctx) == 0
    assert (out_d.float() - out_p.float()).abs().max().item() <= 2e-2
    assert (lse_d - lse_p).abs().max().item() <= 1e-3
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


def test_decode_page_id_out_of_range_flagged():
    """A page-table entry outside [0, num_pages) is read as page 0 and flagged
    with FI_DEV_PAGE_OOB (the run neither faults nor reads outside the cache)."""
    d = device_inputs("decode_small")
    d["page_table"][3, 2] = 1 << 20
    d["page_table"][4, 0] = -5
    _, _, _, status, _ = _run_decode(d)
    assert status & fi().FI_DEV_PAGE_OOB


@pytest.mark.parametrize("name", ["decode", "decode_spec"])
def test_decode_full_size_sampled(name):
    """The bench's decode batches (128 x 4096 keys; 1 and 8 query tokens per
    sequence) in the bench's launch configuration: every query row of six
    sampled sequences against the oracle."""
    d = device_inputs(name, gen_device="cuda")
    out, lse, _, status, info = _run_decode(d)
    assert status == 0
    sp = d["spec"]
    h = d["host"]
    qo = h["qo_indptr"].cpu().numpy()
    kv = h["kv_indptr"].cpu().numpy()
    seqs = np.random.default_rng(11).choice(len(qo) - 1, size=6, replace=False)
    mask = torch.zeros(int(kv[-1]), dtype=torch.bool)
    for b in seqs:
        mask[kv[b]:kv[b + 1]] = True
    for k in ("k", "v", "slot_mapping"):
        h[k] = h[k].cpu()
    host_cache = oracle_cache(d, token_mask=mask)
    rows = np.array([(t, hq) for b in sorted(seqs) for t in range(qo[b], qo[b + 1])
                     for hq in range(sp.num_qo_heads)], np.int64)
    ref_out, ref_lse = oracle_attention_subset(d, host_cache, seqs, rows)
    res = compare_attention(out, lse, ref_out, ref_lse, rows=rows)
    print(name, info["num_units"], res)
    assert_within_tolerance(res)


def test_one_plan_object_replanned_across_kinds():
    """One plan object planned in turn for a ragged prefill, a decode, a
    uniform prefill (no work list), a balanced prefill and the decode again:
    every plan keeps only its own lists (the plan reuses their memory), and
    every run matches the oracle."""
    m = fi()
    ctx = m.fi_context_create()
    plan = m.fi_plan_create(ctx)
    # tiny: one 64-token sequence, a balanced plan (slot lists)
    for name in ["ragged_small", "decode_small", "uniform_small", "tiny", "decode_mixed"]:
        d = device_inputs(name)
        sp = d["spec"]
        c = gpu_cache(d)
        m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
        args = (plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size)
        out = torch.empty_like(d["q"])
        lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
        if sp.attn == "decode":
            m.fi_decode_plan(*args, sm_scale=d["sm_scale"])
            m.fi_decode_run(plan, d["q"], c, out, lse)
        else:
            m.fi_prefill_plan(*args, sm_scale=d["sm_scale"])
            m.fi_prefill_run(plan, d["q"], c, out, lse)
        assert m.fi_device_status(ctx) == 0, name
        ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
        assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)
