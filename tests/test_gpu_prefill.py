"""Causal NVFP4 prefill through the C ABI (append -> plan -> run) vs the fp64
oracle: max-abs 2e-2, mean-abs 2e-3 on the output, 1e-3 on the LSE."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import (assert_within_tolerance, cache_to_host, compare_attention, device_inputs,
                      fi, gpu_cache, oracle_attention, oracle_attention_subset, oracle_cache,
                      run_path, sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", ["tiny", "ragged_small", "ragged_small_d64", "uniform_small",
                                  "gqa3_small", "mha_small_d64"])
@pytest.mark.parametrize("schedule", [0, 1, 2])
def test_prefill_matches_oracle(name, schedule):
    d = device_inputs(name)
    out, lse, cache, status, info = run_path(d, schedule=schedule)
    assert status == 0
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    res = compare_attention(out, lse, ref_out, ref_lse)
    print(name, schedule, info, res)
    assert_within_tolerance(res)


@pytest.mark.parametrize("name", ["ragged_small", "uniform_small"])
@pytest.mark.parametrize("schedule", [0, 1])
def test_prefill_single_cta_path_for_groups_of_four(name, schedule):
    """GQA groups of 4 run on CTA pairs by default; the single-CTA kernel (two
    heads per CTA, no shared staging) must give the same results."""
    d = device_inputs(name)
    out, lse, _, status, info = run_path(d, schedule=schedule, cta_pairs=1)
    assert status == 0 and info["ctas_per_unit"] == 1
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))
    pair_out, pair_lse, _, status, info = run_path(d, schedule=schedule)
    assert status == 0 and info["ctas_per_unit"] == 2
    assert_within_tolerance(compare_attention(pair_out, pair_lse, ref_out, ref_lse))


@pytest.mark.parametrize("name", ["offset_small", "offset_gqa3_d64", "offset_uniform_small"])
@pytest.mark.parametrize("schedule", [0, 1, 2])
@pytest.mark.parametrize("cta_pairs", [0, 1])
def test_prefill_bottom_right_causal_matches_oracle(name, schedule, cta_pairs):
    """qo_len < kv_len: query row i of a sequence sees keys j <= i + kv_len -
    qo_len (the newest qo_len tokens query the whole cache), including a
    sequence with no query rows inside a ragged batch, on the arithmetic
    (uniform) and list (ragged) tile decodings, every schedule, and both the
    CTA-pair and single-CTA kernels."""
    d = device_inputs(name)
    sp = d["spec"]
    out, lse, cache, status, info = run_path(d, schedule=schedule, cta_pairs=cta_pairs)
    assert status == 0
    assert info["is_uniform"] == (len(set(sp.seq_lens)) == 1 and len(set(sp.qo_lens)) == 1)
    if sp.group % 4 == 0:
        assert info["ctas_per_unit"] == (1 if cta_pairs else 2)
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    res = compare_attention(out, lse, ref_out, ref_lse)
    print(name, schedule, cta_pairs, info, res)
    assert_within_tolerance(res)


@pytest.mark.parametrize("cta_pairs", [0, 1])
def test_prefill_rescale_when_only_some_rows_of_a_warp_grow(cta_pairs):
    """A key of large norm at position 200 of a 300-token sequence, aligned
    with query row 210: in the second KV tile the running maximum of some rows
    (those at or after the key, and aligned with it) grows past the lazy
    rescale threshold while the other rows of their warps do not see the key
    (causal mask) and keep theirs.  The rescale of O must still match the
    oracle."""
    sp = W.Spec("rescale_split", 19000, num_kv_heads=2, head_dim=128, page_size=16,
                num_qo_heads=8, seq_lens=[300])
    d = device_inputs(sp)
    g = sp.num_qo_heads // sp.num_kv_heads
    for h in range(sp.num_kv_heads):
        big = 8.0 * torch.sign(d["host"]["q"][210, h * g].float())
        d["host"]["k"][200, h] = big.to(torch.bfloat16)
    d["k"] = d["host"]["k"].to("cuda")
    out, lse, cache, status, info = run_path(d, cta_pairs=cta_pairs)
    assert status == 0
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))


@pytest.mark.parametrize("page_size", [32, 64, 128])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("cta_pairs", [0, 1])
def test_prefill_page_sizes(page_size, head_dim, cta_pairs):
    """Pages of 32, 64 and 128 tokens: a 128-key tile spans 4, 2 or 1 pages.
    On CTA pairs each CTA copies the pages of its 64 rows of a tile (two of 32
    tokens, one of 64, or half of a 128-token page); the single-CTA kernel
    copies whole pages.  Ragged lengths with partial last pages, a length that
    fills its pages exactly, and queries over a longer cache."""
    sp = W.Spec(f"pages{page_size}_d{head_dim}", 20000 + page_size + head_dim, num_kv_heads=2,
                head_dim=head_dim, page_size=page_size, num_qo_heads=8,
                seq_lens=[1, 70, 256, 333, 129], qo_lens=[1, 70, 200, 333, 5])
    d = device_inputs(sp)
    out, lse, cache, status, info = run_path(d, cta_pairs=cta_pairs)
    assert status == 0
    assert info["ctas_per_unit"] == (1 if cta_pairs else 2)
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    res = compare_attention(out, lse, ref_out, ref_lse)
    print(page_size, head_dim, cta_pairs, info, res)
    assert_within_tolerance(res)


def test_prefill_single_sequence_2048_sampled():
    d = device_inputs("single")
    out, lse, cache, status, info = run_path(d)
    assert status == 0 and info["global_reverse"] == 1
    rows = sample_rows(d, 3000, seed=1)
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d), rows=rows)
    res = compare_attention(out, lse, ref_out, ref_lse, rows=rows)
    print(res)
    assert_within_tolerance(res)


def test_prefill_few_ctas_many_units():
    """A persistent grid much smaller than the work (each CTA loops)."""
    d = device_inputs("ragged_small")
    out, lse, _, status, _ = run_path(d, num_ctas=3)
    assert status == 0
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    assert_within_tolerance(compare_attention(out, lse, ref_out, ref_lse))


def test_prefill_without_lse_and_graph_capture():
    m = fi()
    d = device_inputs("ragged_small")
    sp = d["spec"]
    ctx = m.fi_context_create()
    c = gpu_cache(d)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    plan = m.fi_plan_create(ctx)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size)
    eager = torch.empty_like(d["q"])
    m.fi_prefill_run(plan, d["q"], c, eager)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    out = torch.zeros_like(d["q"])
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            m.fi_prefill_run(plan, d["q"], c, out, None, stream=s)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert m.fi_device_status(ctx) == 0
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


def test_bad_page_id_flagged():
    d = device_inputs("tiny")
    d["page_table"][0, 1] = 10_000
    out, lse, _, status, _ = run_path(d)
    assert status & fi().FI_DEV_PAGE_OOB


def test_empty_batch_and_zero_length_sequences():
    m = fi()
    ctx = m.fi_context_create()
    plan = m.fi_plan_create(ctx)
    pt = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    m.fi_prefill_plan(plan, [0, 0], [0, 0], pt, 4, 2, 64, 16)
    assert m.fi_plan_get_info(plan)["num_units"] == 0
    c = m.NVFP4Cache(1, 2, 16, 64)
    q = torch.empty((0, 4, 64), dtype=torch.bfloat16, device="cuda")
    m.fi_prefill_run(plan, q, c, torch.empty_like(q))
    assert m.fi_device_status(ctx) == 0
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


@pytest.mark.parametrize("name", ["uniform", "ragged"])
def test_full_size_sampled(name):
    """Full-size workloads: cache bytes of the sampled sequences bit-exact,
    sampled attention rows within tolerance."""
    d = device_inputs(name, gen_device="cuda")
    out, lse, cache, status, info = run_path(d)
    assert status == 0
    h = d["host"]
    qo = h["qo_indptr"].cpu().numpy()
    B = len(qo) - 1
    rng = np.random.default_rng(7)
    seqs = rng.choice(B, size=min(6, B), replace=False)
    mask = torch.zeros(int(qo[-1]), dtype=torch.bool)
    for b in seqs:
        mask[qo[b]:qo[b + 1]] = True
    for k in ("k", "v", "slot_mapping"):
        h[k] = h[k].cpu()
    host_cache = oracle_cache(d, token_mask=mask)
    g = cache_to_host(cache)
    slots = h["slot_mapping"][mask].numpy()
    pages, offs = slots // d["spec"].page_size, slots % d["spec"].page_size
    for name_ in ("k_data", "v_data", "k_sf", "v_sf"):
        assert np.array_equal(g[name_][pages, :, offs], host_cache[name_][pages, :, offs]), name_
    rows = sample_rows(d, 1500, seed=3, seqs=seqs)
    ref_out, ref_lse = oracle_attention_subset(d, host_cache, seqs, rows)
    res = compare_attention(out, lse, ref_out, ref_lse, rows=rows)
    print(name, info, res)
    assert_within_tolerance(res)


def test_plan_append_run_return_while_the_stream_is_busy():
    """No hidden host synchronization ([#5043]-style planning, [#6204] append):
    with the stream held by a bounded sleep kernel, a steady-state plan (its
    staging buffers already allocated), an append and a run all return
    before the sleep has finished."""
    import time
    m = fi()
    d = device_inputs("ragged_small")
    sp = d["spec"]
    ctx = m.fi_context_create()
    c = gpu_cache(d)
    plan = m.fi_plan_create(ctx)
    args = (d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"], sp.num_qo_heads,
            sp.num_kv_heads, sp.head_dim, sp.page_size)
    out = torch.empty_like(d["q"])
    for _ in range(2):                      # allocate both staging buffers
        m.fi_prefill_plan(plan, *args)
        m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
        m.fi_prefill_run(plan, d["q"], c, out)
    torch.cuda.synchronize()
    done = torch.cuda.Event()
    torch.cuda._sleep(400_000_000)          # ~0.2 s at 2 GHz, bounded
    t0 = time.perf_counter()
    m.fi_prefill_plan(plan, *args)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    m.fi_prefill_run(plan, d["q"], c, out)
    dt = time.perf_counter() - t0
    done.record()
    busy = not done.query()
    torch.cuda.synchronize()
    assert busy and dt < 0.05, (busy, dt)
    assert m.fi_device_status(ctx) == 0
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)
