"""Seeded random shapes through the C ABI against the oracle: head_dim 64 or
128, 1 to 3 KV heads, GQA groups of 1 to 8, pages of 16 to 128 tokens, 1 to 5
sequences of 1 to 700 keys, queries over the newest qo_len tokens (some
sequences with none).  Prefill on the default kernel (CTA pairs where the group
is a multiple of 4) and on single CTAs; decode with up to 8 query tokens and at
most 32 rows per KV head.  Same tolerances as every attention test."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_util import (assert_within_tolerance, compare_attention, device_inputs, fi, gpu_cache,
                      oracle_attention, oracle_cache, run_path)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _random_spec(seed, decode):
    rng = np.random.default_rng(seed)
    head_dim = int(rng.choice([64, 128]))
    kv_heads = int(rng.integers(1, 4))
    page_size = int(rng.choice([16, 32, 64, 128]))
    batch = int(rng.integers(1, 6))
    kv_lens = [int(x) for x in rng.integers(1, 701, size=batch)]
    if decode:
        qo_max = int(rng.choice([1, 2, 4, 8]))
        group = int(rng.choice([g for g in (1, 2, 3, 4, 6, 8) if g * qo_max <= 32]))
        qo_lens = [min(int(rng.integers(1, qo_max + 1)), k) for k in kv_lens]
    else:
        group = int(rng.choice([1, 2, 3, 4, 6, 8]))
        qo_lens = [int(rng.integers(0, k + 1)) if rng.random() < 0.5 else k for k in kv_lens]
        if sum(qo_lens) == 0:
            qo_lens[0] = kv_lens[0]
    return W.Spec(f"random{seed}", 30000 + seed, num_kv_heads=kv_heads, head_dim=head_dim,
                  page_size=page_size, num_qo_heads=kv_heads * group, seq_lens=kv_lens,
                  qo_lens=qo_lens, attn="decode" if decode else "prefill")


@pytest.mark.parametrize("seed", range(16))
def test_random_prefill_matches_oracle(seed):
    sp = _random_spec(seed, decode=False)
    d = device_inputs(sp)
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    for cta_pairs in (0, 1):
        out, lse, _, status, info = run_path(d, cta_pairs=cta_pairs)
        assert status == 0
        res = compare_attention(out, lse, ref_out, ref_lse)
        print(sp, cta_pairs, info["ctas_per_unit"], res)
        assert_within_tolerance(res)


@pytest.mark.parametrize("seed", range(16))
def test_random_decode_matches_oracle(seed):
    m = fi()
    sp = _random_spec(100 + seed, decode=True)
    d = device_inputs(sp)
    ctx = m.fi_context_create()
    c = gpu_cache(d)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    plan = m.fi_plan_create(ctx)
    m.fi_decode_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                     sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                     sm_scale=d["sm_scale"])
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    m.fi_decode_run(plan, d["q"], c, out, lse)
    status = m.fi_device_status(ctx)
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)
    assert status == 0
    ref_out, ref_lse = oracle_attention(d, oracle_cache(d))
    res = compare_attention(out, lse, ref_out, ref_lse)
    print(sp, res)
    assert_within_tolerance(res)
