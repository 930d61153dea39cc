"""FP8 (E4M3) paged KV variant through the C ABI vs the oracle: append bytes
bit-exact (untouched bytes keep the 0xA5 sentinel), prefill within the same
tolerances as the NVFP4 path, plans bound to their cache format."""
import numpy as np
import pytest
import torch

import oracle as O
import workloads as W
from gpu_util import assert_within_tolerance, compare_attention, device_inputs, fi

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def fp8_scales(d):
    """Decode scales that map each tensor's amax to 448 (fp32)."""
    h = d["host"]
    ks = np.float32(h["k"].float().abs().max().item() / 448.0)
    vs = np.float32(h["v"].float().abs().max().item() / 448.0)
    return float(ks), float(vs)


def gpu_fp8_cache(d, ks, vs, fill=0xA5):
    m = fi()
    sp = d["spec"]
    return m.FP8Cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim,
                      k_scale=torch.tensor([ks], dtype=torch.float32, device="cuda"),
                      v_scale=torch.tensor([vs], dtype=torch.float32, device="cuda"), fill=fill)


def oracle_fp8_cache(d, ks, vs):
    sp = d["spec"]
    h = d["host"]
    c = O.new_fp8_cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim)
    assert O.fp8_append(W.bits(h["k"]), W.bits(h["v"]), ks, vs, h["slot_mapping"].numpy(), c) == 0
    return c


def assert_fp8_cache_equal(c, host):
    for name in ("k_data", "v_data"):
        got = getattr(c, name).cpu().numpy()
        diff = np.argwhere(got != host[name])
        assert diff.size == 0, f"{name}: {len(diff)} bytes differ, first at {diff[:4].tolist()}"


@pytest.mark.parametrize("name", ["tiny", "append", "ragged_small", "mha_small_d64"])
def test_fp8_append_bit_exact(name):
    m = fi()
    d = device_inputs(name)
    ks, vs = fp8_scales(d)
    c = gpu_fp8_cache(d, ks, vs)
    ctx = m.fi_context_create()
    m.fi_fp8_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    assert_fp8_cache_equal(c, oracle_fp8_cache(d, ks, vs))


@pytest.mark.parametrize("H,D,N,gk,gv", [
    (8, 128, 333, 1e-32, 7e30),   # scales outside the fast division's range
    (2, 64, 1000, 1e-39, 3e-5),   # subnormal g
    (8, 128, 500, 0.01, 0.02),
])
def test_fp8_append_extreme_magnitudes(oracle, H, D, N, gk, gv):
    """Groups with elements below 2^-100 or far above the scale take the IEEE
    division; zeros, saturation and signed zeros as the oracle."""
    m = fi()
    ps = 16
    P = (N + ps - 1) // ps + 3
    g = torch.Generator().manual_seed(H * 1000 + N)
    x = torch.randn((2, N, H, D), generator=g)
    mag = torch.tensor([1.0, 1e-33, 1e-20, 1e4, 1e30, 3e-5, 0.0])
    pick = torch.randint(0, len(mag), (2, N, H, D // 16, 1), generator=g)
    x = (x.view(2, N, H, D // 16, 16) * mag[pick]).view(2, N, H, D)
    x[0, 0, 0, :8] = -0.0
    kv = x.to(torch.bfloat16)
    slots = torch.randperm(P * ps, generator=g)[:N].to(torch.int64)
    slots[::7] = -1
    c = m.FP8Cache(P, H, ps, D, k_scale=torch.tensor([gk], device="cuda"),
                   v_scale=torch.tensor([gv], device="cuda"), fill=0xA5)
    ctx = m.fi_context_create()
    m.fi_fp8_append(ctx, kv[0].cuda(), kv[1].cuda(), c.k_scale, c.v_scale, slots.cuda(), c)
    assert m.fi_device_status(ctx) == 0
    m.fi_context_destroy(ctx)
    host = oracle.new_fp8_cache(P, H, ps, D)
    assert oracle.fp8_append(W.bits(kv[0]), W.bits(kv[1]), float(np.float32(gk)),
                             float(np.float32(gv)), slots.numpy(), host) == 0
    assert_fp8_cache_equal(c, host)


def _pages_spec(page_size, num_qo_heads):
    """Ragged lengths with partial last pages and queries over a longer cache,
    on pages of `page_size` tokens (GQA 4: CTA pairs; GQA 1: one CTA)."""
    return W.Spec(f"fp8_pages{page_size}_h{num_qo_heads}", 21000 + page_size + num_qo_heads,
                  num_kv_heads=2, head_dim=128, page_size=page_size, num_qo_heads=num_qo_heads,
                  seq_lens=[1, 70, 256, 333, 129], qo_lens=[1, 70, 200, 333, 5])


@pytest.mark.parametrize("name", ["tiny", "ragged_small", "ragged_small_d64", "uniform_small",
                                  "gqa3_small", "mha_small_d64", (32, 8), (64, 8), (128, 8),
                                  (128, 2)])
def test_fp8_prefill_matches_oracle(name):
    m = fi()
    d = device_inputs(_pages_spec(*name) if isinstance(name, tuple) else name)
    sp = d["spec"]
    ks, vs = fp8_scales(d)
    c = gpu_fp8_cache(d, ks, vs)
    ctx = m.fi_context_create()
    m.fi_fp8_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    plan = m.fi_plan_create(ctx)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                      sm_scale=d["sm_scale"], kv_format=1)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
    m.fi_prefill_run_fp8(plan, d["q"], c, out, lse)
    assert m.fi_device_status(ctx) == 0
    host = oracle_fp8_cache(d, ks, vs)
    assert_fp8_cache_equal(c, host)
    h = d["host"]
    ref_out, ref_lse = O.prefill(W.bits(h["q"]), h["qo_indptr"].numpy(), h["kv_indptr"].numpy(),
                                 h["page_table"].numpy(), host, sp.num_qo_heads, ks, vs,
                                 d["sm_scale"])
    res = compare_attention(out, lse, ref_out, ref_lse)
    print(name, res)
    assert_within_tolerance(res)
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


def test_plans_are_bound_to_their_cache_format():
    m = fi()
    d = device_inputs("tiny")
    sp = d["spec"]
    ctx = m.fi_context_create()
    plan = m.fi_plan_create(ctx)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size)
    c8 = gpu_fp8_cache(d, 1.0, 1.0)
    out = torch.empty_like(d["q"])
    with pytest.raises(m.FiError):
        m.fi_prefill_run_fp8(plan, d["q"], c8, out)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size, kv_format=1)
    c4 = m.NVFP4Cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim)
    with pytest.raises(m.FiError):
        m.fi_prefill_run(plan, d["q"], c4, out)
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)


@pytest.mark.parametrize("bad", [0.0, -1.0, float("inf"), float("nan")])
def test_fp8_bad_device_scale_writes_nothing(bad):
    m = fi()
    d = device_inputs("tiny")
    c = gpu_fp8_cache(d, 1.0, 1.0)
    c.k_scale.fill_(bad)
    ctx = m.fi_context_create()
    m.fi_fp8_append(ctx, d["k"], d["v"], c.k_scale, c.v_scale, d["slot_mapping"], c)
    assert m.fi_device_status(ctx) == m.FI_DEV_BAD_K_SCALE
    assert bool((c.k_data == 0xA5).all()) and bool((c.v_data == 0xA5).all())
    m.fi_context_destroy(ctx)
