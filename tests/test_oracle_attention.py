"""Pins for the oracle's fp64 paged causal prefill (CPU only).

The comparison reference is built independently of the oracle's C code: the
cache is decoded with library tables (ml_dtypes float4_e2m1fn, torch
float8_e4m3fn), gathered with numpy fancy indexing, and attention is numpy
matmul + scipy logsumexp on a dense causal mask.  Closed forms pin the rest.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import workloads as W

mld = pytest.importorskip("ml_dtypes")
E2M1 = np.arange(16, dtype=np.uint8).view(mld.float4_e2m1fn).astype(np.float64)
E4M3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def lib_gather(cache, which, pt_row, kv_len, hk, g):
    ps, D = cache["page_size"], cache["head_dim"]
    j = np.arange(kv_len)
    page = pt_row[j // ps].astype(np.int64)
    off = j % ps
    data = cache[f"{which}_data"][page, hk, off]               # [kv][D/2]
    codes = np.stack([data & 0xF, data >> 4], -1).reshape(kv_len, D)
    sf = cache[f"{which}_sf"][page, hk, off]                   # [kv][D/16]
    return E2M1[codes] * np.repeat(E4M3[sf], 16, axis=1) * g


def dense_reference(q_bits, qo_indptr, kv_indptr, page_table, cache, Hq, ks, vs, sm):
    Hk, D = cache["num_kv_heads"], cache["head_dim"]
    G = Hq // Hk
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    total = int(qo_indptr[-1])
    out = np.zeros((total, Hq, D))
    lse = np.zeros((total, Hq))
    for b in range(len(qo_indptr) - 1):
        q0, q1 = int(qo_indptr[b]), int(qo_indptr[b + 1])
        qo, kv = q1 - q0, int(kv_indptr[b + 1] - kv_indptr[b])
        if qo == 0:
            continue
        for hq in range(Hq):
            K = lib_gather(cache, "k", page_table[b], kv, hq // G, ks)
            V = lib_gather(cache, "v", page_table[b], kv, hq // G, vs)
            s = sm * (q[q0:q1, hq] @ K.T)
            i = np.arange(qo)[:, None]
            j = np.arange(kv)[None, :]
            s = np.where(j <= i + kv - qo, s, -np.inf)
            l = logsumexp(s, axis=1)
            out[q0:q1, hq] = np.exp(s - l[:, None]) @ V
            lse[q0:q1, hq] = l
    return out.reshape(total * Hq, D), lse.reshape(-1)


def build_case(oracle, seq_qo, seq_kv, Hq, Hk, D, ps, seed):
    g = torch.Generator().manual_seed(seed)
    B = len(seq_kv)
    kv_indptr = np.concatenate([[0], np.cumsum(seq_kv)]).astype(np.int32)
    qo_indptr = np.concatenate([[0], np.cumsum(seq_qo)]).astype(np.int32)
    npages = [(L + ps - 1) // ps for L in seq_kv]
    P = sum(npages) + 3
    perm = torch.randperm(P, generator=g).numpy()
    pt = np.zeros((B, max(max(npages), 1) + 2), np.int32)
    slots = []
    o = 0
    for b in range(B):
        pt[b, :npages[b]] = perm[o:o + npages[b]]
        o += npages[b]
        pos = np.arange(seq_kv[b])
        slots.append(pt[b, pos // ps].astype(np.int64) * ps + pos % ps)
    slots = np.concatenate(slots) if slots else np.zeros(0, np.int64)
    N = int(kv_indptr[-1])
    k = torch.randn((N, Hk, D), generator=g).to(torch.bfloat16)
    v = torch.randn((N, Hk, D), generator=g).to(torch.bfloat16)
    q = torch.randn((int(qo_indptr[-1]), Hq, D), generator=g).to(torch.bfloat16)
    cache = oracle.new_cache(P, Hk, ps, D)
    ks, vs = W.global_scale(k), W.global_scale(v)
    assert oracle.append(W.bits(k), W.bits(v), ks, vs, slots, cache) == 0
    return dict(q=W.bits(q), qo=qo_indptr, kv=kv_indptr, pt=pt, cache=cache, ks=ks, vs=vs)


@pytest.mark.parametrize("shape", [
    # (qo lens, kv lens, Hq, Hk, D, ps)
    ([64], [64], 4, 2, 64, 16),
    ([5, 1, 37], [5, 1, 37], 6, 3, 32, 16),
    ([3, 20, 0, 7], [9, 20, 4, 30], 4, 1, 16, 8),          # qo < kv: bottom-right causal
    ([130], [200], 2, 2, 48, 32),
])
def test_paged_prefill_equals_dense_library_reference(oracle, shape):
    qo, kv, Hq, Hk, D, ps = shape
    c = build_case(oracle, qo, kv, Hq, Hk, D, ps, seed=sum(kv) + D)
    sm = 1.0 / math.sqrt(D)
    out, lse = oracle.prefill(c["q"], c["qo"], c["kv"], c["pt"], c["cache"], Hq, c["ks"],
                              c["vs"], sm)
    ref_out, ref_lse = dense_reference(c["q"], c["qo"], c["kv"], c["pt"], c["cache"], Hq,
                                       c["ks"], c["vs"], sm)
    assert np.max(np.abs(out - ref_out)) < 1e-12
    assert np.max(np.abs(lse - ref_lse)) < 1e-12


def test_tiny_workload_vs_reference(oracle):
    d = W.make(W.spec("tiny"))
    sp = d["spec"]
    cache = oracle.new_cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim)
    assert oracle.append(W.bits(d["k"]), W.bits(d["v"]), d["k_scale"], d["v_scale"],
                         d["slot_mapping"].numpy(), cache) == 0
    args = (W.bits(d["q"]), d["qo_indptr"].numpy(), d["kv_indptr"].numpy(),
            d["page_table"].numpy(), cache, sp.num_qo_heads, d["k_scale"], d["v_scale"],
            d["sm_scale"])
    out, lse = oracle.prefill(*args)
    ref_out, ref_lse = dense_reference(*args)
    assert np.max(np.abs(out - ref_out)) < 1e-12 and np.max(np.abs(lse - ref_lse)) < 1e-12
    # the tiny workload's pages really are shuffled
    assert not np.array_equal(d["page_table"].numpy()[0], np.arange(4))


def test_sampled_rows_equal_full(oracle):
    c = build_case(oracle, [40, 70], [40, 70], 4, 2, 32, 16, seed=3)
    sm = 0.17
    out, lse = oracle.prefill(c["q"], c["qo"], c["kv"], c["pt"], c["cache"], 4, c["ks"],
                              c["vs"], sm)
    rows = np.array([[0, 0], [39, 3], [40, 1], [109, 2], [75, 0]], np.int64)
    o2, l2 = oracle.prefill(c["q"], c["qo"], c["kv"], c["pt"], c["cache"], 4, c["ks"],
                            c["vs"], sm, rows=rows)
    idx = rows[:, 0] * 4 + rows[:, 1]
    assert np.array_equal(o2, out[idx]) and np.array_equal(l2, lse[idx])


def _one_seq_cache(oracle, k, v, ps=16):
    """Append one sequence in order into pages [2, 0, 1, ...] (shuffled)."""
    N, Hk, D = k.shape
    npg = (N + ps - 1) // ps
    order = np.roll(np.arange(npg), 1)
    pt = order[None, :].astype(np.int32)
    pos = np.arange(N)
    slots = pt[0, pos // ps].astype(np.int64) * ps + pos % ps
    cache = oracle.new_cache(npg, Hk, ps, D)
    ks, vs = W.global_scale(k), W.global_scale(v)
    assert oracle.append(W.bits(k), W.bits(v), ks, vs, slots, cache) == 0
    return cache, pt, ks, vs


def test_closed_form_first_row_and_identical_keys(oracle):
    """Row 0 sees only key 0: o = V_0 and lse = s_00.  With every key equal,
    all logits of a row are equal: o_i = mean(V_0..V_i), lse_i = s + ln(i+1)."""
    N, D = 40, 32
    g = torch.Generator().manual_seed(9)
    krow = torch.randn((1, 1, D), generator=g)
    k = krow.expand(N, 1, D).contiguous().to(torch.bfloat16)
    v = torch.randn((N, 1, D), generator=g).to(torch.bfloat16)
    q = torch.randn((N, 1, D), generator=g).to(torch.bfloat16)
    cache, pt, ks, vs = _one_seq_cache(oracle, k, v)
    ind = np.array([0, N], np.int32)
    sm = 0.3
    out, lse = oracle.prefill(W.bits(q), ind, ind, pt, cache, 1, ks, vs, sm)
    V = np.stack([oracle.dequant_row(cache, "v", int(pt[0, j // 16]) * 16 + j % 16, 0, vs)
                  for j in range(N)])
    K0 = oracle.dequant_row(cache, "k", int(pt[0, 0]) * 16, 0, ks)
    qd = q.double().numpy()[:, 0]
    for i in range(N):
        s = sm * float(qd[i] @ K0)
        assert np.allclose(out[i], V[:i + 1].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[i] - (s + math.log(i + 1))) < 1e-12
    assert np.array_equal(out[0], V[0])


def test_closed_form_dominant_logit(oracle):
    """A key aligned with the query and 40x larger than the rest takes all the
    weight: o = V_j to within exp(-gap)."""
    N, D = 24, 16
    g = torch.Generator().manual_seed(4)
    k = (torch.randn((N, 1, D), generator=g) * 0.01)
    q = torch.zeros((N, 1, D))
    q[:, 0, 0] = 1.0
    jstar = 5
    k[jstar, 0, 0] = 40.0
    k = k.to(torch.bfloat16)
    q = q.to(torch.bfloat16)
    v = torch.randn((N, 1, D), generator=g).to(torch.bfloat16)
    cache, pt, ks, vs = _one_seq_cache(oracle, k, v)
    ind = np.array([0, N], np.int32)
    out, _ = oracle.prefill(W.bits(q), ind, ind, pt, cache, 1, ks, vs, 1.0)
    Vj = oracle.dequant_row(cache, "v", int(pt[0, 0]) * 16 + jstar, 0, vs)
    for i in range(jstar, N):
        assert np.max(np.abs(out[i] - Vj)) < 1e-9


def test_output_is_convex_combination(oracle):
    c = build_case(oracle, [50], [50], 2, 1, 16, 16, seed=8)
    out, _ = oracle.prefill(c["q"], c["qo"], c["kv"], c["pt"], c["cache"], 2, c["ks"],
                            c["vs"], 0.25)
    V = lib_gather(c["cache"], "v", c["pt"][0], 50, 0, c["vs"])
    out = out.reshape(50, 2, 16)
    for i in range(50):
        lo, hi = V[:i + 1].min(0), V[:i + 1].max(0)
        assert np.all(out[i] >= lo - 1e-12) and np.all(out[i] <= hi + 1e-12)


def test_rejects_qo_longer_than_kv(oracle):
    c = build_case(oracle, [4], [4], 1, 1, 16, 16, seed=1)
    with pytest.raises(ValueError):
        oracle.prefill(c["q"], np.array([0, 5], np.int32), c["kv"], c["pt"], c["cache"], 1,
                       c["ks"], c["vs"], 1.0)
