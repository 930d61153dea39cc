"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs (drawn by workloads.py)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workloads as W

# Acceptance on attention outputs (fp64 oracle vs bf16 output).
OUT_MAX_ABS = 2e-2
OUT_MEAN_ABS = 2e-3
LSE_MAX_ABS = 1e-3


def fi():
    import nvfp4_paged_kv_slot_b300 as m
    return m


def device_inputs(name_or_spec, device="cuda", gen_device="cpu"):
    sp = W.spec(name_or_spec) if isinstance(name_or_spec, str) else name_or_spec
    d = W.make(sp, device=gen_device)
    dev = {}
    for k, v in d.items():
        dev[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    dev["host"] = d
    return dev


def gpu_cache(d, fill=0xA5):
    m = fi()
    sp = d["spec"]
    ks = torch.tensor([d["k_scale"]], dtype=torch.float32, device="cuda")
    vs = torch.tensor([d["v_scale"]], dtype=torch.float32, device="cuda")
    return m.NVFP4Cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim,
                        device="cuda", k_scale=ks, v_scale=vs, fill=fill)


def oracle_cache(d, token_mask=None, fill=0xA5):
    """Oracle append of the workload's tokens (optionally only those in
    token_mask) into a host cache."""
    sp = d["spec"]
    h = d["host"]
    cache = O.new_cache(d["num_pages"], sp.num_kv_heads, sp.page_size, sp.head_dim, fill)
    k, v, slots = h["k"], h["v"], h["slot_mapping"]
    if token_mask is not None:
        k, v, slots = k[token_mask], v[token_mask], slots[token_mask]
    st = O.append(W.bits(k), W.bits(v), d["k_scale"], d["v_scale"], slots.numpy(), cache)
    assert st == 0
    return cache


def cache_to_host(c):
    return {"k_data": c.k_data.cpu().numpy(), "v_data": c.v_data.cpu().numpy(),
            "k_sf": c.k_sf.cpu().numpy(), "v_sf": c.v_sf.cpu().numpy(),
            "num_pages": c.num_pages, "num_kv_heads": c.num_kv_heads,
            "page_size": c.page_size, "head_dim": c.head_dim}


def run_path(d, cache=None, schedule=0, num_ctas=0, with_lse=True, cta_pairs=0):
    """append -> plan -> run through the C ABI; returns (out, lse, cache, ctx, plan info)."""
    m = fi()
    sp = d["spec"]
    ctx = m.fi_context_create()
    cache = cache or gpu_cache(d)
    m.fi_nvfp4_append(ctx, d["k"], d["v"], cache.k_scale, cache.v_scale, d["slot_mapping"], cache)
    plan = m.fi_plan_create(ctx)
    m.fi_prefill_plan(plan, d["host"]["qo_indptr"], d["host"]["kv_indptr"], d["page_table"],
                      sp.num_qo_heads, sp.num_kv_heads, sp.head_dim, sp.page_size,
                      sm_scale=d["sm_scale"], schedule=schedule, num_ctas=num_ctas,
                      cta_pairs=cta_pairs)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda") if with_lse else None
    m.fi_prefill_run(plan, d["q"], cache, out, lse)
    info = m.fi_plan_get_info(plan)
    status = m.fi_device_status(ctx)
    m.fi_plan_destroy(plan)
    m.fi_context_destroy(ctx)
    return out, lse, cache, status, info


def compare_attention(out_gpu, lse_gpu, ref_out, ref_lse, rows=None):
    """out_gpu [T][H][D] bf16, ref_out [n][D] fp64 for rows (token, head) or all."""
    o = out_gpu.float().cpu().numpy()
    ls = lse_gpu.cpu().numpy() if lse_gpu is not None else None
    H, D = o.shape[1], o.shape[2]
    if rows is None:
        got = o.reshape(-1, D)
        got_lse = ls.reshape(-1) if ls is not None else None
    else:
        got = o[rows[:, 0], rows[:, 1]]
        got_lse = ls[rows[:, 0], rows[:, 1]] if ls is not None else None
    err = np.abs(got.astype(np.float64) - ref_out)
    res = {"max_abs": float(err.max()), "mean_abs": float(err.mean())}
    if got_lse is not None:
        res["lse_max_abs"] = float(np.abs(got_lse.astype(np.float64) - ref_lse).max())
    return res


def assert_within_tolerance(res):
    assert res["max_abs"] <= OUT_MAX_ABS, res
    assert res["mean_abs"] <= OUT_MEAN_ABS, res
    if "lse_max_abs" in res:
        assert res["lse_max_abs"] <= LSE_MAX_ABS, res


def oracle_attention(d, cache_host, rows=None, threads=0):
    h = d["host"]
    sp = d["spec"]
    return O.prefill(W.bits(h["q"]), h["qo_indptr"].numpy(), h["kv_indptr"].numpy(),
                     h["page_table"].numpy(), cache_host, sp.num_qo_heads, d["k_scale"],
                     d["v_scale"], d["sm_scale"], rows=rows, threads=threads)


def sample_rows(d, n, seed=0, seqs=None):
    """n (token, q head) rows, spread over sequences (optionally restricted)."""
    h = d["host"]
    sp = d["spec"]
    rng = np.random.default_rng(seed)
    qo = h["qo_indptr"].numpy()
    B = len(qo) - 1
    seqs = np.arange(B) if seqs is None else np.asarray(seqs)
    rows = []
    for _ in range(n):
        b = int(rng.choice(seqs))
        L = qo[b + 1] - qo[b]
        if L == 0:
            continue
        # bias towards the end of the sequence (longest rows) and the tile edges
        i = int(rng.choice([L - 1, 0, rng.integers(0, L), min(L - 1, 127), min(L - 1, 128)]))
        rows.append((qo[b] + i, int(rng.integers(0, sp.num_qo_heads))))
    return np.array(sorted(set(rows)), np.int64)


def oracle_attention_subset(d, cache_host, seqs, rows):
    """Oracle attention for `rows` (global (token, head)) that all belong to the
    sequences `seqs`, using only those sequences' queries (a compact batch)."""
    h = d["host"]
    sp = d["spec"]
    qo = h["qo_indptr"].cpu().numpy().astype(np.int64)
    kv = h["kv_indptr"].cpu().numpy().astype(np.int64)
    seqs = sorted(int(b) for b in seqs)
    qlens = [qo[b + 1] - qo[b] for b in seqs]
    kvlens = [kv[b + 1] - kv[b] for b in seqs]
    qo_sub = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    kv_sub = np.concatenate([[0], np.cumsum(kvlens)]).astype(np.int32)
    q_sub = torch.cat([h["q"][qo[b]:qo[b + 1]] for b in seqs]).cpu()
    pt_sub = h["page_table"].cpu().numpy()[seqs]
    pos = {b: i for i, b in enumerate(seqs)}
    seq_of = np.searchsorted(qo, rows[:, 0], side="right") - 1
    sub_rows = np.stack([qo_sub[[pos[int(b)] for b in seq_of]] + (rows[:, 0] - qo[seq_of]),
                         rows[:, 1]], 1).astype(np.int64)
    return O.prefill(W.bits(q_sub), qo_sub, kv_sub, pt_sub, cache_host, sp.num_qo_heads,
                     d["k_scale"], d["v_scale"], d["sm_scale"], rows=sub_rows)
