"""Seeded synthetic inputs for the NVFP4 paged-KV append + causal prefill path.

This module only draws inputs (normal K/V/Q, outliers, slot mappings, page
tables, sequence lengths, global decode scales).  It holds none of the method's
arithmetic, and both the CUDA path and the CPU oracle take their inputs from it.

Workloads (shapes follow the pages' workloads; data is synthetic):
  tiny        1 x 64 tokens, H_kv=2, H_q=4, D=64, ps=16, 4 pages in shuffled order
  append      8192 tokens, H_kv=8, D=128, ps=16, 512 pages; 0.1% outliers x20;
              slots through a random page permutation, 5% (410) slots = -1
  single      1 x 2048 tokens, H_q=32, H_kv=8, D=128, ps=16, random page table
  uniform     1024 x 1024 tokens, H_q=32, H_kv=8, D=128, ps=16, random page table
  ragged      256 sequences, L = round(exp(U[ln 128, ln 16384])), qo_len = kv_len,
              H_q=32, H_kv=8, D=128, ps=16, random page table
plus small ragged cases used by the parity tests (several tiles and ragged tails,
head_dim 64 and 128, page sizes 16 to 64, GQA groups of 1 to 4).

K, V, Q ~ N(0, 1) in fp32, rounded to bf16.  The global decode scales are
k_scale = amax|K| / (6 * 448) and likewise v_scale (fp32, host).  The seed of
workload index c is 1000 * c.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

E4M3_MAX = 448.0
E2M1_MAX = 6.0


@dataclass
class Spec:
    name: str
    seed: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_qo_heads: int = 0          # 0: append-only workload
    seq_lens: list = field(default_factory=list)   # kv_len per sequence (qo_len too, unless qo_lens)
    qo_lens: list = field(default_factory=list)    # the newest qo_len tokens query (else all)
    attn: str = "prefill"          # attention the workload feeds: "prefill" or "decode"
    append_tokens: int = 0         # append-only workloads
    num_pages: int = 0             # append-only workloads
    skip_fraction: float = 0.0     # fraction of slots set to -1 (append-only)
    outlier_p: float = 0.0
    outlier_scale: float = 20.0

    @property
    def batch(self) -> int:
        return len(self.seq_lens)

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads


def ragged_lengths(batch: int, lo: int, hi: int, seed: int) -> list:
    g = torch.Generator().manual_seed(seed + 1)
    u = torch.rand(batch, generator=g, dtype=torch.float64)
    lens = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [int(round(x)) for x in lens.tolist()]


def spec(name: str) -> Spec:
    if name == "tiny":
        return Spec("tiny", 0, num_kv_heads=2, head_dim=64, page_size=16, num_qo_heads=4,
                    seq_lens=[64])
    if name == "append":
        return Spec("append", 1000, num_kv_heads=8, head_dim=128, page_size=16,
                    append_tokens=8192, num_pages=512, skip_fraction=0.05, outlier_p=0.001)
    if name == "single":
        return Spec("single", 2000, num_kv_heads=8, head_dim=128, page_size=16,
                    num_qo_heads=32, seq_lens=[2048])
    if name == "uniform":
        return Spec("uniform", 3000, num_kv_heads=8, head_dim=128, page_size=16,
                    num_qo_heads=32, seq_lens=[1024] * 1024)
    if name == "ragged":
        return Spec("ragged", 4000, num_kv_heads=8, head_dim=128, page_size=16,
                    num_qo_heads=32, seq_lens=ragged_lengths(256, 128, 16384, 4000))
    # Other shapes of the uniform batch, for the measurements of head_dim 64,
    # a GQA group of 8 and 64-token pages (first 256 sequences in the bench).
    if name == "uniform_d64":
        return Spec("uniform_d64", 3100, num_kv_heads=8, head_dim=64, page_size=16,
                    num_qo_heads=32, seq_lens=[1024] * 1024)
    if name == "uniform_g8":
        return Spec("uniform_g8", 3200, num_kv_heads=8, head_dim=128, page_size=16,
                    num_qo_heads=64, seq_lens=[1024] * 1024)
    if name == "uniform_ps64":
        return Spec("uniform_ps64", 3300, num_kv_heads=8, head_dim=128, page_size=64,
                    num_qo_heads=32, seq_lens=[1024] * 1024)
    # Small cases for the parity tests: several tiles and ragged tails.
    if name == "ragged_small":
        return Spec("ragged_small", 5000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=[1, 17, 128, 129, 300, 520])
    if name == "ragged_small_d64":
        return Spec("ragged_small_d64", 6000, num_kv_heads=2, head_dim=64, page_size=32,
                    num_qo_heads=4, seq_lens=[5, 130, 257, 64])
    # Odd GQA groups (one query head per CTA): group of 3, and plain multi-head.
    if name == "gqa3_small":
        return Spec("gqa3_small", 8000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=6, seq_lens=[100, 300, 129])
    if name == "mha_small_d64":
        return Spec("mha_small_d64", 9000, num_kv_heads=2, head_dim=64, page_size=64,
                    num_qo_heads=2, seq_lens=[70, 200])
    # Decode: the newest 1..8 tokens of each sequence query its whole cache.
    if name == "decode":
        return Spec("decode", 10000, num_kv_heads=8, head_dim=128, page_size=16,
                    num_qo_heads=32, seq_lens=[4096] * 128, qo_lens=[1] * 128, attn="decode")
    if name == "decode_spec":
        return Spec("decode_spec", 10500, num_kv_heads=8, head_dim=128, page_size=16,
                    num_qo_heads=32, seq_lens=[4096] * 128, qo_lens=[8] * 128, attn="decode")
    if name == "decode_small":
        return Spec("decode_small", 11000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=[1, 40, 300, 1000, 5000], qo_lens=[1] * 5, attn="decode")
    if name == "decode_spec_small":
        return Spec("decode_spec_small", 12000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=[8, 130, 700, 2600], qo_lens=[1, 3, 8, 2], attn="decode")
    if name == "decode_d64":
        return Spec("decode_d64", 13000, num_kv_heads=4, head_dim=64, page_size=32,
                    num_qo_heads=8, seq_lens=[257, 1500, 90], qo_lens=[1, 2, 1], attn="decode")
    # Decode with 9..16 rows per KV head (GQA 8 with two-token steps; GQA 6
    # at head_dim 64 with a 1-key sequence and a sequence split into chunks).
    if name == "decode_g8":
        return Spec("decode_g8", 13100, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=16, seq_lens=[33, 700, 3000, 64], qo_lens=[1, 2, 2, 1],
                    attn="decode")
    if name == "decode_g6_d64":
        return Spec("decode_g6_d64", 13200, num_kv_heads=2, head_dim=64, page_size=64,
                    num_qo_heads=12, seq_lens=[1, 2049, 400], qo_lens=[1, 2, 2], attn="decode")
    # Many short sequences and one long one: warps that run several pieces of
    # different sequences, and pairs cut across warps.
    if name == "decode_mixed":
        return Spec("decode_mixed", 13300, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=[3, 17, 33, 64, 5, 100, 31, 32, 2, 700, 9, 12, 40,
                                              1, 250, 48] * 2 + [3000], qo_lens=[1] * 33,
                    attn="decode")
    # 17..32 rows per KV head at head_dim 64 (GQA 4 with up to 8-token steps).
    if name == "decode_spec_d64":
        return Spec("decode_spec_d64", 13500, num_kv_heads=2, head_dim=64, page_size=32,
                    num_qo_heads=8, seq_lens=[9, 300, 1200, 64], qo_lens=[8, 5, 8, 1],
                    attn="decode")
    # Pages of 128 tokens (one page holds four 32-key steps).
    if name == "decode_ps128":
        return Spec("decode_ps128", 13400, num_kv_heads=2, head_dim=128, page_size=128,
                    num_qo_heads=8, seq_lens=[1, 129, 1000, 4100], qo_lens=[1, 1, 1, 1],
                    attn="decode")
    if name == "uniform_small":
        return Spec("uniform_small", 7000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=[384] * 6)
    # Prefill of the newest qo_len tokens of each sequence over a longer cache
    # (bottom-right causal alignment), with a sequence that has no query rows
    # inside a non-empty ragged batch; GQA 4 (CTA pairs) and 3 (one head per CTA).
    if name == "offset_small":
        return Spec("offset_small", 14000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=[300, 130, 64, 900], qo_lens=[1, 130, 0, 257])
    if name == "offset_gqa3_d64":
        return Spec("offset_gqa3_d64", 15000, num_kv_heads=2, head_dim=64, page_size=32,
                    num_qo_heads=6, seq_lens=[200, 77, 1000, 129], qo_lens=[200, 0, 129, 5])
    # The same offset for every sequence: the uniform (arithmetic) tile decoding
    # with qo_len < kv_len.
    if name == "offset_uniform_small":
        return Spec("offset_uniform_small", 16000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=[600] * 4, qo_lens=[200] * 4)
    # Many ragged work units (more than two thousand (sequence, q-tile) items).
    if name == "many_units":
        return Spec("many_units", 17000, num_kv_heads=2, head_dim=128, page_size=16,
                    num_qo_heads=8, seq_lens=ragged_lengths(512, 1, 4000, 17000))
    raise KeyError(name)


def sample_spec(name: str, n_seqs: int, seed: int = 0) -> Spec:
    """A bounded sample of workload `name`: n_seqs of its sequence lengths
    (chosen with `seed`), same heads, head_dim and page size, its own seed."""
    sp = spec(name)
    g = torch.Generator().manual_seed(sp.seed + 100 + seed)
    idx = torch.randperm(sp.batch, generator=g)[:min(n_seqs, sp.batch)].tolist()
    return Spec(f"{name}_sample{seed}", sp.seed + 100 + seed, num_kv_heads=sp.num_kv_heads,
                head_dim=sp.head_dim, page_size=sp.page_size, num_qo_heads=sp.num_qo_heads,
                seq_lens=[sp.seq_lens[i] for i in sorted(idx)],
                qo_lens=[sp.qo_lens[i] for i in sorted(idx)] if sp.qo_lens else [],
                attn=sp.attn)


def _bf16_normal(shape, gen, device, outlier_p=0.0, outlier_scale=20.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if outlier_p > 0:
        mask = torch.rand(shape, generator=gen, device=device) < outlier_p
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def global_scale(x: torch.Tensor) -> float:
    """amax|x| / (6 * 448) in fp32 (the workloads' recipe for k_scale/v_scale)."""
    amax = x.abs().max().float().item()
    return float(torch.tensor(amax / (E2M1_MAX * E4M3_MAX), dtype=torch.float32).item())


def make(sp: Spec, device="cpu") -> dict:
    """Draw every input of workload `sp` on `device` (deterministic per device)."""
    device = torch.device(device)
    gen = torch.Generator(device=device).manual_seed(sp.seed)
    hg = torch.Generator().manual_seed(sp.seed + 7)     # host-side permutations
    H, D, ps = sp.num_kv_heads, sp.head_dim, sp.page_size
    out = {"spec": sp}
    if sp.append_tokens:
        n = sp.append_tokens
        k = _bf16_normal((n, H, D), gen, device, sp.outlier_p, sp.outlier_scale)
        v = _bf16_normal((n, H, D), gen, device, sp.outlier_p, sp.outlier_scale)
        perm = torch.randperm(sp.num_pages, generator=hg)
        tok = torch.arange(n)
        slots = perm[tok // ps] * ps + tok % ps
        n_skip = int(round(sp.skip_fraction * n))
        skip = torch.randperm(n, generator=hg)[:n_skip]
        slots[skip] = -1
        out.update(k=k, v=v, slot_mapping=slots.to(torch.int64), num_pages=sp.num_pages,
                   k_scale=global_scale(k), v_scale=global_scale(v))
        return out
    lens = torch.tensor(sp.seq_lens, dtype=torch.int64)
    indptr = torch.zeros(sp.batch + 1, dtype=torch.int64)
    indptr[1:] = torch.cumsum(lens, 0)
    total = int(indptr[-1])
    pages_per_seq = (lens + ps - 1) // ps
    num_pages = int(pages_per_seq.sum())
    max_pages = int(pages_per_seq.max()) if sp.batch else 0
    perm = torch.randperm(num_pages, generator=hg)
    page_table = torch.zeros((sp.batch, max(max_pages, 1)), dtype=torch.int32)
    slot_mapping = torch.empty(total, dtype=torch.int64)
    off = 0
    for b in range(sp.batch):
        npg = int(pages_per_seq[b])
        page_table[b, :npg] = perm[off:off + npg].to(torch.int32)
        off += npg
        L = int(lens[b])
        pos = torch.arange(L)
        slot_mapping[int(indptr[b]):int(indptr[b]) + L] = (
            page_table[b, pos // ps].to(torch.int64) * ps + pos % ps)
    k = _bf16_normal((total, H, D), gen, device)
    v = _bf16_normal((total, H, D), gen, device)
    if sp.qo_lens:
        qlens = torch.tensor(sp.qo_lens, dtype=torch.int64)
        qo_indptr = torch.zeros(sp.batch + 1, dtype=torch.int64)
        qo_indptr[1:] = torch.cumsum(qlens, 0)
    else:
        qo_indptr = indptr
    q = _bf16_normal((int(qo_indptr[-1]), sp.num_qo_heads, D), gen, device)
    out.update(k=k, v=v, q=q, slot_mapping=slot_mapping, page_table=page_table,
               qo_indptr=qo_indptr.to(torch.int32), kv_indptr=indptr.to(torch.int32),
               num_pages=num_pages, k_scale=global_scale(k), v_scale=global_scale(v),
               sm_scale=1.0 / math.sqrt(D))
    return out


def causal_flops(qo_lens, kv_lens, num_qo_heads: int, head_dim: int) -> int:
    """Algorithmic causal FLOPs: 4 * D * H_q * sum_b sum_i (i + kv - qo + 1)."""
    total = 0
    for qo, kv in zip(qo_lens, kv_lens):
        d = kv - qo
        total += qo * (qo + 1) // 2 + qo * d
    return 4 * head_dim * num_qo_heads * total


def bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
