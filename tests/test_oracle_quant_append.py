"""Pins for the oracle's block quantizer and slot_mapping append (CPU only)."""
import math
import pathlib

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = pathlib.Path(__file__).parent / "golden" / "quant_block_cases.txt"


def _bf16_bits(vals):
    t = torch.tensor(vals, dtype=torch.float32)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t), "fixture value not exact in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


def _cases():
    for line in GOLDEN.read_text().splitlines():
        if not line.startswith("case "):
            continue
        name, g, xs, s8, packed = [p.strip() for p in line[5:].split("|")]
        yield (name, float(g), [float(v) for v in xs.split()], int(s8, 16),
               [int(b, 16) for b in packed.split()])


@pytest.mark.parametrize("case", list(_cases()), ids=lambda c: c[0])
def test_hand_worked_blocks(oracle, case):
    _, g, xs, s8, packed = case
    got_packed, got_s8 = oracle.quantize_block16(_bf16_bits(xs), g)
    assert got_s8 == s8
    assert list(got_packed) == packed


def _nibbles(packed):
    out = []
    for b in packed:
        out += [int(b) & 0xF, int(b) >> 4]
    return out


def _random_blocks(n, seed):
    rng = np.random.default_rng(seed)
    scale = np.exp2(rng.uniform(-12, 12, size=(n, 1)))
    x = rng.standard_normal((n, 16)) * scale
    x[rng.random((n, 16)) < 0.02] *= 20.0
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)


def test_steps_round_like_library_codecs(oracle):
    """Each rounding step of the quantizer equals a library conversion of the
    same fp32 operand: torch float8_e4m3fn for s8 (t < 448 here), ml_dtypes
    float4_e2m1fn for the codes."""
    mld = pytest.importorskip("ml_dtypes")
    xb = _random_blocks(4000, 11)
    for g in (1.0, 0.00173, 3.7e-5):
        g32 = np.float32(g)
        for row in xb:
            x = row.float().numpy()
            packed, s8 = oracle.quantize_block16(row.view(torch.int16).numpy().view(np.uint16), g)
            amax = np.float32(np.max(np.abs(x)))
            t = np.float32(amax / np.float32(np.float32(6.0) * g32))
            if t >= 448:
                continue
            ref_s8 = int(torch.tensor([t]).to(torch.float8_e4m3fn).view(torch.uint8)[0])
            if ref_s8 == 0:
                assert s8 == 0 and not packed.any()
                continue
            assert s8 == ref_s8
            d = np.float32(np.float32(oracle.e4m3_value(s8)) * g32)
            y = (x / d).astype(np.float32)
            ref_codes = list(y.astype(mld.float4_e2m1fn).view(np.uint8) & 0xF)
            assert _nibbles(packed) == ref_codes


def test_grid_and_amax_invariants(oracle):
    """Dequantized values lie on +-grid * e4m3(s8) * g; every element is within
    half a grid step of its exact scaled value unless saturated; when s8 is a
    normal E4M3 number the block's amax element maps to +-6."""
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    xb = _random_blocks(3000, 12)
    g = 0.0021
    normal_hits = 0
    for row in xb:
        x = row.double().numpy()
        packed, s8 = oracle.quantize_block16(row.view(torch.int16).numpy().view(np.uint16), g)
        if s8 == 0:
            continue
        codes = _nibbles(packed)
        sv = oracle.e4m3_value(s8)
        d = sv * g
        for j in range(16):
            gv = abs(oracle.e2m1_value(codes[j]))
            assert gv in grid
            assert math.copysign(1.0, oracle.e2m1_value(codes[j])) == math.copysign(1.0, x[j])
            yj = abs(x[j]) / d
            if yj <= 6:
                k = int(np.searchsorted(grid, gv))
                lo = grid[k - 1] if k > 0 else grid[0]
                hi = grid[k + 1] if k + 1 < len(grid) else grid[-1]
                half = max(gv - lo, hi - gv) / 2
                assert abs(yj - gv) <= half * (1 + 1e-6) + 1e-12
        amax = np.max(np.abs(x))
        t = amax / (6 * g)
        if s8 >= 0x08 and t >= 2.0 ** -6:          # normal s8 (or saturated)
            normal_hits += 1
            jm = int(np.argmax(np.abs(x)))
            assert codes[jm] & 0x7 == 0x7
    assert normal_hits > 1000


def test_append_scatter_gather_identity(oracle):
    """Every written slot, read back through the page it was scattered to,
    equals the direct quantization of that token's rows; skipped tokens and
    untouched slots keep the 0xA5 sentinel."""
    H, D, ps, P, N = 3, 64, 16, 9, 100
    g = torch.Generator().manual_seed(5)
    k = torch.randn((N, H, D), generator=g).to(torch.bfloat16)
    v = torch.randn((N, H, D), generator=g).to(torch.bfloat16)
    perm = torch.randperm(P * ps, generator=g)[:N]
    slots = perm.clone().to(torch.int64)
    slots[torch.randperm(N, generator=g)[:7]] = -1
    cache = oracle.new_cache(P, H, ps, D)
    ks, vs = W.global_scale(k), W.global_scale(v)
    st = oracle.append(W.bits(k), W.bits(v), ks, vs, slots.numpy(), cache)
    assert st == 0
    written = np.zeros((P, ps), bool)
    kb, vb = W.bits(k), W.bits(v)
    for i in range(N):
        s = int(slots[i])
        if s < 0:
            continue
        page, off = divmod(s, ps)
        written[page, off] = True
        for h in range(H):
            for blk in range(D // 16):
                pk, sk = oracle.quantize_block16(kb[i, h, blk * 16:(blk + 1) * 16], ks)
                pv, sv = oracle.quantize_block16(vb[i, h, blk * 16:(blk + 1) * 16], vs)
                assert np.array_equal(cache["k_data"][page, h, off, blk * 8:(blk + 1) * 8], pk)
                assert np.array_equal(cache["v_data"][page, h, off, blk * 8:(blk + 1) * 8], pv)
                assert cache["k_sf"][page, h, off, blk] == sk
                assert cache["v_sf"][page, h, off, blk] == sv
    for name in ("k_data", "v_data", "k_sf", "v_sf"):
        arr = cache[name]
        untouched = arr.transpose(0, 2, 1, 3)[~written]
        assert np.all(untouched == 0xA5), name


@pytest.mark.parametrize("bad", [0.0, -0.0, -1.0, float("inf"), float("nan"), -float("inf")])
@pytest.mark.parametrize("which", ["k", "v", "both"])
def test_append_bad_scale_writes_nothing(oracle, bad, which):
    H, D, ps, P, N = 2, 32, 16, 2, 8
    k = torch.randn((N, H, D)).to(torch.bfloat16)
    v = torch.randn((N, H, D)).to(torch.bfloat16)
    slots = np.arange(N, dtype=np.int64)
    cache = oracle.new_cache(P, H, ps, D)
    ks = bad if which in ("k", "both") else 0.01
    vs = bad if which in ("v", "both") else 0.01
    st = oracle.append(W.bits(k), W.bits(v), ks, vs, slots, cache)
    want = (oracle.BAD_K_SCALE if which in ("k", "both") else 0) | \
           (oracle.BAD_V_SCALE if which in ("v", "both") else 0)
    assert st == want
    for name in ("k_data", "v_data", "k_sf", "v_sf"):
        assert np.all(cache[name] == 0xA5)


def test_append_subnormal_scale_is_valid(oracle):
    k = torch.randn((4, 1, 16)).to(torch.bfloat16)
    cache = oracle.new_cache(1, 1, 16, 16)
    st = oracle.append(W.bits(k), W.bits(k), 1e-42, 1e-42, np.arange(4, dtype=np.int64), cache)
    assert st == 0
    assert not np.all(cache["k_sf"][0, 0, :4] == 0xA5)


def test_append_slot_out_of_range_flagged(oracle):
    k = torch.randn((4, 1, 16)).to(torch.bfloat16)
    cache = oracle.new_cache(1, 1, 16, 16)
    slots = np.array([0, 16, 3, 1000], np.int64)
    st = oracle.append(W.bits(k), W.bits(k), 0.01, 0.01, slots, cache)
    assert st == oracle.SLOT_OOB
    assert cache["k_sf"][0, 0, 0] != 0xA5 and cache["k_sf"][0, 0, 3] != 0xA5
    assert np.all(cache["k_sf"][0, 0, [1, 2] + list(range(4, 16))] == 0xA5)


def test_config_append_workload_shape(oracle):
    """The append workload: 8192 tokens, exactly 410 skipped slots, every
    written slot distinct and inside the 512 x 16 slots."""
    d = W.make(W.spec("append"))
    s = d["slot_mapping"]
    assert int((s < 0).sum()) == 410
    w = s[s >= 0]
    assert len(torch.unique(w)) == w.numel() and int(w.max()) < 512 * 16
