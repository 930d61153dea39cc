"""GPU pins of the device building blocks, each against the CPU oracle or an
exact fp64 product: native conversions over all 2^32 fp32 inputs, the block
quantizer, the tile repack and the tcgen05 operand layouts."""
import time

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def diag():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_paged_kv_slot_b300.diag as d
    return d


def test_native_conversions_match_oracle_codec_exhaustively(diag, oracle):
    """All 2^32 fp32 bit patterns: cvt.rn.satfinite E4M3 and E2M1 codes equal
    the oracle's bit-level codec (itself pinned to brute force and libraries).
    NaN inputs are reported separately: the format leaves them unspecified."""
    chunk = 1 << 28
    e4 = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    e2 = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    nan_e2m1 = set()
    t0 = time.time()
    for c in range(1 << 4):
        first = c * chunk
        diag.codec_span(first, chunk, e4, e2)
        g4, g2 = e4.cpu().numpy(), e2.cpu().numpy()
        r4 = oracle.e4m3_encode_span(first, chunk)
        r2 = oracle.e2m1_encode_span(first, chunk)
        bits = np.arange(first, first + chunk, dtype=np.uint64).astype(np.uint32)
        is_nan = (bits & 0x7FFFFFFF) > 0x7F800000
        bad4 = (g4 != r4) & ~is_nan
        bad2 = (g2 != r2) & ~is_nan
        assert not bad4.any(), f"E4M3 mismatch at {bits[bad4][:8]}: {g4[bad4][:8]} vs {r4[bad4][:8]}"
        assert not bad2.any(), f"E2M1 mismatch at {bits[bad2][:8]}: {g2[bad2][:8]} vs {r2[bad2][:8]}"
        # NaN inputs: E4M3 gives a NaN code; record what E2M1 gives
        assert np.all((g4[is_nan] & 0x7F) == 0x7F)
        nan_e2m1 |= set(np.unique(g2[is_nan]).tolist())
    print(f"exhaustive codec check {time.time() - t0:.1f}s; E2M1 codes for NaN inputs: "
          f"{sorted(nan_e2m1)}")


def _golden_blocks():
    import pathlib
    rows = []
    for line in (pathlib.Path(__file__).parent / "golden" / "quant_block_cases.txt").read_text() \
            .splitlines():
        if line.startswith("case "):
            _, g, xs, s8, packed = [p.strip() for p in line[5:].split("|")]
            rows.append((float(g), [float(v) for v in xs.split()], int(s8, 16),
                         [int(b, 16) for b in packed.split()]))
    return rows


def test_block_quantizer_golden_cases(diag):
    for g, xs, s8, packed in _golden_blocks():
        x = torch.tensor(xs, dtype=torch.float32).to(torch.bfloat16).cuda()
        p = torch.empty(8, dtype=torch.uint8, device="cuda")
        s = torch.empty(1, dtype=torch.uint8, device="cuda")
        diag.quantize_blocks(x, g, p, s)
        assert int(s.item()) == s8 and p.cpu().tolist() == packed, (xs, g)


@pytest.mark.parametrize("g", [1.0, 0.0021, 3.7e-5, 1e-42, 7.5e30])
def test_block_quantizer_bit_exact_vs_oracle(diag, oracle, g):
    rng = np.random.default_rng(int(abs(np.log2(g))) + 3)
    n = 20000
    scale = np.exp2(rng.uniform(-20, 20, size=(n, 1)))
    x = (rng.standard_normal((n, 16)) * scale).astype(np.float32)
    x[rng.random((n, 16)) < 0.05] = 0.0
    x[rng.random((n, 16)) < 0.01] *= -0.0
    x[:50] = 0.0
    xb = torch.from_numpy(x).to(torch.bfloat16)
    p = torch.empty((n, 8), dtype=torch.uint8, device="cuda")
    s = torch.empty(n, dtype=torch.uint8, device="cuda")
    diag.quantize_blocks(xb.cuda(), g, p, s)
    gp, gs = p.cpu().numpy(), s.cpu().numpy()
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    for i in range(n):
        rp, rs = oracle.quantize_block16(bits[i], g)
        assert gs[i] == rs and np.array_equal(gp[i], rp), (i, x[i], g)


def test_markstein_division_matches_ieee_division(diag, oracle):
    """The append divides each element by its block's decode scale d with one
    rounded reciprocal and a fused-multiply-add correction (Markstein).  Over
    every bf16 input and divisors d = RN(e4m3(s8) * g) for all positive E4M3
    scales and many global scales g, plus log-uniform and edge divisors, the
    quotient must give the IEEE quotient's E2M1 code wherever the quantizer
    uses that path, and its exact bits wherever Markstein's theorem applies
    (|x| >= 2^-100, normal quotient).  The block scale amax / RN(6 g) is
    divided the same way for amax >= 2^-100: divisors RN(6 g) are included and
    the E4M3 code of the quotient is compared as well."""
    e4 = np.array([oracle.e4m3_value(c) for c in range(1, 127)], np.float32)
    rng = np.random.default_rng(11)
    gs = np.concatenate([[1.0, 0.0021, 3.7e-5, 1 / 2688.0, 1e-20, 7.5e30, 2.0 ** -60],
                         np.exp2(rng.uniform(-80, 80, 40))]).astype(np.float32)
    ds = (e4[None, :] * gs[:, None]).astype(np.float32).reshape(-1)   # RN(sv * g) in fp32
    extra = np.exp2(rng.uniform(-98, 100, 4000)).astype(np.float32)
    edges = np.array([2.0 ** -98, 2.0 ** 100, np.nextafter(np.float32(2.0 ** -98), np.float32(1)),
                      np.nextafter(np.float32(2.0 ** 100), np.float32(0)), 1.0, 3.0, 448.0],
                     np.float32)
    d6 = (np.float32(6.0) * gs).astype(np.float32)                      # RN(6 g)
    d = np.concatenate([ds, d6, extra, edges]).astype(np.float32)
    dv = torch.from_numpy(d).cuda()
    counts = torch.zeros(4, dtype=torch.int64, device="cuda")
    first = torch.zeros(2, dtype=torch.int32, device="cuda")
    diag.div_check(dv, counts, first)
    checked, bad_code, bad_bits, small_bits = counts.cpu().tolist()
    print(f"checked {checked}; bit differences with |x| < 2^-100 (same code): {small_bits}")
    # expected number of (x, d) pairs on the Markstein path, counted on the host
    xs = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    ax = np.sort(np.abs(xs[np.isfinite(xs)]))
    with np.errstate(over="ignore"):
        lim = (d * np.float32(2.0 ** 100)).astype(np.float32)
    ok = (d >= np.float32(2.0 ** -98)) & (d <= np.float32(2.0 ** 100))
    want = int(np.searchsorted(ax, lim[ok], side="right").sum())
    assert checked == want, (checked, want)
    assert bad_code == 0 and bad_bits == 0, (bad_code, bad_bits, first.cpu().tolist())


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("is_v", [False, True])
@pytest.mark.parametrize("valid", [128, 77])
def test_repack_exact(diag, oracle, head_dim, is_v, valid):
    rng = np.random.default_rng(head_dim + 2 * is_v + valid)
    codes = rng.integers(0, 256, size=128 * head_dim // 2, dtype=np.uint8)
    sf = rng.integers(0, 256, size=128 * head_dim // 16, dtype=np.uint8)
    sf[(sf & 0x7F) == 0x7F] = 0x38            # no NaN scales
    raw = torch.from_numpy(np.concatenate([codes, sf])).cuda()
    out = torch.empty((128, head_dim), dtype=torch.int16, device="cuda")
    diag.repack_tile(raw, head_dim, is_v, valid, out)
    got = out.cpu().view(torch.float16 if is_v else torch.bfloat16).double().numpy()
    e2 = np.array([oracle.e2m1_value(c) for c in range(16)])
    e4 = np.array([oracle.e4m3_value(c) for c in range(256)])
    c2 = codes.reshape(128, head_dim // 2)
    nib = np.stack([c2 & 0xF, c2 >> 4], -1).reshape(128, head_dim)
    want = e2[nib] * np.repeat(e4[sf.reshape(128, head_dim // 16)], 16, axis=1)
    want[valid:] = 0.0
    assert np.array_equal(got, want)


def _umma_inputs(mode, seed=0):
    g = torch.Generator().manual_seed(seed)
    dt = torch.bfloat16 if mode == 0 else torch.float16
    a = (torch.randn((128, 128), generator=g) * 0.5).to(dt)
    b = (torch.randn((128, 128), generator=g) * 0.5).to(dt)
    return a, b


@pytest.mark.parametrize("mode", [0, 1, 3])
def test_tcgen05_layouts(diag, mode):
    a, b = _umma_inputs(mode, seed=mode)
    c = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    diag.umma(mode, a.cuda(), b.cuda(), c, st)
    torch.cuda.synchronize()
    assert st.item() == 0
    want = (a.double() @ b.double().T) if mode == 0 else (a.double() @ b.double())
    err = (c.cpu().double() - want).abs().max().item()
    assert err < 1e-3, f"mode {mode}: max err {err}"


@pytest.mark.parametrize("mode", [0, 1])
def test_tcgen05_pair_mma_layouts(diag, mode):
    """The 2-CTA MMA (cta_group::2, M = 256) of the paired prefill: A split by
    rows between the CTAs, B split by N (K-major rows for S = Q K^T, MN-major
    columns for O = P V); each CTA's tensor memory holds its 128 rows of the
    exact product (fp64 reference)."""
    g = torch.Generator().manual_seed(10 + mode)
    dt = torch.bfloat16 if mode == 0 else torch.float16
    a = (torch.randn((256, 128), generator=g) * 0.5).to(dt)
    b = (torch.randn((128, 128), generator=g) * 0.5).to(dt)
    c = torch.empty((256, 128), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    addrs = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    diag.umma_pair(mode, a.cuda(), b.cuda(), c, st, addrs)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert addrs[0].item() == addrs[1].item(), addrs.tolist()
    want = (a.double() @ b.double().T) if mode == 0 else (a.double() @ b.double())
    err = (c.cpu().double() - want).abs().max().item()
    assert err < 1e-3, f"mode {mode}: max err {err}"
