"""Pins of the FP8 (E4M3) paged-KV oracle: each element is the E4M3 code of
the fp32 quotient x / g (OCP OFP8 E4M3 "FN": bias 7, 3 mantissa bits,
subnormal step 2^-9, largest finite 448, no infinities, S.1111.111 = NaN),
rounded to nearest even, saturating, sign kept."""
import numpy as np
import pytest

import workloads as W


def test_hand_worked_codes(oracle):
    q = oracle.fp8_quantize
    assert q(1.0, 1.0) == 0x38              # 1.0 = 2^0 * 1.000: exponent field 7
    assert q(2.0, 0.5) == 0x48              # 4.0: exponent field 9, code 9 << 3
    assert q(448.0, 1.0) == 0x7E            # largest finite
    assert q(500.0, 1.0) == 0x7E            # saturates
    assert q(-1e30, 1.0) == 0xFE
    assert q(0.0, 1.0) == 0x00
    assert q(-0.0, 1.0) == 0x80             # sign kept
    assert q(2.0 ** -9, 1.0) == 0x01        # smallest subnormal
    assert q(2.0 ** -10, 1.0) == 0x00       # half of it: tie, to the even code 0
    assert q(1.5 * 2.0 ** -10, 1.0) == 0x01
    assert q(1.0625, 1.0) == 0x38           # tie between 1.0 and 1.125: even mantissa
    assert q(1.1875, 1.0) == 0x3A           # tie between 1.125 and 1.25: even mantissa
    assert q(float("nan"), 1.0) == 0x7F
    assert q(3.0, 3.0) == 0x38              # the division comes first


def test_composition_with_the_pinned_encoder_over_all_bf16(oracle):
    """For every bf16 x and several g: the code is the bit-level E4M3 encoder
    (itself pinned against the exhaustive search) of numpy's fp32 quotient."""
    xs = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    xs = xs[~np.isnan(xs)]
    for g in [1.0, 0.0021, 3.7e-5, 7.5e30, 2.0 ** -60]:
        g32 = np.float32(g)
        with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
            t = (xs / g32).astype(np.float32)
        want = oracle.e4m3_encode_array(t, bit_level=True)
        got = np.array([oracle.fp8_quantize(float(x), float(g32)) for x in xs], np.uint8)
        assert np.array_equal(got, want), g


def test_round_trip_error_bound(oracle):
    rng = np.random.default_rng(3)
    g = 0.0123
    x = (rng.standard_normal(4000) * 3.0).astype(np.float32)
    x = x.astype(np.float32)
    for xi in x:
        t = abs(float(np.float32(xi) / np.float32(g)))
        if not (2.0 ** -6 <= t <= 448.0):
            continue
        back = oracle.e4m3_value(oracle.fp8_quantize(float(xi), g)) * float(np.float32(g))
        # half an ulp of a 3-bit mantissa, plus the quotient's fp32 rounding
        assert abs(back - float(xi)) <= (2.0 ** -4 + 2.0 ** -22) * abs(float(xi))


def test_fp8_append_scatter_and_failures(oracle):
    rng = np.random.default_rng(4)
    N, H, D, ps, P = 37, 2, 64, 16, 5
    k = W.bits(__import__("torch").from_numpy(rng.standard_normal((N, H, D)).astype(np.float32)).to(
        __import__("torch").bfloat16))
    v = W.bits(__import__("torch").from_numpy(rng.standard_normal((N, H, D)).astype(np.float32)).to(
        __import__("torch").bfloat16))
    slots = rng.permutation(P * ps)[:N].astype(np.int64)
    slots[3] = -1
    c = oracle.new_fp8_cache(P, H, ps, D)
    assert oracle.fp8_append(k, v, 0.01, 0.02, slots, c) == 0
    written = np.zeros((P, H, ps), bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        pg, off = divmod(int(s), ps)
        for h in range(H):
            written[pg, h, off] = True
            xk = (k[i, h].astype(np.uint32) << 16).view(np.float32)
            want = [oracle.fp8_quantize(float(x), 0.01) for x in xk]
            assert list(c["k_data"][pg, h, off]) == want
            back = oracle.fp8_dequant_row(c, "v", int(s), h, 0.02)
            xv = (v[i, h].astype(np.uint32) << 16).view(np.float32)
            assert np.all(np.abs(back - xv) <= 2.0 ** -4 * np.abs(xv) + 0.02 * 2.0 ** -10)
    assert np.all(c["k_data"][~written] == 0xA5) and np.all(c["v_data"][~written] == 0xA5)
    # out-of-range slot: skipped and flagged; bad scale: nothing written
    c2 = oracle.new_fp8_cache(P, H, ps, D)
    bad = slots.copy()
    bad[0] = P * ps
    assert oracle.fp8_append(k, v, 0.01, 0.02, bad, c2) == 4
    c3 = oracle.new_fp8_cache(P, H, ps, D)
    assert oracle.fp8_append(k, v, 0.0, 0.02, slots, c3) == 1
    assert np.all(c3["k_data"] == 0xA5) and np.all(c3["v_data"] == 0xA5)


def test_fp8_paged_attention_equals_dense_on_dequantized_kv(oracle):
    """The paged prefill over an FP8 cache equals dense causal attention on
    the dequantized K and V (gathered through the page table by hand)."""
    import torch
    rng = np.random.default_rng(6)
    L, H, D, ps = 50, 1, 64, 16
    P = 6
    kv = torch.from_numpy(rng.standard_normal((2, L, H, D)).astype(np.float32)).to(torch.bfloat16)
    q = torch.from_numpy(rng.standard_normal((L, 2, D)).astype(np.float32)).to(torch.bfloat16)
    pages = rng.permutation(P)[:4].astype(np.int32)
    slots = np.array([pages[i // ps] * ps + i % ps for i in range(L)], np.int64)
    c = oracle.new_fp8_cache(P, H, ps, D)
    assert oracle.fp8_append(W.bits(kv[0]), W.bits(kv[1]), 0.03, 0.05, slots, c) == 0
    ind = np.array([0, L], np.int32)
    out, lse = oracle.prefill(W.bits(q), ind, ind, pages.reshape(1, -1), c, 2, 0.03, 0.05, 0.125)
    kd = np.stack([oracle.fp8_dequant_row(c, "k", int(s), 0, 0.03) for s in slots])
    vd = np.stack([oracle.fp8_dequant_row(c, "v", int(s), 0, 0.05) for s in slots])
    qd = W.bits(q).astype(np.uint32)
    for h in range(2):
        qh = (qd[:, h] << 16).view(np.float32).astype(np.float64)
        o_ref, l_ref = oracle.dense_causal(qh, kd, vd, 0.125)
        np.testing.assert_allclose(out[h::2], o_ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[h::2], l_ref, rtol=0, atol=1e-12)
