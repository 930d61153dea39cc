"""Host planner (no GPU): max lengths, uniform flag, L2 gate and tile order.

Mirrors the pages' plan tests: FlashInfer PR #5043 analysis page ("plan() 함수
최적화"), test_batch_prefill_plan_max_lens over seq_lens of dtypes None / int32 /
uint32 and several batch and page sizes; and the scheduling rules of the PR
#3575 page (O(1) uniform decode, global reverse-Q-tile order, L2 gate).
"""
import itertools

import numpy as np
import pytest

import nvfp4_paged_kv_slot_b300 as fi

L2 = 126 * 2**20


def _lens(batch, seed, lo=1, hi=3000):
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi, size=batch)


@pytest.mark.parametrize("dtype", [None, np.int32, np.uint32, np.int64])
@pytest.mark.parametrize("batch", [1, 7, 64, 256, 1024])
@pytest.mark.parametrize("page_size", [16, 64])
def test_plan_max_lens(dtype, batch, page_size):
    kv = _lens(batch, batch)
    qo = np.minimum(kv, _lens(batch, batch + 1))
    if dtype is None:          # lengths given directly as indptr (no seq_lens)
        kv_ind = np.concatenate([[0], np.cumsum(kv)]).astype(np.int32)
    else:
        kv_ind = fi.indptr_from_lens(kv.astype(dtype))
    qo_ind = fi.indptr_from_lens(qo)
    info, _ = fi.fi_prefill_plan_host(qo_ind, kv_ind, 32, 8, 128, page_size, with_list=False)
    assert info["max_qo_len"] == int(qo.max())
    assert info["max_kv_len"] == int(kv.max())
    assert info["total_qo_len"] == int(qo.sum())
    assert info["total_kv_len"] == int(kv.sum())
    assert info["batch"] == batch


@pytest.mark.parametrize("cta_pairs", [0, 1])
def test_uniform_flag_and_o1_decode_orders(cta_pairs):
    B, L = 6, 300
    ind = fi.indptr_from_lens([L] * B)
    for schedule, global_rev in ((1, 1), (2, 0)):
        info, work = fi.fi_prefill_plan_host(ind, ind, 8, 2, 128, 16, schedule=schedule,
                                             cta_pairs=cta_pairs)
        assert info["is_uniform"] == 1 and info["global_reverse"] == global_rev
        q_tiles = (L + 127) // 128
        HU = info["head_units"]
        # G = 4: a unit is the whole group on a CTA pair, or two heads on one CTA
        assert info["heads_per_cta"] == 2
        assert info["ctas_per_unit"] == (2 if cta_pairs == 0 else 1)
        assert HU == (2 * 1 if cta_pairs == 0 else 2 * 2)
        assert info["num_units"] == B * HU * q_tiles == work.shape[0]
        # every (b, hu, qt) exactly once
        assert len({tuple(w[:3]) for w in work}) == work.shape[0]
        for t, (b, hu, qt, _) in enumerate(work):
            if global_rev:   # page formula: q-step from the end, head-major, batch fastest
                assert qt == q_tiles - 1 - t // (B * HU)
                assert hu == (t % (B * HU)) // B and b == (t % (B * HU)) % B
            else:
                assert b == t // (HU * q_tiles)
                assert qt == q_tiles - 1 - (t % (HU * q_tiles)) % q_tiles


@pytest.mark.parametrize("hq,hk,pairs,hu", [(4, 2, 1, 2 * 1), (8, 2, 2, 2 * 1), (16, 2, 2, 2 * 2),
                                             (6, 2, 1, 2 * 3), (2, 2, 1, 2 * 1)])
def test_cta_pair_decision(hq, hk, pairs, hu):
    """Groups of a multiple of 4 query heads run on CTA pairs (two heads per
    CTA); other groups on single CTAs (two heads per CTA if the group is even)."""
    ind = fi.indptr_from_lens([200, 300])
    info, work = fi.fi_prefill_plan_host(ind, ind, hq, hk, 128, 16)
    assert info["ctas_per_unit"] == pairs and info["head_units"] == hu
    assert info["num_units"] == work.shape[0] == hu * (2 + 3)
    assert info["num_ctas"] % pairs == 0
    if pairs == 2:
        off, _ = fi.fi_prefill_plan_host(ind, ind, hq, hk, 128, 16, cta_pairs=1)
        assert off["ctas_per_unit"] == 1 and off["head_units"] == 2 * hu


def test_uniform_check_is_totals_based():
    # lengths that are not all equal are never "uniform"
    qo = fi.indptr_from_lens([128, 128, 127])
    info, _ = fi.fi_prefill_plan_host(qo, qo, 4, 4, 64, 16, with_list=False)
    assert info["is_uniform"] == 0
    # equal qo but different kv -> not uniform either
    kv = fi.indptr_from_lens([128, 129, 128])
    qo = fi.indptr_from_lens([128, 128, 128])
    info, _ = fi.fi_prefill_plan_host(qo, kv, 4, 4, 64, 16, with_list=False)
    assert info["is_uniform"] == 0


def test_l2_gate():
    """Ragged batches: the global order only while 2 * kv_bytes <= L2.  Uniform
    batches take the global order at any size."""
    H_kv, D = 8, 128
    per_token = H_kv * 2 * (D // 2 + D // 16)        # NVFP4 K and V bytes per token
    fits = (L2 // 2) // per_token                    # 2 * kv_bytes <= L2
    ind = fi.indptr_from_lens([fits - 100, 100])
    info, _ = fi.fi_prefill_plan_host(ind, ind, 32, H_kv, D, 16, l2_bytes=L2, with_list=False)
    assert info["is_uniform"] == 0
    assert info["kv_bytes"] == fits * per_token and info["global_reverse"] == 1
    ind = fi.indptr_from_lens([fits - 99, 100])
    info, _ = fi.fi_prefill_plan_host(ind, ind, 32, H_kv, D, 16, l2_bytes=L2, with_list=False)
    assert info["global_reverse"] == 0
    for lens in ([fits + 1], [1024] * 1024):
        ind = fi.indptr_from_lens(lens)
        info, _ = fi.fi_prefill_plan_host(ind, ind, 32, H_kv, D, 16, l2_bytes=L2, with_list=False)
        assert info["is_uniform"] == 1 and 2 * info["kv_bytes"] > L2
        assert info["global_reverse"] == 1


def _n_kv(qt, qo, kv):
    last_row = min(qo, (qt + 1) * 128) - 1
    return (last_row + kv - qo) // 128 + 1


@pytest.mark.parametrize("schedule", [1, 2])
def test_ragged_work_list(schedule):
    qo = [1, 17, 128, 129, 300, 520, 0, 2000]
    kv = [1, 40, 128, 300, 300, 600, 5, 2100]
    qi, ki = fi.indptr_from_lens(qo), fi.indptr_from_lens(kv)
    info, work = fi.fi_prefill_plan_host(qi, ki, 8, 2, 128, 16, schedule=schedule)
    assert info["is_uniform"] == 0
    HU = info["head_units"]
    want = {(b, hu, qt) for b in range(len(qo)) for hu in range(HU)
            for qt in range((qo[b] + 127) // 128)}
    got = [tuple(w[:3]) for w in work]
    assert sorted(got) == sorted(want) and len(got) == len(want)
    for b, hu, qt, cost in work:
        assert cost == _n_kv(qt, qo[b], kv[b])
    # the head units of one (sequence, q-tile) are consecutive units, in order
    assert [int(w[1]) for w in work] == [t % HU for t in range(len(work))]
    items = [(int(w[0]), int(w[2]), int(w[3])) for w in work[::HU]]
    assert all(tuple(work[t, [0, 2, 3]]) == items[t // HU] for t in range(len(work)))
    if schedule == 1:   # global: heaviest first, ties in (sequence, q-tile) order
        assert items == sorted(items, key=lambda x: (-x[2], x[0], x[1]))
    else:               # per sequence (longest first, stable), q-tiles reversed
        order = sorted(range(len(qo)), key=lambda b: -kv[b])
        assert items == [(b, qt, _n_kv(qt, qo[b], kv[b])) for b in order
                         for qt in reversed(range((qo[b] + 127) // 128))]


@pytest.mark.parametrize("args,code", [
    (dict(qo=[0, 5], kv=[0, 4]), fi.FI_ERR_INVALID_ARGUMENT),        # qo_len > kv_len
    (dict(qo=[0, 5, 3], kv=[0, 5, 9]), fi.FI_ERR_INVALID_ARGUMENT),  # decreasing indptr
    (dict(qo=[1, 5], kv=[1, 5]), fi.FI_ERR_INVALID_ARGUMENT),        # indptr not from 0
    (dict(hq=6, hk=4), fi.FI_ERR_INVALID_ARGUMENT),                  # H_q % H_kv != 0
    (dict(d=96), fi.FI_ERR_UNSUPPORTED),
    (dict(ps=8), fi.FI_ERR_UNSUPPORTED),
])
def test_plan_rejects(args, code):
    qo = args.get("qo", [0, 4])
    kv = args.get("kv", [0, 4])
    with pytest.raises(fi.FiError) as e:
        fi.fi_prefill_plan_host(qo, kv, args.get("hq", 4), args.get("hk", 2), args.get("d", 64),
                                args.get("ps", 16))
    assert e.value.status == code


def test_uint32_lengths_converted():
    lens = np.array([5, 4000, 17], dtype=np.uint32)
    ind = fi.indptr_from_lens(lens)
    assert ind.dtype == np.int32 and list(ind) == [0, 5, 4005, 4022]
    with pytest.raises(ValueError):
        fi.indptr_from_lens(np.array([2**31], dtype=np.uint32))


def test_workload_shapes():
    import workloads as W
    info, _ = fi.fi_prefill_plan_host(*([fi.indptr_from_lens(W.spec("uniform").seq_lens)] * 2),
                                      32, 8, 128, 16, with_list=False)
    # 1.2 GB of KV does not fit in L2, but a uniform batch takes the global order
    assert info["is_uniform"] == 1 and info["global_reverse"] == 1
    # G = 4: one unit per (sequence, kv head, q-tile), on a CTA pair
    assert info["ctas_per_unit"] == 2 and info["num_units"] == 1024 * 8 * 8
    sp = W.spec("single")
    ind = fi.indptr_from_lens(sp.seq_lens)
    info, _ = fi.fi_prefill_plan_host(ind, ind, 32, 8, 128, 16, with_list=False)
    assert info["global_reverse"] == 1                                 # 2.4 MB KV fits in L2
    sp = W.spec("ragged")
    assert len(sp.seq_lens) == 256 and min(sp.seq_lens) >= 128 and max(sp.seq_lens) <= 16384
    ind = fi.indptr_from_lens(sp.seq_lens)
    info, _ = fi.fi_prefill_plan_host(ind, ind, 32, 8, 128, 16, with_list=False)
    assert info["is_uniform"] == 0 and info["global_reverse"] == 0    # ragged: the L2 gate


def test_balanced_schedule_for_few_units():
    """A plan with fewer than 16 units per CTA slot assigns units heaviest
    first to the least-loaded slot.  One 2048-token sequence with 32/8 heads
    has 128 pair units of 1..16 KV tiles over 74 pair slots: dealt round-robin
    from a heaviest-first list the first slot would get 16 + 7 tiles; the
    greedy rule keeps every slot within one unit of the average load."""
    ind = fi.indptr_from_lens([2048])
    info, work = fi.fi_prefill_plan_host(ind, ind, 32, 8, 128, 16)
    assert info["num_units"] == 128 and info["ctas_per_unit"] == 2
    assert info["balanced"] == 1
    slots = info["num_ctas"] // info["ctas_per_unit"]
    # a unit's cost: its KV tiles (q-tile index + 1 for a square causal tile
    # grid) plus one for its Q load and epilogue
    costs = [int(w[2]) + 1 + 1 for w in work]
    avg = sum(costs) / slots
    # Graham's bound for the greedy rule on a heaviest-first list
    assert max(costs) <= info["max_slot_tiles"] <= avg + max(costs)
    assert info["max_slot_tiles"] <= 18
    # many units per slot: round-robin, no assignment
    big = fi.indptr_from_lens([1024] * 64)
    info2, _ = fi.fi_prefill_plan_host(big, big, 32, 8, 128, 16, with_list=False)
    assert info2["balanced"] == 0 and info2["max_slot_tiles"] == 0


def test_balanced_ragged_plan_bounds():
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 1500, size=6)]
    ind = fi.indptr_from_lens(lens)
    info, work = fi.fi_prefill_plan_host(ind, ind, 8, 2, 128, 16)
    assert info["balanced"] == 1
    slots = info["num_ctas"] // info["ctas_per_unit"]
    costs = [int(w[3]) + 1 for w in work]
    assert max(costs) <= info["max_slot_tiles"] <= sum(costs) / slots + max(costs)


# ---------------------------------------------------------------- decode plans
# The decode plan of the PR #5043 page (max_kv_len from one reduction over the
# lengths) with this library's split: the keys of all (sequence, KV head)
# pairs in 32-key steps, laid end to end and cut evenly over W warps (the warps
# the kernel keeps resident: 16 per SM up to 8 rows, 12 up to 16, 8 above; at
# least 8 steps a warp); one piece per pair a warp touches, consecutive partial
# slots and one merge for a pair cut into several pieces.

def _decode_plan(qo_lens, kv_lens, hq, hk, num_sms=148, d=128, ps=16):
    return fi.fi_decode_plan_host(fi.indptr_from_lens(qo_lens), fi.indptr_from_lens(kv_lens),
                                  hq, hk, d, ps, num_sms=num_sms)


def _expected_split(qo_lens, kv_lens, hk, warps_per_sm, num_sms):
    """The split by brute force: the owner warp of every step, then the pieces
    as maximal runs of one owner within a pair."""
    pairs = [(b, h, -(-kv_lens[b] // 32)) for b in range(len(kv_lens)) if qo_lens[b] > 0
             for h in range(hk)]
    total = sum(n for _, _, n in pairs)
    warps = 0 if total == 0 else max(1, min(num_sms * warps_per_sm, -(-total // 8)))
    owner = [w for w in range(warps) for _ in range(w * total // warps, (w + 1) * total // warps)]
    assert len(owner) == total
    pieces, merges, slot, s = [], [], 0, 0
    for b, h, n in pairs:
        runs = [(w, [i for i, _ in grp]) for w, grp in
                itertools.groupby(enumerate(owner[s:s + n]), key=lambda x: x[1])]
        first = slot
        for w, steps in runs:
            pslot = -1
            if len(runs) > 1:
                pslot, slot = slot, slot + 1
            pieces.append((w, [b * hk + h, steps[0] * 32, min((steps[-1] + 1) * 32, kv_lens[b]),
                               pslot]))
        if len(runs) > 1:
            merges.append([b, h, first, len(runs)])
        s += n
    return warps, pieces, merges


def _check_decode_split(qo_lens, kv_lens, hk, warps_per_sm, num_sms, plan):
    info, warps, units, merges, off = plan
    want_warps, pieces, want_merges = _expected_split(qo_lens, kv_lens, hk, warps_per_sm, num_sms)
    assert warps == want_warps and info["num_ctas"] == -(-warps // 4)
    assert units.tolist() == [p for _, p in pieces]
    assert merges.tolist() == want_merges
    assert off.tolist() == [sum(1 for w, _ in pieces if w < k) for k in range(warps + 1)]


def test_decode_plan_of_the_decode_workload():
    import workloads as W
    sp = W.spec("decode")
    plan = _decode_plan(sp.qo_lens, sp.seq_lens, 32, 8)
    info, warps, units, merges, off = plan
    # 128 x 8 pairs of 128 steps = 131072 steps over 148 SMs x 16 warps: 55 or
    # 56 steps a warp; every pair is cut into 3 or 4 pieces and merged
    assert warps == 2368 and merges.shape == (1024, 4)
    steps = [sum(-(-(u[2] - u[1]) // 32) for u in units[off[w]:off[w + 1]]) for w in range(warps)]
    assert min(steps) == 55 and max(steps) == 56
    assert set(merges[:, 3].tolist()) <= {3, 4}
    assert info["max_qo_len"] == 1 and info["max_kv_len"] == 4096 and info["is_uniform"] == 1
    _check_decode_split(sp.qo_lens, sp.seq_lens, 8, 16, 148, plan)


@pytest.mark.parametrize("num_sms,want_warps", [(148, 43), (1, 16), (200000, 43)])
def test_decode_warps_are_resident_and_take_at_least_8_steps(num_sms, want_warps):
    # G = 4, 2 query tokens: 8 rows, 16 warps per SM; (4 + 10 + 157) x 2 = 342 steps
    qo, kv = [1, 1, 2], [100, 300, 5000]
    plan = _decode_plan(qo, kv, 8, 2, num_sms=num_sms)
    assert plan[1] == want_warps
    _check_decode_split(qo, kv, 2, 16, num_sms, plan)


@pytest.mark.parametrize("hq,qo_len,warps_per_sm", [(12, 2, 12), (16, 3, 8), (8, 1, 16)])
def test_decode_warps_per_sm_follow_the_rows(hq, qo_len, warps_per_sm):
    # rows G * qo_len with 2 KV heads: 6 * 2 = 12, 8 * 3 = 24, 4 * 1 = 4
    qo, kv = [qo_len] * 64, [3000] * 64
    plan = _decode_plan(qo, kv, hq, 2, num_sms=2)
    assert plan[1] == 2 * warps_per_sm
    _check_decode_split(qo, kv, 2, warps_per_sm, 2, plan)


def test_decode_plan_of_one_short_sequence():
    # one step: one warp, one piece written directly, nothing to merge
    plan = _decode_plan([1], [5], 8, 1)
    info, warps, units, merges, off = plan
    assert warps == 1 and units.tolist() == [[0, 0, 5, -1]] and merges.shape[0] == 0
    assert off.tolist() == [0, 1]


def test_decode_plan_skips_sequences_without_queries():
    qo, kv = [0, 2, 0, 1], [50, 700, 9, 3000]
    plan = _decode_plan(qo, kv, 4, 2)
    assert set((plan[2][:, 0] // 2).tolist()) == {1, 3}
    _check_decode_split(qo, kv, 2, 16, 148, plan)


@pytest.mark.parametrize("args,code", [
    (dict(qo=[9], kv=[20]), fi.FI_ERR_UNSUPPORTED),           # more than 8 query tokens
    (dict(qo=[5], kv=[20], hq=32, hk=4), fi.FI_ERR_UNSUPPORTED),  # G * qo_len = 40 > 32 rows
    (dict(qo=[5], kv=[4]), fi.FI_ERR_INVALID_ARGUMENT),      # qo_len > kv_len
    (dict(d=96), fi.FI_ERR_UNSUPPORTED),
    (dict(ps=8), fi.FI_ERR_UNSUPPORTED),
    (dict(num_sms=0), fi.FI_ERR_INVALID_ARGUMENT),
])
def test_decode_plan_rejects(args, code):
    with pytest.raises(fi.FiError) as e:
        _decode_plan(args.get("qo", [1]), args.get("kv", [16]), args.get("hq", 8),
                     args.get("hk", 2), num_sms=args.get("num_sms", 148), d=args.get("d", 128),
                     ps=args.get("ps", 16))
    assert e.value.status == code


def test_fp8_plan_counts_one_byte_per_element_in_the_l2_gate():
    # a ragged batch of 20 sequences of about 2000 tokens, H_kv = 8, D = 128:
    # the NVFP4 K+V bytes (72 per token and head and tensor) fit the gate
    # 2 kv_bytes <= L2, the FP8 bytes (128) do not
    ind = fi.indptr_from_lens([2000] * 19 + [2001])
    tokens = 40001
    nv, _ = fi.fi_prefill_plan_host(ind, ind, 32, 8, 128, 16, l2_bytes=L2, with_list=False)
    f8, _ = fi.fi_prefill_plan_host(ind, ind, 32, 8, 128, 16, l2_bytes=L2, with_list=False,
                                    kv_format=1)
    assert nv["kv_bytes"] == tokens * 8 * 2 * (64 + 8)
    assert f8["kv_bytes"] == tokens * 8 * 2 * 128
    assert 2 * nv["kv_bytes"] <= L2 < 2 * f8["kv_bytes"]
    assert nv["global_reverse"] == 1 and f8["global_reverse"] == 0
    # everything else about the plan is the same
    for k in ("num_units", "q_tiles", "head_units", "ctas_per_unit", "is_uniform"):
        assert nv[k] == f8[k]


def test_plan_rejects_unknown_kv_format():
    with pytest.raises(fi.FiError) as e:
        fi.fi_prefill_plan_host([0, 4], [0, 4], 4, 2, 64, 16, kv_format=2)
    assert e.value.status == fi.FI_ERR_INVALID_ARGUMENT
