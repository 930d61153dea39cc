// planner.cpp — host planning of the causal batched prefill.
//
// Follows two analysis pages:
//  * FlashInfer PR #5043, "FlashInfer의 plan() 함수 최적화: Python max()에서
//    Tensor.max()로의 전환": max_qo_len / max_kv_len come from one reduction over
//    the int32 length arrays (no per-element Python loop, lengths as int32).
//  * FlashInfer PR #3575, "FlashInfer FP8 Causal Attention 최적화: O(1) 디코딩과
//    글로벌 스케줄링의 힘": §1 the uniform-length flag (checked cheaply as
//    total == batch * max, as in the page's reviewer section) that lets the
//    kernel decode tile -> (batch, head, q-tile) arithmetically; §2 global
//    reverse-Q-tile order (the heaviest causal q-tiles of every sequence and
//    head first); §3 the L2 gate (global order only if 2 * KV bytes fit in L2).
// Ragged batches get an explicit work list in the same spirit: heaviest first.
// Plans with few units per persistent CTA (or CTA pair) are balanced: each
// unit, heaviest first, goes to the least-loaded slot (the longest-processing-
// time-first rule), since dealing a handful of units round-robin leaves some
// slots with twice the average work.
#include <algorithm>
#include <cstring>
#include <functional>
#include <numeric>
#include <queue>

#include "internal.h"

namespace fi {

namespace {

inline int32_t n_kv_tiles(int32_t qt, int32_t qo_len, int32_t kv_len) {
  // last query row of the tile, and the last key it may see
  const int32_t last_row = std::min(qo_len, (qt + 1) * kTileQ) - 1;
  const int32_t last_key = last_row + (kv_len - qo_len);
  return last_key / kTileKV + 1;
}

// Resets a plan for re-planning but keeps the capacity of its lists: a plan
// object re-planned every step then allocates (and faults in) no memory once
// its lists have reached their size.
void reset_plan(HostPlan& P) {
  std::vector<int32_t> keep[6] = {std::move(P.work),       std::move(P.slot_units),
                                  std::move(P.slot_begin), std::move(P.dec_units),
                                  std::move(P.dec_merges), std::move(P.dec_warp_off)};
  P = HostPlan{};
  std::vector<int32_t>* dst[6] = {&P.work,      &P.slot_units, &P.slot_begin,
                                  &P.dec_units, &P.dec_merges, &P.dec_warp_off};
  for (int i = 0; i < 6; ++i) {
    // the work list keeps its contents: every plan resizes it and writes all
    // of its entries, or clears it (no zero fill of a list about to be written)
    if (i > 0) keep[i].clear();
    *dst[i] = std::move(keep[i]);
  }
}

// Plans with fewer units than this per slot are balanced.
constexpr int64_t kBalanceUnitsPerSlot = 16;

// (sequence, head unit, q-tile, KV tiles) of unit t: the arithmetic decoding
// of uniform batches ([#3575] §1, §2), or item t / head_units of the list.
void unit_entry(const HostPlan& P, int64_t t, int32_t* e) {
  const fi_plan_info& I = P.info;
  const int64_t HU = I.head_units;
  if (I.is_uniform) {
    const int64_t B = I.batch;
    int64_t b, hu, qt;
    if (I.global_reverse) {
      qt = I.q_tiles - 1 - t / (B * HU);
      const int64_t r = t % (B * HU);
      hu = r / B;
      b = r % B;
    } else {
      b = t / (HU * I.q_tiles);
      const int64_t r = t % (HU * I.q_tiles);
      hu = r / I.q_tiles;
      qt = I.q_tiles - 1 - r % I.q_tiles;
    }
    e[0] = static_cast<int32_t>(b);
    e[1] = static_cast<int32_t>(hu);
    e[2] = static_cast<int32_t>(qt);
    e[3] = n_kv_tiles(static_cast<int32_t>(qt), P.uniform_qo_len, P.uniform_kv_len);
  } else {
    const int32_t* item = P.work.data() + 4 * (t / HU);
    e[0] = item[0];
    e[1] = static_cast<int32_t>(t % HU);
    e[2] = item[1];
    e[3] = item[2];
  }
}

// Longest-processing-time-first assignment of the plan's units to `slots`
// slots; a unit costs its KV tiles plus one for its Q load and epilogue.
void balance(int32_t slots, HostPlan& P) {
  const int64_t n = P.info.num_units;
  std::vector<int32_t> cost(static_cast<size_t>(n));
  for (int64_t t = 0; t < n; ++t) {
    int32_t e[4];
    unit_entry(P, t, e);
    cost[t] = e[3] + 1;
  }
  std::vector<int32_t> order(static_cast<size_t>(n));
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t x, int32_t y) { return cost[x] > cost[y]; });
  using Load = std::pair<int64_t, int32_t>;  // (load, slot): ties go to the lower slot
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int32_t k = 0; k < slots; ++k) heap.push({0, k});
  std::vector<int32_t> owner(static_cast<size_t>(n));
  int64_t max_load = 0;
  for (int32_t t : order) {
    const Load top = heap.top();
    heap.pop();
    owner[t] = top.second;
    heap.push({top.first + cost[t], top.second});
    max_load = std::max(max_load, top.first + cost[t]);
  }
  P.info.balanced = 1;
  P.info.max_slot_tiles = static_cast<int32_t>(std::min<int64_t>(max_load, 0x7FFFFFFF));
  P.slot_begin.assign(static_cast<size_t>(slots) + 1, 0);
  for (int32_t t : order) ++P.slot_begin[owner[t] + 1];
  for (int32_t k = 0; k < slots; ++k) P.slot_begin[k + 1] += P.slot_begin[k];
  P.slot_units.assign(static_cast<size_t>(n), 0);
  std::vector<int32_t> fill(P.slot_begin.begin(), P.slot_begin.end() - 1);
  for (int32_t t : order) P.slot_units[fill[owner[t]]++] = t;  // heaviest first per slot
}

}  // namespace

fi_status plan_host(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, float sm_scale, int64_t l2_bytes, int32_t default_ctas,
                    const fi_plan_options* opts, HostPlan* out) {
  if (!out || batch < 0 || (batch > 0 && (!qo_indptr || !kv_indptr)))
    return FI_ERR_INVALID_ARGUMENT;
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return FI_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return FI_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return FI_ERR_UNSUPPORTED;
  const int32_t schedule = opts ? opts->schedule : 0;
  if (schedule < 0 || schedule > 2) return FI_ERR_INVALID_ARGUMENT;
  if (opts && (opts->cta_pairs < 0 || opts->cta_pairs > 1)) return FI_ERR_INVALID_ARGUMENT;
  if (opts && (opts->kv_format < 0 || opts->kv_format > 1)) return FI_ERR_INVALID_ARGUMENT;
  if (opts && opts->num_ctas < 0) return FI_ERR_INVALID_ARGUMENT;
  if (batch > 0 && (qo_indptr[0] != 0 || kv_indptr[0] != 0)) return FI_ERR_INVALID_ARGUMENT;

  HostPlan& P = *out;
  reset_plan(P);
  P.num_qo_heads = num_qo_heads;
  P.num_kv_heads = num_kv_heads;
  P.head_dim = head_dim;
  P.page_size = page_size;
  P.group = num_qo_heads / num_kv_heads;
  P.sm_scale = sm_scale;
  P.kv_format = opts ? opts->kv_format : 0;

  // One pass: the maxima, and the validity of every length.
  int32_t max_qo = 0, max_kv = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t qo = qo_indptr[b + 1] - qo_indptr[b];
    const int32_t kv = kv_indptr[b + 1] - kv_indptr[b];
    if (qo < 0 || kv < 0 || qo > kv) return FI_ERR_INVALID_ARGUMENT;
    max_qo = std::max(max_qo, qo);
    max_kv = std::max(max_kv, kv);
  }
  fi_plan_info& I = P.info;
  I.batch = batch;
  I.max_qo_len = max_qo;
  I.max_kv_len = max_kv;
  I.total_qo_len = batch > 0 ? qo_indptr[batch] : 0;
  I.total_kv_len = batch > 0 ? kv_indptr[batch] : 0;
  // every length equals the maximum iff the totals are batch * maximum
  I.is_uniform = (I.total_qo_len == static_cast<int64_t>(batch) * max_qo &&
                  I.total_kv_len == static_cast<int64_t>(batch) * max_kv)
                     ? 1
                     : 0;
  I.heads_per_cta = (P.group % 2 == 0) ? 2 : 1;
  // Groups of a multiple of 4 query heads run on CTA pairs (2 heads each)
  // that share their KV staging tiles, unless the options ask otherwise.
  P.pair = (P.group % 4 == 0) && !(opts && opts->cta_pairs == 1);
  I.ctas_per_unit = P.pair ? 2 : 1;
  P.units_per_kv_head = P.group / (I.heads_per_cta * I.ctas_per_unit);
  I.head_units = num_kv_heads * P.units_per_kv_head;
  I.q_tiles = (max_qo + kTileQ - 1) / kTileQ;
  // K and V bytes per token and head: NVFP4 codes and scales, or one FP8 byte
  // per element ([#3575] §3: the gate counts bytes_per_elt)
  const int64_t row_bytes = P.kv_format == 1 ? head_dim : head_dim / 2 + head_dim / 16;
  I.kv_bytes = I.total_kv_len * num_kv_heads * 2 * row_bytes;
  if (schedule == 1) {
    I.global_reverse = 1;
  } else if (schedule == 2) {
    I.global_reverse = 0;
  } else {
    // [#3575] §3's gate (the global order only when the KV cache fits in half
    // of L2) decides for ragged batches.  Uniform batches always take the
    // global order: all units of a q-step cost the same, so the persistent
    // CTAs run balanced waves, and the KV re-reads from HBM that the gate
    // guards against are cheap for this kernel (a KV tile feeds 4 heads x 128
    // rows of MMAs: even with every tile read from HBM the prefill needs under
    // a tenth of the HBM bandwidth).  Measured on the 1024 x 1024 batch (1.2 GB
    // of KV): 811 TFLOP/s in the global order against 757 in the per-(sequence,
    // head) one; on the ragged batch the gate's choice wins (1086 against 1065).
    I.global_reverse = (I.is_uniform || 2 * I.kv_bytes <= l2_bytes) ? 1 : 0;
  }

  const int32_t HU = I.head_units;
  const int32_t ctas = (opts && opts->num_ctas > 0) ? opts->num_ctas : default_ctas;
  if (I.is_uniform) {
    // no list: the kernel decodes uniform units arithmetically
    P.uniform_qo_len = max_qo;
    P.uniform_kv_len = max_kv;
    I.num_units = static_cast<int64_t>(batch) * HU * I.q_tiles;
    P.work.clear();
  } else {
    // Ragged: one item per (sequence, q-tile) with its cost in KV tiles,
    // written straight into the list in the kernel's order; the head units of
    // an item are consecutive units.
    int64_t items = 0;
    for (int32_t b = 0; b < batch; ++b)
      items += (qo_indptr[b + 1] - qo_indptr[b] + kTileQ - 1) / kTileQ;
    I.num_units = items * HU;
    P.work.resize(static_cast<size_t>(items) * 4);
    int32_t* w = P.work.data();
    auto put = [](int32_t* e, int32_t b, int32_t qt, int32_t cost) {
      e[0] = b;
      e[1] = qt;
      e[2] = cost;
      e[3] = 0;
    };
    if (I.global_reverse) {
      // Heaviest q-tiles of all sequences first (ties in sequence, then
      // q-tile order).  The costs are small integers, so a stable counting
      // sort by cost (descending) puts every item in place in two passes.
      const int32_t max_cost = max_kv / kTileKV + 1;
      std::vector<int64_t> pos(static_cast<size_t>(max_cost) + 2, 0);
      for (int32_t b = 0; b < batch; ++b) {
        const int32_t qo = qo_indptr[b + 1] - qo_indptr[b];
        const int32_t kv = kv_indptr[b + 1] - kv_indptr[b];
        const int32_t tiles = (qo + kTileQ - 1) / kTileQ;
        for (int32_t qt = 0; qt < tiles; ++qt) ++pos[n_kv_tiles(qt, qo, kv)];
      }
      int64_t acc = 0;  // first position of each cost, highest cost first
      for (int32_t c = max_cost + 1; c >= 0; --c) {
        const int64_t cnt = pos[c];
        pos[c] = acc;
        acc += cnt;
      }
      for (int32_t b = 0; b < batch; ++b) {
        const int32_t qo = qo_indptr[b + 1] - qo_indptr[b];
        const int32_t kv = kv_indptr[b + 1] - kv_indptr[b];
        const int32_t tiles = (qo + kTileQ - 1) / kTileQ;
        for (int32_t qt = 0; qt < tiles; ++qt) {
          const int32_t cost = n_kv_tiles(qt, qo, kv);
          put(w + 4 * pos[cost]++, b, qt, cost);
        }
      }
    } else {
      // per sequence, q-tiles from the last (heaviest) to the first, all head
      // units of a q-tile together; sequences longest first so the longest
      // chains start early
      std::vector<int32_t> order(batch);
      std::iota(order.begin(), order.end(), 0);
      std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) {
        return (kv_indptr[x + 1] - kv_indptr[x]) > (kv_indptr[y + 1] - kv_indptr[y]);
      });
      for (int32_t b : order) {
        const int32_t qo = qo_indptr[b + 1] - qo_indptr[b];
        const int32_t kv = kv_indptr[b + 1] - kv_indptr[b];
        const int32_t tiles = (qo + kTileQ - 1) / kTileQ;
        for (int32_t qt = tiles - 1; qt >= 0; --qt, w += 4) put(w, b, qt, n_kv_tiles(qt, qo, kv));
      }
    }
  }
  I.num_ctas = static_cast<int32_t>(std::min<int64_t>(I.num_units * I.ctas_per_unit,
                                                      std::max(ctas, I.ctas_per_unit)));
  if (P.pair) I.num_ctas &= ~1;
  const int32_t slots = I.num_ctas / I.ctas_per_unit;
  if (slots > 0 && I.num_units > 0 && I.num_units < kBalanceUnitsPerSlot * slots)
    balance(slots, P);
  return FI_OK;
}

// Decode plan ([#5043] decode.py: max_kv_len from one reduction over the
// lengths).  The keys of all (sequence, KV head) pairs are split evenly over
// the warps the decode kernel keeps resident (below); a pair split over
// several warps gets one partial slot per piece and one merge.
fi_status plan_decode_host(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                           int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t page_size, float sm_scale, int32_t num_sms, HostPlan* out) {
  if (!out || batch < 0 || (batch > 0 && (!qo_indptr || !kv_indptr)))
    return FI_ERR_INVALID_ARGUMENT;
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return FI_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return FI_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return FI_ERR_UNSUPPORTED;
  if (batch > 0 && (qo_indptr[0] != 0 || kv_indptr[0] != 0)) return FI_ERR_INVALID_ARGUMENT;
  HostPlan& P = *out;
  reset_plan(P);
  P.decode = true;
  P.num_qo_heads = num_qo_heads;
  P.num_kv_heads = num_kv_heads;
  P.head_dim = head_dim;
  P.page_size = page_size;
  P.group = num_qo_heads / num_kv_heads;
  P.sm_scale = sm_scale;
  int32_t max_qo = 0, max_kv = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t qo = qo_indptr[b + 1] - qo_indptr[b];
    const int32_t kv = kv_indptr[b + 1] - kv_indptr[b];
    if (qo < 0 || kv < 0 || qo > kv) return FI_ERR_INVALID_ARGUMENT;
    max_qo = std::max(max_qo, qo);
    max_kv = std::max(max_kv, kv);
  }
  if (max_qo > kDecodeMaxQo || P.group * max_qo > kDecodeMaxRows) return FI_ERR_UNSUPPORTED;
  fi_plan_info& I = P.info;
  I.batch = batch;
  I.max_qo_len = max_qo;
  I.max_kv_len = max_kv;
  I.total_qo_len = batch > 0 ? qo_indptr[batch] : 0;
  I.total_kv_len = batch > 0 ? kv_indptr[batch] : 0;
  I.is_uniform = (I.total_qo_len == static_cast<int64_t>(batch) * max_qo &&
                  I.total_kv_len == static_cast<int64_t>(batch) * max_kv)
                     ? 1
                     : 0;
  I.heads_per_cta = P.group;
  I.head_units = num_kv_heads;
  I.ctas_per_unit = 1;
  I.kv_bytes = I.total_kv_len * num_kv_heads * 2 * (head_dim / 2 + head_dim / 16);
  P.dec_rows = std::max(1, P.group * max_qo);
  // Balanced split: the keys of every (sequence, KV head) pair with queries,
  // in steps of kDecodeStep keys, laid end to end in (sequence, head) order
  // and cut into W runs of equal length (to one step), one per warp.  A run
  // that crosses pairs becomes one piece per pair; a pair cut into several
  // pieces gets one partial slot per piece (consecutive) and one merge item.
  if (static_cast<int64_t>(batch) * num_kv_heads > 0x7FFFFFFF) return FI_ERR_UNSUPPORTED;
  int64_t total = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t qo = qo_indptr[b + 1] - qo_indptr[b];
    const int32_t kv = kv_indptr[b + 1] - kv_indptr[b];
    if (qo > 0)
      total += static_cast<int64_t>(num_kv_heads) * ((kv + kDecodeStep - 1) / kDecodeStep);
  }
  const int64_t resident = static_cast<int64_t>(num_sms) * decode_warps_per_sm(P.dec_rows);
  const int64_t W =
      total == 0 ? 0
                 : std::max<int64_t>(1, std::min(resident, (total + kDecodeMinSteps - 1) /
                                                                kDecodeMinSteps));
  // warp w's first step is floor(w * total / W): the W + 1 boundaries, by
  // exact integer steps without a division per warp
  std::vector<int64_t> bnd(static_cast<size_t>(W) + 2, total);
  {
    const int64_t q = W > 0 ? total / W : 0, r = W > 0 ? total % W : 0;
    int64_t f = 0, rem = 0;
    for (int64_t k = 0; k <= W; ++k) {
      bnd[k] = f;
      f += q;
      rem += r;
      if (rem >= W) {
        ++f;
        rem -= W;
      }
    }
  }
  auto first_step = [&](int64_t w) { return bnd[static_cast<size_t>(w)]; };
  P.dec_warp_off.assign(static_cast<size_t>(W) + 1, 0);
  P.dec_units.reserve(static_cast<size_t>(4 * (W + static_cast<int64_t>(batch) * num_kv_heads)));
  int64_t s0 = 0, w = 0, slots = 0, pieces = 0;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t qo = qo_indptr[b + 1] - qo_indptr[b];
    const int32_t kv = kv_indptr[b + 1] - kv_indptr[b];
    if (qo == 0) continue;
    const int64_t n = (kv + kDecodeStep - 1) / kDecodeStep;  // >= 1: kv >= qo > 0
    for (int32_t hk = 0; hk < num_kv_heads; ++hk) {
      const int64_t pe = s0 + n;
      int64_t wl = w;  // the warp that takes the pair's last step
      while (first_step(wl + 1) <= pe - 1) ++wl;
      const bool split = wl > w;
      const int64_t first_slot = slots;
      for (int64_t st = s0; st < pe;) {
        const int64_t end = std::min(pe, first_step(w + 1));
        P.dec_units.push_back(b * num_kv_heads + hk);
        P.dec_units.push_back(static_cast<int32_t>((st - s0) * kDecodeStep));
        P.dec_units.push_back(
            static_cast<int32_t>(std::min<int64_t>((end - s0) * kDecodeStep, kv)));
        P.dec_units.push_back(split ? static_cast<int32_t>(slots++) : -1);
        ++pieces;
        if (end == first_step(w + 1)) P.dec_warp_off[++w] = static_cast<int32_t>(pieces);
        st = end;
      }
      if (split) {
        P.dec_merges.push_back(b);
        P.dec_merges.push_back(hk);
        P.dec_merges.push_back(static_cast<int32_t>(first_slot));
        P.dec_merges.push_back(static_cast<int32_t>(slots - first_slot));
      }
      s0 = pe;
    }
  }
  if (slots > 0x7FFFFFFF || pieces > 0x7FFFFFFF) return FI_ERR_UNSUPPORTED;
  P.dec_parts = slots;
  P.dec_warps = static_cast<int32_t>(W);
  P.dec_steps = W > 0 ? static_cast<int32_t>((total + W - 1) / W) : 0;
  I.num_units = pieces;
  I.num_ctas = static_cast<int32_t>((W + 3) / 4);
  return FI_OK;
}

}  // namespace fi

extern "C" fi_status fi_decode_plan_host(const int32_t* qo_indptr_host,
                                         const int32_t* kv_indptr_host, int32_t batch,
                                         int32_t num_qo_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t page_size, int32_t num_sms,
                                         fi_plan_info* info, int32_t* num_warps_out,
                                         int64_t* num_merges_out, int32_t* units_out,
                                         int64_t unit_capacity, int32_t* merges_out,
                                         int64_t merge_capacity, int32_t* warp_off_out,
                                         int64_t warp_off_capacity) {
  if (!info || !num_warps_out || !num_merges_out || num_sms <= 0 ||
      (units_out && unit_capacity < 0) || (merges_out && merge_capacity < 0) ||
      (warp_off_out && warp_off_capacity < 0))
    return FI_ERR_INVALID_ARGUMENT;
  fi::HostPlan P;
  const fi_status st = fi::plan_decode_host(qo_indptr_host, kv_indptr_host, batch, num_qo_heads,
                                            num_kv_heads, head_dim, page_size, 0.0f, num_sms, &P);
  if (st != FI_OK) return st;
  *info = P.info;
  *num_warps_out = P.dec_warps;
  const int64_t merges = static_cast<int64_t>(P.dec_merges.size() / 4);
  *num_merges_out = merges;
  if (units_out) {
    const int64_t n = std::min<int64_t>(unit_capacity, P.info.num_units);
    std::memcpy(units_out, P.dec_units.data(), static_cast<size_t>(n) * 4 * sizeof(int32_t));
  }
  if (merges_out) {
    const int64_t n = std::min<int64_t>(merge_capacity, merges);
    std::memcpy(merges_out, P.dec_merges.data(), static_cast<size_t>(n) * 4 * sizeof(int32_t));
  }
  if (warp_off_out) {
    const int64_t n = std::min<int64_t>(warp_off_capacity, P.dec_warps + 1);
    std::memcpy(warp_off_out, P.dec_warp_off.data(), static_cast<size_t>(n) * sizeof(int32_t));
  }
  return FI_OK;
}

extern "C" fi_status fi_prefill_plan_host(const int32_t* qo_indptr_host,
                                          const int32_t* kv_indptr_host, int32_t batch,
                                          int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t page_size, int64_t l2_bytes,
                                          const fi_plan_options* opts, fi_plan_info* info,
                                          int32_t* work_out, int64_t work_capacity) {
  if (!info || (work_out && work_capacity < 0)) return FI_ERR_INVALID_ARGUMENT;
  fi::HostPlan P;
  const fi_status st = fi::plan_host(qo_indptr_host, kv_indptr_host, batch, num_qo_heads,
                                     num_kv_heads, head_dim, page_size, 0.0f, l2_bytes, 148,
                                     opts, &P);
  if (st != FI_OK) return st;
  *info = P.info;
  if (work_out) {
    const int64_t n = std::min<int64_t>(work_capacity, P.info.num_units);
    for (int64_t t = 0; t < n; ++t) fi::unit_entry(P, t, work_out + 4 * t);
  }
  return FI_OK;
}
