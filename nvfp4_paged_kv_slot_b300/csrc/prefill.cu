// prefill.cu — causal batched prefill over the NVFP4 paged KV cache, sm_103a.
//
// What it computes follows the analysis pages of FlashInfer PRs:
//  * #4769 "FlashInfer NVFP4 KV 타일 리팩(Repack)을 통한 성능 최적화": every NVFP4
//    KV tile is dequantized once into a 16-bit staging tile outside the MMA loop
//    (there: repack_fp4_tile_to_16b feeding ldmatrix on SM80).
//  * #3575 "FlashInfer FP8 Causal Attention 최적화: O(1) 디코딩과 글로벌 스케줄링의
//    힘": causal attention with GQA; §1 O(1) tile decoding for uniform lengths;
//    §2 global reverse-Q-tile order, heaviest tiles first; §3 the L2 gate.
//
// B300 design (one persistent CTA per SM, warp-specialized):
//   warp 0        KV loads: bulk copies of the FP4 pages and E4M3 scales of
//                 each KV tile into a raw ring
//   warp 2        Q loads: TMA of the Q tiles (128B swizzle)
//   warp 1        MMA: one thread issues tcgen05.mma (QK^T: bf16 SS; PV: fp16
//                 TS with P in tensor memory) and tcgen05.commit
//   warp 3        idle
//   WG 1..NQ      softmax, one warpgroup per Q tile, one thread per query row:
//                 the row of S in registers (one tensor-memory read), online
//                 softmax in fp32 (base 2, paired fp32 arithmetic, exp2 on the
//                 MUFU unit), P written back to tensor memory over S as fp16,
//                 lazy O rescale, epilogue
//   last WG       repack: raw FP4 tile -> exact 16-bit tile in the swizzled
//                 layout the tensor cores read (K as bf16, V as fp16)
// The NQ Q tiles of a CTA are NQ query heads of one GQA group at the same
// positions, so every staged KV tile is repacked once and used NQ times.
// Tensor memory: S_i at column 128 i, O_i after all S.  Registers are moved
// to the softmax warpgroups with setmaxnreg.  All waits are bounded.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "internal.h"
#include "nvfp4.cuh"

namespace fi {

namespace {

constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainNs = 100000000ull;     // 0.1 s per wait while aborting
// The running max is moved (and O rescaled) only when it grows by more than
// 2^kLazyRescale, so P stays below 2^kLazyRescale (exact range for fp16 P).
constexpr float kLazyRescale = 8.0f;
// Threads of the repack role: the last warpgroup.  (Adding warps 2-3 was
// measured slower: they share the schedulers of two softmax warps.)
constexpr int kRepackThreads = 128;
// Devices whose cluster occupancy is cached by the launcher.
constexpr int kMaxDevices = 64;

// n / d for a divisor d fixed for the launch and any n in [0, 2^31) (fast_div
// below gives the constants; the remainder is n - (n / d) d).
struct FastDiv {
  uint32_t d, m, sh1, sh2;
  __device__ __forceinline__ int div(int n) const {
    const uint32_t t = __umulhi(m, static_cast<uint32_t>(n));
    return static_cast<int>((t + ((static_cast<uint32_t>(n) - t) >> sh1)) >> sh2);
  }
};

struct PrefillParams {
  CUtensorMap tmap_q;  // 3-D view of q: (head_dim, num_qo_heads, total_qo)
  const __nv_bfloat16* q;  // the same memory (L2 prefetch before the grid wait)
  const uint8_t* k_data;
  const uint8_t* v_data;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
  const float* k_scale;
  const float* v_scale;
  __nv_bfloat16* out;
  float* lse;
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int4* work;
  const int32_t* slot_units;  // balanced plans: work-list indices grouped by slot
  const int32_t* slot_begin;  // slot s: slot_units[slot_begin[s] .. slot_begin[s + 1])
  int32_t num_slots;
  const int32_t* page_table;
  int32_t* status;
  int64_t pt_stride;
  int32_t batch, num_qo_heads, num_kv_heads, num_pages, page_size;
  int32_t group, units_per_kv_head, head_units;
  int32_t uniform, global_reverse, uni_qo_len, uni_kv_len, q_tiles;
  int32_t num_units;
  float sm_scale;
  int32_t out_align32;  // `out` is 32-byte aligned: 32-byte stores in the epilogue
  // divisions of the tile decoding, by one multiply-high and shifts each:
  // head units, batch * head units, batch, head units * q-tiles, q-tiles,
  // head units per KV head
  FastDiv div_hu, div_bh, div_b, div_per_b, div_qt, div_upk;
};

// Division by a divisor fixed for the launch (Granlund and Montgomery,
// "Division by Invariant Integers using Multiplication", 1994, the unsigned
// method of their Figure 4.1): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (t + ((n - t) >> min(l, 1)))
// >> max(l - 1, 0) where t = mulhi(m, n), exact for every 32-bit n.
FastDiv fast_div(uint32_t d) {
  FastDiv f;
  f.d = d < 1 ? 1 : d;
  uint32_t l = 0;
  while ((uint64_t{1} << l) < f.d) ++l;
  f.m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << l) - f.d)) / f.d + 1);
  f.sh1 = l < 1 ? l : 1;
  f.sh2 = l > 1 ? l - 1 : 0;
  return f;
}

// PAIR: a 2-CTA cluster shares its KV staging tiles; each CTA loads and
// repacks half of every tile's rows (64 of 128) and writes them into both
// CTAs' staging tiles, so the raw slots hold 64 rows.
// KVF: cache format, 0 NVFP4 (codes and E4M3 block scales), 1 FP8 (one E4M3
// code per element, no block scales).
template <int D, int NQ, bool PAIR, int KVF = 0>
struct Layout {
  static constexpr int kQTile = kTileQ * D * 2;
  static constexpr int kStg = kTileKV * D * 2;
  static constexpr int kRawRows = PAIR ? kTileKV / 2 : kTileKV;
  // Ring depths.  Staging slots are used K0 V0 K1 V1 ...; with 3 slots, K of
  // the next tile reuses the slot of V of the previous one and must be
  // repacked within about one head's PV + QK^T; with 4 (pairs, whose raw
  // slots are half size) the deadline doubles.
  static constexpr int kStgStages = PAIR ? 4 : 3;
  static constexpr int kRawStages = 4;
  static constexpr int kRowBytes = KVF ? D : D / 2;  // code bytes per row
  static constexpr int kRawData = kRawRows * kRowBytes;
  static constexpr int kRawSf = KVF ? 0 : kRawRows * D / 16;
  static constexpr int kRaw = kRawData + kRawSf;
  static constexpr int kOffQ = 0;
  static constexpr int kOffStg = kOffQ + NQ * kQTile;
  static constexpr int kOffRaw = kOffStg + kStgStages * kStg;
  static constexpr int kOffBar = kOffRaw + kRawStages * kRaw;
  // q_full, q_empty, raw_full[], raw_empty[], stg_full[], stg_empty[],
  // s_full[NQ], p_full[2 NQ] (P columns of keys 0-63 / 64-127 of head i at
  // 2i / 2i+1), o_full[NQ], drain, rep_done[] (PAIR: this CTA's rows of a
  // staging slot are written)
  static constexpr int kNumBars = 2 + 2 * kRawStages + 3 * kStgStages + 4 * NQ + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base to 1024
  static constexpr int kTmemCols = (NQ * 128 + NQ * D) <= 256 ? 256 : 512;
  static constexpr int kThreads = 128 * (NQ + 2);
  // Per-thread register counts after the warpgroup reallocation: the repack
  // warpgroup gives registers up, each softmax warpgroup takes more (a whole
  // row of S), the load/MMA warpgroup keeps the launch's count.  The
  // launcher checks that the sum fits in what the CTA is launched with.
  static constexpr int kRegRepack = NQ == 2 ? 48 : 64;
  static constexpr int kRegSoftmax = NQ == 2 ? 168 : 232;
  static_assert(kOffStg % 1024 == 0 && kStg % 1024 == 0, "swizzled tiles need 1 KB alignment");
  static_assert(kAlloc <= 232448, "at most 227 KB of shared memory per CTA");
  static_assert(kRaw % 16 == 0 && kOffRaw % 16 == 0, "bulk copies need 16 B alignment");
};

struct Unit {
  int b, hk, hq0, qt, qo_start, qo_len, kv_len, n_kv;
};

// tile id -> (sequence, head unit, q-tile): arithmetic for uniform batches
// (#3575 §1, §2), the planner's list otherwise.
// A unit covers heads_per_unit query heads of one GQA group; this CTA takes
// the nq of them starting head_off heads into the unit.
__device__ __forceinline__ Unit decode_unit(const PrefillParams& p, int u, int heads_per_unit,
                                            int head_off) {
  Unit w;
  int hu;
  if (p.uniform) {
    if (p.global_reverse) {
      const int t = p.div_bh.div(u);  // u / (batch * head units)
      w.qt = p.q_tiles - 1 - t;
      const int r = u - t * static_cast<int>(p.div_bh.d);
      hu = p.div_b.div(r);
      w.b = r - hu * p.batch;
    } else {
      w.b = p.div_per_b.div(u);  // u / (head units * q-tiles)
      const int r = u - w.b * static_cast<int>(p.div_per_b.d);
      hu = p.div_qt.div(r);
      w.qt = p.q_tiles - 1 - (r - hu * p.q_tiles);
    }
    w.qo_len = p.uni_qo_len;
    w.kv_len = p.uni_kv_len;
    w.qo_start = w.b * p.uni_qo_len;
  } else {
    // the list holds one item per (sequence, q-tile); its head units are
    // consecutive units
    const int item = p.div_hu.div(u);
    hu = u - item * p.head_units;
    const int4 it = __ldg(p.work + item);
    w.b = it.x;
    w.qt = it.y;
    w.qo_start = __ldg(p.qo_indptr + w.b);
    w.qo_len = __ldg(p.qo_indptr + w.b + 1) - w.qo_start;
    w.kv_len = __ldg(p.kv_indptr + w.b + 1) - __ldg(p.kv_indptr + w.b);
  }
  w.hk = p.div_upk.div(hu);
  w.hq0 = w.hk * p.group + (hu - w.hk * p.units_per_kv_head) * heads_per_unit + head_off;
  const int last_row = min(w.qo_len, (w.qt + 1) * kTileQ) - 1;
  w.n_kv = (last_row + w.kv_len - w.qo_len) / kTileKV + 1;
  return w;
}

// The units one CTA (or CTA pair) runs: round-robin over the unit index
// (u0, u0 + stride, ...), or, for balanced plans, the units of slots u0,
// u0 + stride, ... (a launch with fewer CTAs than planned slots runs several
// slots).  Every role of the CTA walks the same sequence.
struct UnitCursor {
  int unit;  // -1 once done
  int k, end, slot;
};

__device__ __forceinline__ void unit_seek(const PrefillParams& p, int stride, UnitCursor& c) {
  for (; c.slot < p.num_slots; c.slot += stride) {
    c.k = __ldg(p.slot_begin + c.slot);
    c.end = __ldg(p.slot_begin + c.slot + 1);
    if (c.k < c.end) {
      c.unit = __ldg(p.slot_units + c.k);
      return;
    }
  }
  c.unit = -1;
}

__device__ __forceinline__ UnitCursor unit_first(const PrefillParams& p, int u0, int stride) {
  UnitCursor c{u0 < p.num_units ? u0 : -1, 0, 0, u0};
  if (p.slot_units) unit_seek(p, stride, c);
  return c;
}

__device__ __forceinline__ void unit_next(const PrefillParams& p, int stride, UnitCursor& c) {
  if (p.slot_units) {
    if (++c.k < c.end) {
      c.unit = __ldg(p.slot_units + c.k);
      return;
    }
    c.slot += stride;
    unit_seek(p, stride, c);
  } else {
    c.unit += stride;
    if (c.unit >= p.num_units) c.unit = -1;
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int D, int NQ, bool PAIR, int KVF>
__global__ void __launch_bounds__(Layout<D, NQ, PAIR, KVF>::kThreads, 1)
    nvfp4_prefill_kernel(const __grid_constant__ PrefillParams p) {
  using L = Layout<D, NQ, PAIR, KVF>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* q_smem = smem + L::kOffQ;
  uint8_t* stg_smem = smem + L::kOffStg;
  uint8_t* raw_smem = smem + L::kOffRaw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* raw_full = bars + 2;
  uint64_t* raw_empty = raw_full + L::kRawStages;
  uint64_t* stg_full = raw_empty + L::kRawStages;
  uint64_t* stg_empty = stg_full + L::kStgStages;
  uint64_t* s_full = stg_empty + L::kStgStages;
  uint64_t* p_full = s_full + NQ;
  uint64_t* o_full = p_full + 2 * NQ;
  uint64_t* drain = o_full + NQ;
  uint64_t* rep_done = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // Units: one per CTA, or one per CTA pair (both CTAs walk the same units;
  // CTA rank r takes the unit's query heads r*NQ .. r*NQ+NQ-1).
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int u0 = PAIR ? static_cast<int>(blockIdx.x / 2) : static_cast<int>(blockIdx.x);
  const int ustride = PAIR ? static_cast<int>(gridDim.x / 2) : static_cast<int>(gridDim.x);
  const int heads_per_unit = PAIR ? 2 * NQ : NQ;
  const int head_off = static_cast<int>(rank) * NQ;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < L::kRawStages; ++s) {
      mbar_init(raw_full + s, 1);
      mbar_init(raw_empty + s, kRepackThreads);
    }
    for (int s = 0; s < L::kStgStages; ++s) {
      // PAIR: the other CTA's rows arrive as bytes (expected by one local
      // arrival), and a slot is free once both CTAs' MMAs have read it.
      mbar_init(stg_full + s, kRepackThreads);
      mbar_init(stg_empty + s, PAIR ? 2 : 1);
    }
    for (int i = 0; i < NQ; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + 2 * i, 128);
      mbar_init(p_full + 2 * i + 1, 128);
      mbar_init(o_full + i, 1);
    }
    mbar_init(drain, 1);
    for (int s = 0; s < L::kStgStages; ++s) mbar_init(rep_done + s, kRepackThreads);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  if (PAIR) {
    __syncwarp();
    cluster_sync();  // the other CTA's barriers are initialized before any remote arrive
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const AbortState ab{abort_flag, p.status, kTimeoutNs, FI_DEV_WAIT_TIMEOUT};
  // Everything up to grid_dep_wait overlaps the previous grid of the stream
  // when this one is launched as its programmatic dependent (the prefetch
  // before the wait of the FlashInfer PR #8210 page, "FlashInfer: sm_107a
  // 아키텍처를 위한 Fused Decode List Scorer 프리페칭 최적화").  The Q rows and
  // the page-table row of this CTA's first unit are pulled into L2 here: a
  // prefetch writes nothing and L2 stays coherent with the previous grid's
  // writes, so results cannot change.  Finding the first unit reads only the
  // plan's memory, which no kernel writes (its copy completed before the
  // previous grid started).  Every input is read after the wait.
  if (warp == 2) {
    const UnitCursor uc = unit_first(p, u0, ustride);
    if (uc.unit >= 0) {
      const Unit w = decode_unit(p, uc.unit, heads_per_unit, head_off);
      const int rows = min(kTileQ, w.qo_len - w.qt * kTileQ);
      const __nv_bfloat16* q0 =
          p.q + (static_cast<int64_t>(w.qo_start + w.qt * kTileQ) * p.num_qo_heads + w.hq0) * D;
      for (int r = lane; r < rows; r += 32)
        prefetch_l2_bulk(q0 + static_cast<int64_t>(r) * p.num_qo_heads * D, NQ * D * 2);
      if (lane == 0) prefetch_l2_line(p.page_table + static_cast<int64_t>(w.b) * p.pt_stride);
    }
  }
  grid_dep_wait();
  grid_dep_launch();

  const int wg = threadIdx.x / 128;
  // Repack: raw FP4 tiles -> 16-bit staging tiles, by kRepackThreads threads
  // (rt = 0 .. kRepackThreads-1).
  auto repack_role = [&](int rt) {
    uint32_t raw_k = 0, stg_k = 0;
    bool ok = true;
    for (UnitCursor uc = unit_first(p, u0, ustride); ok && uc.unit >= 0; unit_next(p, ustride, uc)) {
      const int u = uc.unit;
      const Unit w = decode_unit(p, u, heads_per_unit, head_off);
      for (int j = 0; ok && j < w.n_kv; ++j) {
        const int valid = min(kTileKV, w.kv_len - j * kTileKV);
        for (int t = 0; t < 2; ++t, ++raw_k, ++stg_k) {
          const int rs = raw_k % L::kRawStages;
          const int ss = stg_k % L::kStgStages;
          if (!mbar_wait(raw_full + rs, (raw_k / L::kRawStages) & 1, ab)) { ok = false; break; }
          if (!mbar_wait<PAIR>(stg_empty + ss, ((stg_k / L::kStgStages) & 1) ^ 1, ab)) { ok = false; break; }
          if (PAIR) {
            // This CTA's 64 rows go into its own staging tile; once all the
            // repack threads have written them, one thread bulk-copies them
            // into the other CTA's tile (D/64 contiguous 8 KB pieces, one per
            // 64-column block), counted in bytes on that CTA's stg_full.
            const int half_valid = min(max(valid - 64 * static_cast<int>(rank), 0), 64);
            uint8_t* dst = stg_smem + ss * L::kStg;
            const uint8_t* raw = raw_smem + rs * L::kRaw;
            if constexpr (KVF == 1) {
              if (t)
                repack_half_fp8<D, true, kRepackThreads>(raw, dst, 64 * rank, half_valid, rt);
              else
                repack_half_fp8<D, false, kRepackThreads>(raw, dst, 64 * rank, half_valid, rt);
            } else {
              if (t)
                repack_half<D, true, kRepackThreads>(raw, dst, 64 * rank, half_valid, rt);
              else
                repack_half<D, false, kRepackThreads>(raw, dst, 64 * rank, half_valid, rt);
            }
            fence_proxy_async_smem();
            mbar_arrive(rep_done + ss);
            if (rt == 0) {
              // every repack thread's rows of this slot are written (a bounded
              // wait, like all others: a timed-out sibling cannot hang it)
              if (!mbar_wait(rep_done + ss, (stg_k / L::kStgStages) & 1, ab)) { ok = false; break; }
              const uint32_t peer_bar = mapa_shared(smem_u32(stg_full + ss), rank ^ 1u);
#pragma unroll
              for (int cb = 0; cb < D / 64; ++cb) {
                uint8_t* piece = dst + cb * 16384 + 64 * rank * 128;
                bulk_s2s_cluster(mapa_shared(smem_u32(piece), rank ^ 1u), piece, 64 * 128,
                                 peer_bar);
              }
              // the bytes the other CTA sends into this CTA's tile
              mbar_arrive_expect_tx(stg_full + ss, (D / 64) * 64 * 128);
            } else {
              mbar_arrive(stg_full + ss);
            }
          } else {
            const uint8_t* raw = raw_smem + rs * L::kRaw;
            uint8_t* dst = stg_smem + ss * L::kStg;
            if constexpr (KVF == 1) {
              if (t)
                repack_tile_fp8<D, true, kRepackThreads>(raw, dst, valid, rt);
              else
                repack_tile_fp8<D, false, kRepackThreads>(raw, dst, valid, rt);
            } else {
              if (t)
                repack_tile<D, true, kRepackThreads>(raw, dst, valid, rt);
              else
                repack_tile<D, false, kRepackThreads>(raw, dst, valid, rt);
            }
            fence_proxy_async_smem();
            mbar_arrive(stg_full + ss);
          }
          mbar_arrive(raw_empty + rs);
        }
      }
    }
  };
  if (warp == 0) {
    // ------------------------------------------------------- KV load warp
    uint32_t raw_k = 0;
    int it = 0;
    bool ok = true;
    const uint32_t pg_data = static_cast<uint32_t>(p.page_size) * L::kRowBytes;
    const uint32_t pg_sf = static_cast<uint32_t>(p.page_size) * (D / 16);
    const int pages_per_tile = kTileKV / p.page_size;
    // PAIR: this CTA's rows of a tile are 64*rank .. 64*rank+63: whole pages
    // for page sizes up to 64, half a page (its rows 64*rank ..) for 128.
    const int rows_per_copy = PAIR ? min(p.page_size, 64) : p.page_size;
    const uint32_t cp_data = static_cast<uint32_t>(rows_per_copy) * L::kRowBytes;
    const uint32_t cp_sf = KVF ? 0u : static_cast<uint32_t>(rows_per_copy) * (D / 16);
    const int copies_per_tile = PAIR ? max(pages_per_tile / 2, 1) : pages_per_tile;
    const uint32_t src_row_off = (PAIR && p.page_size == 128) ? 64u * rank : 0u;
    for (UnitCursor uc = unit_first(p, u0, ustride); ok && uc.unit >= 0;
         unit_next(p, ustride, uc), ++it) {
      const int u = uc.unit;
      const Unit w = decode_unit(p, u, heads_per_unit, head_off);
      const int32_t* pt = p.page_table + static_cast<int64_t>(w.b) * p.pt_stride;
      const int seq_pages = (w.kv_len + p.page_size - 1) / p.page_size;
      for (int j = 0; ok && j < w.n_kv; ++j) {
        for (int t = 0; t < 2; ++t, ++raw_k) {
          const int slot = raw_k % L::kRawStages;
          if (!mbar_wait(raw_empty + slot, ((raw_k / L::kRawStages) & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          const int first = j * pages_per_tile +
                            ((PAIR && pages_per_tile > 1) ? static_cast<int>(rank) * copies_per_tile : 0);
          const int npg = max(min(copies_per_tile, seq_pages - first), 0);
          if (lane == 0) mbar_arrive_expect_tx(raw_full + slot, npg * (cp_data + cp_sf));
          __syncwarp();
          if (lane < npg) {
            int page = __ldg(pt + first + lane);
            if (page < 0 || page >= p.num_pages) {
              atomicOr(p.status, FI_DEV_PAGE_OOB);
              page = 0;
            }
            const int64_t blk = static_cast<int64_t>(page) * p.num_kv_heads + w.hk;
            const uint8_t* gd =
                (t ? p.v_data : p.k_data) + blk * pg_data + src_row_off * L::kRowBytes;
            uint8_t* sd = raw_smem + slot * L::kRaw;
            bulk_g2s(sd + lane * cp_data, gd, cp_data, raw_full + slot);
            if constexpr (KVF == 0) {
              const uint8_t* gs = (t ? p.v_sf : p.k_sf) + blk * pg_sf + src_row_off * (D / 16);
              bulk_g2s(sd + L::kRawData + lane * cp_sf, gs, cp_sf, raw_full + slot);
            }
          }
          __syncwarp();
        }
      }
    }
    if (!ok) {
      // Aborting: wait (briefly) for the copies this warp may still have in
      // flight so that no copy lands in shared memory after the CTA exits.
      volatile int drain_flag = 0;
      const AbortState drain_ab{&drain_flag, nullptr, kDrainNs, 0};
      const uint32_t n = raw_k < L::kRawStages ? raw_k : L::kRawStages;
      for (uint32_t f = raw_k - n; f < raw_k; ++f)
        mbar_wait(raw_full + (f % L::kRawStages), (f / L::kRawStages) & 1, drain_ab);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA warp
    if (lane == 0) {
      constexpr uint32_t kIdescQK = idesc_f16(1, 0, 0, kTileQ, kTileKV);
      constexpr uint32_t kIdescPV = idesc_f16(0, 0, 1, kTileQ, D);
      const uint32_t q_addr = smem_u32(q_smem);
      const uint32_t stg_addr = smem_u32(stg_smem);
      uint32_t stg_k = 0;
      uint32_t pk[NQ];
      for (int i = 0; i < NQ; ++i) pk[i] = 0;
      int it = 0;
      bool ok = true;
      // Descriptors are built once; a start address inside the region is
      // reached by adding (byte offset >> 4) to the low 14-bit address field
      // (shared-memory offsets stay below 2^18 bytes, so nothing carries out).
      const uint64_t q_desc0 = smem_desc_sw128(q_addr, 16, 1024);
      const uint64_t k_desc0 = smem_desc_sw128(stg_addr, 16, 1024);
      const uint64_t v_desc0 = smem_desc_sw128(stg_addr, 16384, 1024);
      auto issue_qk = [&](int i, uint32_t ss) {
        const uint32_t d_tmem = tmem_base + i * 128;
        const uint64_t qd = q_desc0 + ((i * L::kQTile) >> 4);
        const uint64_t kd = k_desc0 + ((ss * L::kStg) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_ss(d_tmem, qd + off, kd + off, kIdescQK, kk > 0 ? 1u : 0u);
        }
      };
      // A staging slot is free once this CTA's MMAs have read it (PAIR: the
      // arrival goes to the slot's barrier in both CTAs, whose repack threads
      // both write into it).
      auto release_stg = [&](uint32_t ss) {
        if (PAIR)
          mma_commit_multicast(stg_empty + ss, 3);
        else
          mma_commit(stg_empty + ss);
      };
      // PV over keys 64h .. 64h+63 (P columns 32h .. 32h+31)
      auto issue_pv_half = [&](int i, uint32_t ss, int h, bool acc) {
        const uint32_t d_tmem = tmem_base + NQ * 128 + i * D;
        const uint32_t a_tmem = tmem_base + i * 128;
        const uint64_t vd = v_desc0 + ((ss * L::kStg) >> 4);
#pragma unroll
        for (int s = 4 * h; s < 4 * h + 4; ++s)
          mma_ts(d_tmem, a_tmem + s * 8, vd + ((s * 2048) >> 4), kIdescPV,
                 (acc || s > 0) ? 1u : 0u);
      };
      for (UnitCursor uc = unit_first(p, u0, ustride); ok && uc.unit >= 0;
           unit_next(p, ustride, uc), ++it) {
        const int u = uc.unit;
        const Unit w = decode_unit(p, u, heads_per_unit, head_off);
        if (!mbar_wait(q_full, it & 1, ab)) { ok = false; break; }
        // K tile 0
        uint32_t ss_k = stg_k % L::kStgStages;
        if (!mbar_wait<PAIR>(stg_full + ss_k, (stg_k / L::kStgStages) & 1, ab)) { ok = false; break; }
        ++stg_k;
        tc_fence_after();
        for (int i = 0; i < NQ; ++i) {
          issue_qk(i, ss_k);
          mma_commit(s_full + i);
        }
        if (w.n_kv == 1) mma_commit(q_empty);
        release_stg(ss_k);
        for (int j = 0; ok && j < w.n_kv; ++j) {
          const uint32_t ss_v = stg_k % L::kStgStages;
          if (!mbar_wait<PAIR>(stg_full + ss_v, (stg_k / L::kStgStages) & 1, ab)) { ok = false; break; }
          ++stg_k;
          const bool more = j + 1 < w.n_kv;
          for (int i = 0; i < NQ; ++i) {
            // the first half of P may be multiplied while the softmax still
            // computes the second
            if (!mbar_wait(p_full + 2 * i, pk[i] & 1, ab)) { ok = false; break; }
            tc_fence_after();
            issue_pv_half(i, ss_v, 0, j > 0);
            if (!mbar_wait(p_full + 2 * i + 1, pk[i] & 1, ab)) { ok = false; break; }
            ++pk[i];
            tc_fence_after();
            issue_pv_half(i, ss_v, 1, true);
            if (i == NQ - 1) release_stg(ss_v);
            // O_i of this unit is complete once this PV is: the epilogue of
            // head i need not wait for the other heads' last PVs
            if (!more) mma_commit(o_full + i);
            if (more) {
              if (i == 0) {
                ss_k = stg_k % L::kStgStages;
                if (!mbar_wait<PAIR>(stg_full + ss_k, (stg_k / L::kStgStages) & 1, ab)) { ok = false; break; }
                ++stg_k;
                tc_fence_after();
              }
              issue_qk(i, ss_k);
              mma_commit(s_full + i);
              if (i == NQ - 1) {
                release_stg(ss_k);
                if (j + 2 == w.n_kv) mma_commit(q_empty);
              }
            }
          }
        }
        if (!ok) break;
      }
      // Every MMA this thread issued has completed once `drain` arrives.
      mma_commit(drain);
      volatile int drain_flag = 0;
      const AbortState drain_ab{&drain_flag, nullptr, ok ? kTimeoutNs : kDrainNs, 0};
      mbar_wait(drain, 0, drain_ab);
    }
  } else if (warp == 2) {
    // -------------------------------------------------------- Q load warp
    // Q tiles are loaded as soon as the buffer is free (the last QK^T of the
    // previous unit has completed), independently of the KV loads, so the
    // next unit's Q is in flight while the current unit finishes.
    if (lane == 0) {
      prefetch_tensormap(&p.tmap_q);
      int it = 0;
      int q_issued = -1;  // iteration of the last Q load issued
      for (UnitCursor uc = unit_first(p, u0, ustride); uc.unit >= 0;
           unit_next(p, ustride, uc), ++it) {
        const int u = uc.unit;
        const Unit w = decode_unit(p, u, heads_per_unit, head_off);
        if (!mbar_wait(q_empty, (it & 1) ^ 1, ab)) break;
        mbar_arrive_expect_tx(q_full, NQ * L::kQTile);
        for (int i = 0; i < NQ; ++i)
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(q_smem + i * L::kQTile + h * 16384, &p.tmap_q, q_full, h * 64,
                        w.hq0 + i, w.qo_start + w.qt * kTileQ);
        q_issued = it;
      }
      // no copy may land in shared memory after the CTA exits
      volatile int drain_flag = 0;
      const AbortState drain_ab{&drain_flag, nullptr, kDrainNs, 0};
      if (q_issued >= 0) mbar_wait(q_full, q_issued & 1, drain_ab);
    }
  } else if (wg == 0) {
    // warp 3: no role
  } else if (wg <= NQ) {
    // ------------------------------------------------------------- softmax
    setmaxnreg_inc<L::kRegSoftmax>();
    const int i = wg - 1;
    const int r = threadIdx.x - 128 * wg;  // query row within the tile
    const uint32_t lane_base = tmem_base + ((static_cast<uint32_t>(r / 32) * 32) << 16);
    const uint32_t s_col = lane_base + i * 128;
    const uint32_t o_col = lane_base + NQ * 128 + i * D;
    const float ks = __ldg(p.k_scale);
    const float vs = __ldg(p.v_scale);
    if (blockIdx.x == 0 && threadIdx.x == 128) {
      int bad = 0;
      if (!(isfinite(ks) && ks > 0.0f)) bad |= FI_DEV_BAD_K_SCALE;
      if (!(isfinite(vs) && vs > 0.0f)) bad |= FI_DEV_BAD_V_SCALE;
      if (bad) atomicOr(p.status, bad);
    }
    const float scale_log2 = p.sm_scale * ks * 1.4426950408889634f;
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    uint32_t sk = 0;
    int it = 0;
    bool ok = true;
    for (UnitCursor uc = unit_first(p, u0, ustride); ok && uc.unit >= 0;
         unit_next(p, ustride, uc), ++it) {
      const int u = uc.unit;
      const Unit w = decode_unit(p, u, heads_per_unit, head_off);
      const int row_q = w.qt * kTileQ + r;
      const int delta = w.kv_len - w.qo_len;
      const int limit = row_q + delta;                 // last key this row sees
      const int tile_first_limit = w.qt * kTileQ + delta;
      float m_ref = -INFINITY;                         // running max (log2 units)
      float l = 0.0f;                                  // running sum of p
      for (int j = 0; j < w.n_kv; ++j) {
        if (!mbar_wait(s_full + i, sk & 1, ab)) { ok = false; break; }
        ++sk;
        tc_fence_after();
        const int key0 = j * kTileKV;
        // keys beyond this row's causal limit exist only in tiles that reach
        // past the first row's limit (the diagonal tiles)
        const bool masked = key0 + kTileKV - 1 > tile_first_limit;
        // The whole row of S in registers: one tensor-memory read per tile
        // (each read costs hundreds of cycles, so their number matters more
        // than the registers).
        uint32_t sv[128];
        tmem_ld128(s_col, sv);
        if (masked) {
#pragma unroll
          for (int k = 0; k < 128; ++k)
            if (key0 + k > limit) sv[k] = 0xFF800000u;  // -inf
        }
        float mx;
        {
          // four independent chains over columns 32c .. 32c+31: element 32c,
          // fifteen three-input steps over 32c+1 .. 32c+30, then 32c+31
          float mc[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            mc[c] = __uint_as_float(sv[32 * c]);
#pragma unroll
            for (int k = 1; k < 31; k += 2)
              mc[c] = fmax3(mc[c], __uint_as_float(sv[32 * c + k]),
                            __uint_as_float(sv[32 * c + k + 1]));
            mc[c] = fmaxf(mc[c], __uint_as_float(sv[32 * c + 31]));
          }
          mx = fmaxf(fmax3(mc[0], mc[1], mc[2]), mc[3]);
        }
        const float m_new = fmaxf(m_ref, mx * scale_log2);
        // lazy rescale: the running max moves only when it grows by more than
        // 2^kLazyRescale (P stays below that power of two otherwise).  O holds
        // the PV products of tiles < j, all complete (the commit behind this
        // tile's s_full follows them); it is rescaled, 16 columns at a time,
        // before any P of this tile is released.  The tensor-memory accesses
        // are warp-wide, so the decision is the warp's: when any of its rows
        // grows past the threshold, every row of the warp moves its max to
        // m_new (for the others an ordinary online-softmax step, alpha <= 1).
        if (__any_sync(0xFFFFFFFFu, m_new > m_ref + kLazyRescale)) {
          const float alpha = ex2(m_ref - m_new);
          l *= alpha;
          m_ref = m_new;
          if (j > 0) {
#pragma unroll 1
            for (int c = 0; c < D / 16; ++c) {
              uint32_t o[16];
              tmem_ld16(o_col + c * 16, o);
#pragma unroll
              for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st16(o_col + c * 16, o);
            }
          }
        }
        const uint64_t negm2 = f2_pack(-m_ref, -m_ref);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // P (fp16 pairs) over the consumed S registers, pair k in sv[k];
        // columns 64h..64h+63 of S give P columns 32h..32h+31.  Half 0 is
        // stored, half 1 computed while that store completes, then half 0
        // is released to the MMA, then half 1 stored and released.
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int k = 32 * h; k < 32 * h + 32; ++k) {
            const uint64_t x2 =
                f2_fma(f2_pack(__uint_as_float(sv[2 * k]), __uint_as_float(sv[2 * k + 1])),
                       scale2, negm2);
            float x0, x1;
            f2_unpack(x2, x0, x1);
            const uint64_t p2 = f2_pack(ex2(x0), ex2(x1));
            acc[k & 3] = f2_add(acc[k & 3], p2);
            float p0, p1;
            f2_unpack(p2, p0, p1);
            sv[k] = pack_f16x2(p0, p1);
          }
          if (h == 0) {
            tmem_st32(s_col, *reinterpret_cast<uint32_t(*)[32]>(sv));
          } else {
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_full + 2 * i);
            tmem_st32(s_col + 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_full + 2 * i + 1);
          }
        }
        acc[0] = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
        float a0, a1;
        f2_unpack(acc[0], a0, a1);
        l += a0 + a1;
      }
      if (!ok) break;
      if (!mbar_wait(o_full + i, it & 1, ab)) { ok = false; break; }
      tc_fence_after();
      const bool valid = row_q < w.qo_len;
      const float inv = vs / l;
      __nv_bfloat16* dst =
          p.out + (static_cast<int64_t>(w.qo_start + row_q) * p.num_qo_heads + w.hq0 + i) * D;
      // the whole row of O in one tensor-memory read, then 32-byte stores
      // (full sectors; 16-byte stores when `out` is only 16-byte aligned)
      uint32_t o[D];
      if constexpr (D == 128)
        tmem_ld128(o_col, o);
      else
        tmem_ld64(o_col, o);
      if (valid) {
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          uint32_t v[8];
#pragma unroll
          for (int k = 0; k < 8; ++k)
            v[k] = pack_bf16x2(__uint_as_float(o[16 * c + 2 * k]) * inv,
                               __uint_as_float(o[16 * c + 2 * k + 1]) * inv);
          if (p.out_align32) {
            st_global_v8(dst + 16 * c, v);
          } else {
            reinterpret_cast<uint4*>(dst + 16 * c)[0] = make_uint4(v[0], v[1], v[2], v[3]);
            reinterpret_cast<uint4*>(dst + 16 * c)[1] = make_uint4(v[4], v[5], v[6], v[7]);
          }
        }
      }
      if (valid && p.lse)
        p.lse[static_cast<int64_t>(w.qo_start + row_q) * p.num_qo_heads + w.hq0 + i] =
            (m_ref + log2f(l)) * 0.6931471805599453f;
      // the next unit's first PV may overwrite O_i only after these loads
      tc_fence_before();
    }
  } else {
    // ------------------------------------------------------------- repack
    setmaxnreg_dec<L::kRegRepack>();
    repack_role(threadIdx.x - 128 * (NQ + 1));
  }

  __syncwarp();
  tc_fence_before();
  // PAIR: neither CTA leaves while the other may still write into its
  // staging tiles or arrive on its barriers.
  if (PAIR)
    cluster_sync();
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, L::kTmemCols);
}

template <int D, int NQ, bool PAIR, int KVF>
fi_status launch_impl(const PrefillParams& p, int grid, cudaStream_t stream) {
  using L = Layout<D, NQ, PAIR, KVF>;
  auto kern = nvfp4_prefill_kernel<D, NQ, PAIR, KVF>;
  // at least ~116 KB so that a single CTA (and its 256-512 TMEM columns)
  // occupies each SM
  const int smem = L::kAlloc > 118784 ? L::kAlloc : 118784;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FI_ERR_UNSUPPORTED;
  // The shared-memory attribute and the register check are done once per
  // device (1 = done; a race between host threads only repeats them).
  static std::atomic<int> checked[kMaxDevices];
  if (checked[dev].load(std::memory_order_relaxed) == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return FI_ERR_CUDA;
    // The warpgroup register reallocation must fit in what the launch gives
    // the CTA, or a warpgroup's increase would never be granted.
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return FI_ERR_CUDA;
    if (128 * (attr.numRegs + L::kRegRepack + NQ * L::kRegSoftmax) > attr.numRegs * L::kThreads)
      return FI_ERR_UNSUPPORTED;
    checked[dev].store(1, std::memory_order_relaxed);
  }
  if (!PAIR) return launch_pdl(kern, dim3(grid), dim3(L::kThreads), smem, stream, p);
  cudaLaunchAttribute cl[1];
  cl[0].id = cudaLaunchAttributeClusterDimension;
  cl[0].val.clusterDim.x = 2;
  cl[0].val.clusterDim.y = 1;
  cl[0].val.clusterDim.z = 1;
  // As many pairs as can be resident at once (persistent), at most one per
  // unit.  The occupancy query is cached per device (0 = not yet known); a
  // race between host threads only repeats the same query.
  static std::atomic<int> max_clusters[kMaxDevices];
  int n_clusters = max_clusters[dev].load(std::memory_order_relaxed);
  if (n_clusters == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return FI_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * std::max(sms / 2, 1));
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = cl;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n_clusters, kern, &cfg) != cudaSuccess || n_clusters <= 0)
      return FI_ERR_CUDA;
    max_clusters[dev].store(n_clusters, std::memory_order_relaxed);
  }
  const int pairs = std::max(1, std::min(grid / 2, n_clusters));
  return launch_pdl(kern, dim3(2 * pairs), dim3(L::kThreads), smem, stream, p, cl, 1);
}

template <int KVF>
fi_status dispatch(const HostPlan& P, const PrefillParams& p, int grid, cudaStream_t stream) {
  const int D = P.head_dim;
  const int nq = P.info.heads_per_cta;
  if (P.pair) {
    if (nq != 2) return FI_ERR_UNSUPPORTED;
    return D == 128 ? launch_impl<128, 2, true, KVF>(p, grid, stream)
                    : launch_impl<64, 2, true, KVF>(p, grid, stream);
  }
  if (D == 128)
    return nq == 2 ? launch_impl<128, 2, false, KVF>(p, grid, stream)
                   : launch_impl<128, 1, false, KVF>(p, grid, stream);
  return nq == 2 ? launch_impl<64, 2, false, KVF>(p, grid, stream)
                 : launch_impl<64, 1, false, KVF>(p, grid, stream);
}

}  // namespace

fi_status launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  const HostPlan& P = *a.plan;
  if (P.info.num_units == 0) return FI_OK;
  PrefillParams p;
  memset(&p, 0, sizeof(p));
  const int D = P.head_dim;
  if (!encode_tensor_map_3d_bf16(&p.tmap_q, a.q, D, P.num_qo_heads, P.info.total_qo_len,
                                 static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(P.num_qo_heads) * D * 2, 64, 1, kTileQ))
    return FI_ERR_CUDA;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.k_data = a.cache.k_data;
  p.v_data = a.cache.v_data;
  p.k_sf = a.cache.k_sf;
  p.v_sf = a.cache.v_sf;
  p.k_scale = a.cache.k_scale;
  p.v_scale = a.cache.v_scale;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.out_align32 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 ? 1 : 0;
  p.lse = a.lse;
  p.qo_indptr = a.qo_indptr_dev;
  p.kv_indptr = a.kv_indptr_dev;
  p.work = reinterpret_cast<const int4*>(a.work_dev);
  p.page_table = a.page_table;
  p.status = a.status;
  p.pt_stride = a.page_table_stride;
  p.batch = P.info.batch;
  p.num_qo_heads = P.num_qo_heads;
  p.num_kv_heads = P.num_kv_heads;
  p.num_pages = a.cache.num_pages;
  p.page_size = P.page_size;
  p.group = P.group;
  p.units_per_kv_head = P.units_per_kv_head;
  p.head_units = P.info.head_units;
  p.div_hu = fast_div(static_cast<uint32_t>(P.info.head_units));
  p.div_upk = fast_div(static_cast<uint32_t>(P.units_per_kv_head));
  p.uniform = (P.info.is_uniform && !a.work_dev) ? 1 : 0;  // else: decode from the work list
  p.slot_units = a.slot_units_dev;
  p.slot_begin = a.slot_begin_dev;
  p.num_slots = a.num_slots;
  p.global_reverse = P.info.global_reverse;
  p.uni_qo_len = P.uniform_qo_len;
  p.uni_kv_len = P.uniform_kv_len;
  p.q_tiles = P.info.q_tiles;
  p.div_b = fast_div(static_cast<uint32_t>(P.info.batch));
  p.div_qt = fast_div(static_cast<uint32_t>(P.info.q_tiles));
  p.div_bh = fast_div(static_cast<uint32_t>(P.info.batch) * static_cast<uint32_t>(P.info.head_units));
  p.div_per_b =
      fast_div(static_cast<uint32_t>(P.info.head_units) * static_cast<uint32_t>(P.info.q_tiles));
  if (P.info.num_units > 0x7FFFFFFF) return FI_ERR_UNSUPPORTED;
  p.num_units = static_cast<int32_t>(P.info.num_units);
  p.sm_scale = P.sm_scale;
  const int grid = P.info.num_ctas;
  return P.kv_format == 1 ? dispatch<1>(P, p, grid, stream) : dispatch<0>(P, p, grid, stream);
}

}  // namespace fi
