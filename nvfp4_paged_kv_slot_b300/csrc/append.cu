// append.cu — NVFP4 quantize-append of bf16 K/V rows through a slot_mapping
// (FlashInfer PR #6204 analysis page, "FlashInfer: NVFP4 KV 캐시 어펜드 성능
// 최적화로 인한 동기화 제거": the append kernel checks the device scales itself
// instead of the host reading them back).
//
// Two kernels, one result.  The staged kernel (long appends, rows of up to
// 8192 elements): one CTA per SM; a producer warp moves groups of T tokens
// (both tensors, all heads, about 32 KB) into a ring of shared-memory stages
// with bulk copies counted on the stage's mbarrier (one copy per tensor when
// its tokens are contiguous); 16 consumer warps load the token slots one
// stage ahead and quantize from shared memory, each thread two 16-element
// blocks of one (tensor, token, head) row, with the per-tensor quantizer
// constants (reciprocals of every possible block scale) built once per CTA.
// The direct kernel (short appends and wider rows): grid y = (tensor, kv
// head), x = persistent CTAs striding over token groups, each thread loading
// its two blocks of a row one step ahead from global memory.  Both are
// HBM-bound: per written token they read 2*H*D*2 bytes and write
// 2*H*(D/2 + D/16) bytes (the algorithmic count; the values of skipped tokens
// are read as well).  The page size is a power of two (shift and mask).
#include <algorithm>

#include "internal.h"
#include "nvfp4.cuh"

namespace fi {

namespace {

constexpr int kAppendThreads = 256;
constexpr int kCtasPerSm = 3;  // resident CTAs per SM the persistent grid aims for
// Passes of the direct kernel whose input rows are pulled into L2 before the
// grid-dependency wait (measured: 2 beats 1, 3 and all).
constexpr int kPrefetchPasses = 2;
constexpr int kDirectBlocksPerThread = 2;

// Staged kernel: 16 consumer warps and one producer warp; stages of about
// kStageBytes (whole tokens); at most kMaxStages of them, within kSmemBudget.
constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kStagedThreads = kConsumers + 32;
constexpr int kStageBytes = 32768;
constexpr int kMaxStages = 6;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kMaxTokPerStage = 32;              // tokens per stage at most
constexpr int64_t kStagedMinTokens = 65536;      // shorter appends take the direct kernel
constexpr uint64_t kWaitNs = 2000000000ull;      // 2 s per pipeline wait
constexpr uint64_t kDrainWaitNs = 100000000ull;  // 0.1 s per wait while aborting

struct AppendParams {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t k_tok_stride, v_tok_stride;
  const float* k_scale_dev;
  const float* v_scale_dev;
  float k_scale_host, v_scale_host;
  const int64_t* slot_mapping;
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_sf;
  uint8_t* v_sf;
  int64_t num_tokens;
  int64_t num_slots;  // num_pages * page_size
  int32_t num_kv_heads, log2_page_size;
  int32_t* status;
  // staged kernel only
  int32_t tok_per_stage, num_stages, row_bytes, stage_bytes;
};

__device__ __forceinline__ bool scale_ok(float g) { return isfinite(g) && g > 0.0f; }

// One work item of the direct kernel: a token's slot and BPT 16-element bf16
// blocks (j, j + D/(16 BPT), ...) of one of its (tensor, head) rows.
template <int BPT>
struct ItemB {
  int64_t slot;
  uint4 w[BPT][2];
};

template <int D, int BPT>
__device__ __forceinline__ ItemB<BPT> load_item(const AppendParams& p,
                                                const __nv_bfloat16* src0, int64_t tok_stride,
                                                int64_t tok) {
  constexpr int kTpr = D / 16 / BPT;
  ItemB<BPT> it;
  it.slot = -1;
  if (tok < p.num_tokens) {
    const uint4* src = reinterpret_cast<const uint4*>(src0 + tok * tok_stride);
    it.slot = __ldg(p.slot_mapping + tok);
#pragma unroll
    for (int b = 0; b < BPT; ++b) {
      it.w[b][0] = __ldcs(src + 2 * kTpr * b);
      it.w[b][1] = __ldcs(src + 2 * kTpr * b + 1);
    }
  } else {
#pragma unroll
    for (int b = 0; b < BPT; ++b) it.w[b][0] = it.w[b][1] = make_uint4(0u, 0u, 0u, 0u);
  }
  return it;
}

// Direct kernel: each thread owns BPT blocks of one (token, tensor, head) row
// per step; kTpr = D / (16 BPT) threads share a row.
template <int D, int BPT>
__global__ void __launch_bounds__(kAppendThreads, kCtasPerSm)
    nvfp4_append_kernel(const AppendParams p) {
  constexpr int kBlocks = D / 16;
  constexpr int kTpr = kBlocks / BPT;  // threads per (token, tensor, head) row
  constexpr int kTokPerCta = kAppendThreads / kTpr;
  __shared__ float4 tab[128];
  const int64_t step = static_cast<int64_t>(gridDim.x) * kTokPerCta;
  {
    // While the previous grid of the stream finishes (programmatic dependent
    // launch), pull the K or V row segments of this CTA's first
    // kPrefetchPasses passes into L2: the tokens blockIdx.x * kTokPerCta + r
    // + k * step, k < kPrefetchPasses, of (tensor, head) blockIdx.y.  Only
    // kernel parameters are read here, and a prefetch cannot change what the
    // loads after the wait see.  (Prefetching every pass queued the whole
    // input ahead of the first real loads and was slower.)
    const int Hp = p.num_kv_heads;
    const int tp = static_cast<int>(blockIdx.y) >= Hp ? 1 : 0;
    const __nv_bfloat16* src = (tp ? p.v : p.k) + (static_cast<int>(blockIdx.y) - tp * Hp) * D;
    const int64_t ts = tp ? p.v_tok_stride : p.k_tok_stride;
    if (((reinterpret_cast<uintptr_t>(src) | static_cast<uintptr_t>(ts * 2)) & 15u) == 0) {
      constexpr int kRowsPerPass = kAppendThreads / kTokPerCta;
      const int64_t first = static_cast<int64_t>(blockIdx.x) * kTokPerCta;
      const int64_t end = min(p.num_tokens, first + kPrefetchPasses * step);
      for (int64_t tok = first + threadIdx.x % kTokPerCta + (threadIdx.x / kTokPerCta) * step;
           tok < end; tok += kRowsPerPass * step)
        prefetch_l2_bulk(src + tok * ts, D * 2);
    }
  }
  // Inputs may come from the previous grid of the stream: wait for it, then
  // let the next grid start launching.
  grid_dep_wait();
  grid_dep_launch();

  // Scale check, once per CTA before any store: a bad scale means no CTA
  // writes anything, for K and V alike.
  const float ks = p.k_scale_dev ? __ldg(p.k_scale_dev) : p.k_scale_host;
  const float vs = p.v_scale_dev ? __ldg(p.v_scale_dev) : p.v_scale_host;
  if (!scale_ok(ks) || !scale_ok(vs)) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
      atomicOr(p.status, (scale_ok(ks) ? 0 : FI_DEV_BAD_K_SCALE) |
                             (scale_ok(vs) ? 0 : FI_DEV_BAD_V_SCALE));
    return;  // uniform across the grid
  }

  const int H = p.num_kv_heads;
  const int t = static_cast<int>(blockIdx.y) >= H ? 1 : 0;  // 0 = K, 1 = V
  const int h = static_cast<int>(blockIdx.y) - t * H;
  const float g = t ? vs : ks;
  if (threadIdx.x < 128) tab[threadIdx.x] = quant_scale_entry(threadIdx.x, g);
  const QuantConsts qc = quant_consts(g);
  __syncthreads();

  const int j = threadIdx.x % kTpr;
  const uint32_t hrow = static_cast<uint32_t>(h) << p.log2_page_size;
  uint8_t* const dbase = (t ? p.v_data : p.k_data) + static_cast<uint64_t>(hrow) * (D / 2) + j * 8;
  uint8_t* const sbase = (t ? p.v_sf : p.k_sf) + static_cast<uint64_t>(hrow) * kBlocks + j;
  const __nv_bfloat16* const src0 = (t ? p.v : p.k) + h * D + j * 16;
  const int64_t tok_stride = t ? p.v_tok_stride : p.k_tok_stride;
  const uint32_t page_rows = static_cast<uint32_t>(H) << p.log2_page_size;
  const uint32_t pmask = (1u << p.log2_page_size) - 1u;
  const uint64_t num_slots = static_cast<uint64_t>(p.num_slots);
  const bool report_oob = t == 0 && h == 0 && j == 0;  // one report per token
  int64_t tok = static_cast<int64_t>(blockIdx.x) * kTokPerCta + threadIdx.x / kTpr;
  // Persistent over token groups: the next group's slot and values are
  // loaded before the current group is quantized and stored, so every thread
  // keeps memory requests in flight.
  ItemB<BPT> cur = load_item<D, BPT>(p, src0, tok_stride, tok);
  while (tok < p.num_tokens) {
    const ItemB<BPT> nxt = load_item<D, BPT>(p, src0, tok_stride, tok + step);
    // (uint64) slot < num_slots: a token to write (negative slots wrap high)
    if (static_cast<uint64_t>(cur.slot) < num_slots) {
      // cache row = (page * H + h) * page_size + offset
      const uint32_t page = static_cast<uint32_t>(static_cast<uint64_t>(cur.slot) >> p.log2_page_size);
      const uint32_t off = static_cast<uint32_t>(cur.slot) & pmask;
      const uint64_t r = static_cast<uint64_t>(page) * page_rows + off;
      uint8_t* d = dbase + r * (D / 2);
      uint8_t* sc = sbase + r * kBlocks;
#pragma unroll
      for (int b = 0; b < BPT; ++b) {
        const Quant16 q = quantize16_tab(cur.w[b][0], cur.w[b][1], qc, tab);
        *reinterpret_cast<uint2*>(d + kTpr * 8 * b) = make_uint2(q.lo, q.hi);
        sc[kTpr * b] = static_cast<uint8_t>(q.s8);
      }
    } else if (cur.slot >= 0 && report_oob) {
      atomicOr(p.status, FI_DEV_SLOT_OOB);
    }
    cur = nxt;
    tok += step;
  }
}

// FP8 (E4M3) append: each thread quantizes one 16-element group of one
// (token, tensor, head) row per step (D/16 threads share a row), with the
// next step's slot and values loaded first; 16 codes are one 16-byte store.
template <int D>
__global__ void __launch_bounds__(kAppendThreads, kCtasPerSm)
    fp8_append_kernel(const AppendParams p) {
  constexpr int kTpr = D / 16;
  constexpr int kTokPerCta = kAppendThreads / kTpr;
  grid_dep_wait();  // inputs may come from the previous grid (programmatic launch)
  grid_dep_launch();
  const float ks = p.k_scale_dev ? __ldg(p.k_scale_dev) : p.k_scale_host;
  const float vs = p.v_scale_dev ? __ldg(p.v_scale_dev) : p.v_scale_host;
  if (!scale_ok(ks) || !scale_ok(vs)) {
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
      atomicOr(p.status, (scale_ok(ks) ? 0 : FI_DEV_BAD_K_SCALE) |
                             (scale_ok(vs) ? 0 : FI_DEV_BAD_V_SCALE));
    return;  // uniform across the grid
  }
  const int H = p.num_kv_heads;
  const int t = static_cast<int>(blockIdx.y) >= H ? 1 : 0;  // 0 = K, 1 = V
  const int h = static_cast<int>(blockIdx.y) - t * H;
  const Fp8Consts qc = fp8_consts(t ? vs : ks);
  const int j = threadIdx.x % kTpr;
  const uint32_t hrow = static_cast<uint32_t>(h) << p.log2_page_size;
  uint8_t* const dbase = (t ? p.v_data : p.k_data) + static_cast<uint64_t>(hrow) * D + j * 16;
  const __nv_bfloat16* const src0 = (t ? p.v : p.k) + h * D + j * 16;
  const int64_t tok_stride = t ? p.v_tok_stride : p.k_tok_stride;
  const uint32_t page_rows = static_cast<uint32_t>(H) << p.log2_page_size;
  const uint32_t pmask = (1u << p.log2_page_size) - 1u;
  const uint64_t num_slots = static_cast<uint64_t>(p.num_slots);
  const bool report_oob = t == 0 && h == 0 && j == 0;  // one report per token
  const int64_t step = static_cast<int64_t>(gridDim.x) * kTokPerCta;
  int64_t tok = static_cast<int64_t>(blockIdx.x) * kTokPerCta + threadIdx.x / kTpr;
  ItemB<1> cur = load_item<D, 1>(p, src0, tok_stride, tok);
  while (tok < p.num_tokens) {
    const ItemB<1> nxt = load_item<D, 1>(p, src0, tok_stride, tok + step);
    if (static_cast<uint64_t>(cur.slot) < num_slots) {
      const uint32_t page = static_cast<uint32_t>(static_cast<uint64_t>(cur.slot) >> p.log2_page_size);
      const uint32_t off = static_cast<uint32_t>(cur.slot) & pmask;
      const uint64_t r = static_cast<uint64_t>(page) * page_rows + off;
      *reinterpret_cast<uint4*>(dbase + r * D) = fp8_quantize16(cur.w[0][0], cur.w[0][1], qc);
    } else if (cur.slot >= 0 && report_oob) {
      atomicOr(p.status, FI_DEV_SLOT_OOB);
    }
    cur = nxt;
    tok += step;
  }
}

// Shared memory of the staged kernel (dynamic, 128-byte aligned base):
// [num_stages][stage_bytes] token rows, stage layout [K|V][token][H*D] bf16;
// [2][128] float4 quantizer entries (K, V); full[num_stages],
// empty[num_stages] mbarriers; one abort flag.
struct StagedSmem {
  uint8_t* rows;
  float4* tab;
  uint64_t* full;
  uint64_t* empty;
  int* abort_flag;
};

__host__ __device__ inline int staged_smem_bytes(int num_stages, int stage_bytes) {
  return num_stages * stage_bytes + 2 * 128 * 16 + 2 * num_stages * 8 + 16;
}

__device__ __forceinline__ StagedSmem staged_smem(uint8_t* base, const AppendParams& p) {
  StagedSmem m;
  m.rows = base;
  m.tab = reinterpret_cast<float4*>(base + p.num_stages * p.stage_bytes);
  m.full = reinterpret_cast<uint64_t*>(m.tab + 256);
  m.empty = m.full + p.num_stages;
  m.abort_flag = reinterpret_cast<int*>(m.empty + p.num_stages);
  return m;
}

template <int D>
__global__ void __launch_bounds__(kStagedThreads, 1)
    nvfp4_append_staged_kernel(const AppendParams p) {
  constexpr int kBlocks = D / 16;  // 16-element blocks per head row
  grid_dep_wait();  // inputs may come from the previous grid (see the direct kernel)
  grid_dep_launch();
  const float ks = p.k_scale_dev ? __ldg(p.k_scale_dev) : p.k_scale_host;
  const float vs = p.v_scale_dev ? __ldg(p.v_scale_dev) : p.v_scale_host;
  if (!scale_ok(ks) || !scale_ok(vs)) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      atomicOr(p.status, (scale_ok(ks) ? 0 : FI_DEV_BAD_K_SCALE) |
                             (scale_ok(vs) ? 0 : FI_DEV_BAD_V_SCALE));
    return;  // uniform across the grid
  }
  extern __shared__ __align__(128) uint8_t smem[];
  const StagedSmem m = staged_smem(smem, p);
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int S = p.num_stages;
  const int T = p.tok_per_stage;
  const int64_t groups = (p.num_tokens + T - 1) / T;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(m.full + i, 1);  // the producer's expect_tx arrival
      mbar_init(m.empty + i, kConsumerWarps);
    }
    *m.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const AbortState ab{m.abort_flag, p.status, kWaitNs, FI_DEV_WAIT_TIMEOUT};

  if (tid >= kConsumers) {
    // ---- producer warp: stage g's rows and slots into ring slot it % S
    const bool k_dense = p.k_tok_stride * 2 == p.row_bytes;
    const bool v_dense = p.v_tok_stride * 2 == p.row_bytes;
    int it = 0, st = 0;
    uint32_t ph = 0;  // parity of the ring round of stage `it`
    for (int64_t g = blockIdx.x; g < groups; g += gridDim.x, ++it) {
      if (it >= S && !mbar_wait(m.empty + st, ph ^ 1u, ab)) break;
      const int64_t tok0 = g * T;
      const int64_t left = p.num_tokens - tok0;
      const int nt = left < T ? static_cast<int>(left) : T;
      if (lane == 0) mbar_arrive_expect_tx(m.full + st, static_cast<uint32_t>(nt) * 2 * p.row_bytes);
      __syncwarp();
      uint8_t* dst = m.rows + st * p.stage_bytes;
      if (lane < 2 && (lane ? v_dense : k_dense)) {
        // tokens contiguous in memory: one copy of all nt rows per tensor
        const __nv_bfloat16* src = lane ? p.v + tok0 * p.v_tok_stride : p.k + tok0 * p.k_tok_stride;
        bulk_g2s(dst + lane * T * p.row_bytes, src, static_cast<uint32_t>(nt) * p.row_bytes,
                 m.full + st);
      }
      for (int c = lane; c < 2 * nt; c += 32) {
        const int ten = c >= nt ? 1 : 0;
        const int tl = c - ten * nt;
        if (ten ? v_dense : k_dense) continue;
        const int64_t tok = tok0 + tl;
        const __nv_bfloat16* src = ten ? p.v + tok * p.v_tok_stride : p.k + tok * p.k_tok_stride;
        bulk_g2s(dst + (ten * T + tl) * p.row_bytes, src, p.row_bytes, m.full + st);
      }
      if (++st == S) {
        st = 0;
        ph ^= 1u;
      }
    }
    __syncthreads();
    // After a timeout: wait (bounded) until the copies of the last issued
    // stages have landed before the CTA's shared memory goes away.
    if (*m.abort_flag && lane == 0) {
      volatile int drain_flag = 0;
      const AbortState dab{&drain_flag, nullptr, kDrainWaitNs, 0};
      for (int k = max(0, it - S); k < it; ++k) mbar_wait(m.full + k % S, (k / S) & 1, dab);
    }
    return;
  }

  // ---- consumers: quantizer constants, then the stages
  if (tid < 256) {
    const int t = tid >> 7;
    m.tab[tid] = quant_scale_entry(static_cast<uint32_t>(tid & 127), t ? vs : ks);
  }
  const QuantConsts qk = quant_consts(ks), qv = quant_consts(vs);
  named_bar_sync(1, kConsumers);


  // Each thread owns two blocks of one (tensor, token, head) row of every
  // stage: blocks j and j + kTpr, kTpr = kBlocks / 2 threads per row, so
  // that the token's slot and cache address are worked out once for both.
  // Stage rows are ordered (tensor, token, head).
  constexpr int kTpr = kBlocks / 2;
  const int H = p.num_kv_heads;
  const int TH = T * H;
  const int row = tid / kTpr;
  const int j = tid - row * kTpr;
  const bool use = row < 2 * TH;
  const int ten = row >= TH ? 1 : 0;
  const int tl = (row - ten * TH) / H;
  const int hh = row - ten * TH - tl * H;
  const uint32_t hrow = static_cast<uint32_t>(hh) << p.log2_page_size;
  // code and scale bytes of (page 0, head hh, offset 0, block j)
  uint8_t* const dbase = (ten ? p.v_data : p.k_data) + static_cast<uint64_t>(hrow) * (D / 2) + j * 8;
  uint8_t* const sbase = (ten ? p.v_sf : p.k_sf) + static_cast<uint64_t>(hrow) * kBlocks + j;
  const uint32_t page_rows = static_cast<uint32_t>(H) << p.log2_page_size;
  const QuantConsts qc = ten ? qv : qk;
  const float4* const tab = m.tab + 128 * ten;
  const bool report_oob = ten == 0 && hh == 0 && j == 0;  // one report per token
  const uint32_t soff = static_cast<uint32_t>(row) * (D * 2) + j * 32;  // in a stage
  const uint32_t pmask = (1u << p.log2_page_size) - 1u;
  const uint64_t num_slots = static_cast<uint64_t>(p.num_slots);
  // The slot of this thread's token in the next stage (-1: none), loaded one
  // stage ahead.
  const int64_t tok_step = static_cast<int64_t>(gridDim.x) * T;
  int64_t tok = static_cast<int64_t>(blockIdx.x) * T + tl;
  int64_t slot_next = (use && tok < p.num_tokens) ? __ldg(p.slot_mapping + tok) : -1;
  int st = 0;
  uint32_t ph = 0;
  for (int64_t g = blockIdx.x; g < groups; g += gridDim.x) {
    const int64_t slot = slot_next;
    tok += tok_step;
    slot_next = (use && tok < p.num_tokens) ? __ldg(p.slot_mapping + tok) : -1;
    if (!mbar_wait(m.full + st, ph, ab)) break;
    // (uint64) slot < num_slots: a token to write (negative slots wrap high)
    const bool live = static_cast<uint64_t>(slot) < num_slots;
    uint4 a0, a1, b0, b1;
    if (live) {
      const uint8_t* src = m.rows + st * p.stage_bytes + soff;
      a0 = *reinterpret_cast<const uint4*>(src);
      a1 = *reinterpret_cast<const uint4*>(src + 16);
      b0 = *reinterpret_cast<const uint4*>(src + kTpr * 32);
      b1 = *reinterpret_cast<const uint4*>(src + kTpr * 32 + 16);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(m.empty + st);  // the stage's shared memory is free again
    if (live) {
      const Quant16 qa = quantize16_tab(a0, a1, qc, tab);
      const Quant16 qb = quantize16_tab(b0, b1, qc, tab);
      // cache row = (page * H + hh) * page_size + offset
      const uint32_t page = static_cast<uint32_t>(static_cast<uint64_t>(slot) >> p.log2_page_size);
      const uint32_t off = static_cast<uint32_t>(slot) & pmask;
      const uint64_t r = static_cast<uint64_t>(page) * page_rows + off;
      uint8_t* d = dbase + r * (D / 2);
      uint8_t* sc = sbase + r * kBlocks;
      *reinterpret_cast<uint2*>(d) = make_uint2(qa.lo, qa.hi);
      *reinterpret_cast<uint2*>(d + kTpr * 8) = make_uint2(qb.lo, qb.hi);
      sc[0] = static_cast<uint8_t>(qa.s8);
      sc[kTpr] = static_cast<uint8_t>(qb.s8);
    } else if (slot >= 0 && report_oob) {
      atomicOr(p.status, FI_DEV_SLOT_OOB);
    }
    if (++st == S) {
      st = 0;
      ph ^= 1u;
    }
  }
  __syncthreads();
}

int log2_exact(int v) {
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

}  // namespace

fi_status launch_append(const AppendArgs& a, cudaStream_t stream) {
  AppendParams p;
  p.k = static_cast<const __nv_bfloat16*>(a.k);
  p.v = static_cast<const __nv_bfloat16*>(a.v);
  p.k_tok_stride = a.k_tok_stride;
  p.v_tok_stride = a.v_tok_stride;
  p.k_scale_dev = a.k_scale_dev;
  p.v_scale_dev = a.v_scale_dev;
  p.k_scale_host = a.k_scale_host;
  p.v_scale_host = a.v_scale_host;
  p.slot_mapping = a.slot_mapping;
  p.k_data = a.cache.k_data;
  p.v_data = a.cache.v_data;
  p.k_sf = a.cache.k_sf;
  p.v_sf = a.cache.v_sf;
  p.num_kv_heads = a.cache.num_kv_heads;
  p.log2_page_size = log2_exact(a.cache.page_size);
  p.num_tokens = a.num_tokens;
  p.num_slots = static_cast<int64_t>(a.cache.num_pages) * a.cache.page_size;
  p.status = a.status;
  const int D = a.cache.head_dim;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FI_ERR_CUDA;
  if (a.kv_format == 1) {
    const int64_t gy = 2 * static_cast<int64_t>(a.cache.num_kv_heads);
    if (gy > 65535) return FI_ERR_INVALID_ARGUMENT;
    const int tpc = kAppendThreads / (D / 16);
    const int64_t groups = (a.num_tokens + tpc - 1) / tpc;
    const int64_t want = (static_cast<int64_t>(sms) * kCtasPerSm + gy - 1) / gy;
    const int64_t per_cta = (groups + want - 1) / want;
    const dim3 grid(static_cast<unsigned>(std::max<int64_t>(1, (groups + per_cta - 1) / per_cta)),
                    static_cast<unsigned>(gy));
    void (*kern)(AppendParams) = D == 128 ? fp8_append_kernel<128> : fp8_append_kernel<64>;
    return launch_pdl(kern, grid, dim3(kAppendThreads), 0, stream, p);
  }
  // Staged kernel for large appends whose (token, K|V) row pair fits a stage;
  // the direct kernel otherwise (its many resident warps start streaming at
  // once, which short appends need more than deep staging).
  const int64_t row_bytes = static_cast<int64_t>(a.cache.num_kv_heads) * D * 2;
  if (2 * row_bytes <= kStageBytes && a.num_tokens >= kStagedMinTokens) {
    p.row_bytes = static_cast<int32_t>(row_bytes);
    p.tok_per_stage = static_cast<int32_t>(std::min<int64_t>(kMaxTokPerStage, kStageBytes / (2 * row_bytes)));
    p.stage_bytes = p.tok_per_stage * 2 * p.row_bytes;
    p.num_stages = kMaxStages;
    while (p.num_stages > 2 &&
           staged_smem_bytes(p.num_stages, p.stage_bytes) > kSmemBudget)
      --p.num_stages;
    const int smem = staged_smem_bytes(p.num_stages, p.stage_bytes);
    const int64_t groups = (a.num_tokens + p.tok_per_stage - 1) / p.tok_per_stage;
    const unsigned grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(groups, sms)));
    void (*kern)(AppendParams) =
        D == 128 ? nvfp4_append_staged_kernel<128> : nvfp4_append_staged_kernel<64>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return FI_ERR_CUDA;
    return launch_pdl(kern, dim3(grid), dim3(kStagedThreads), smem, stream, p);
  }
  const int tok_per_cta = kAppendThreads / (D / 16 / kDirectBlocksPerThread);
  const int64_t groups = (a.num_tokens + tok_per_cta - 1) / tok_per_cta;
  const int64_t gy = 2 * static_cast<int64_t>(a.cache.num_kv_heads);
  if (gy > 65535) return FI_ERR_INVALID_ARGUMENT;
  // Persistent grid: about kCtasPerSm resident CTAs on every SM in total,
  // spread over the gy (tensor, head) rows, each looping over token groups.
  const int64_t want = (static_cast<int64_t>(sms) * kCtasPerSm + gy - 1) / gy;
  // as many groups per CTA as `want` CTAs need, spread evenly
  const int64_t per_cta = (groups + want - 1) / want;
  const int64_t gx = std::max<int64_t>(1, (groups + per_cta - 1) / per_cta);
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  void (*kern)(AppendParams) = D == 128 ? nvfp4_append_kernel<128, kDirectBlocksPerThread>
                                         : nvfp4_append_kernel<64, kDirectBlocksPerThread>;
  return launch_pdl(kern, grid, dim3(kAppendThreads), 0, stream, p);
}

}  // namespace fi
