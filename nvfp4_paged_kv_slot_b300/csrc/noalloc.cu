// noalloc.cu — fi_prefill_noalloc: plan and run the causal NVFP4 prefill in
// one call without allocating any memory, for callers that cannot allocate:
// a serving engine that reserves all device memory for its KV cache and
// activations up front and forbids allocations while it serves, or a plugin
// whose enqueue callback must not allocate (the host framework owns memory).
//
// The prefill kernel reads a small amount of global scratch besides its
// inputs and outputs: copies of qo_indptr / kv_indptr and, for ragged
// batches, the list of work units.  fi_prefill_plan keeps these in memory the
// plan allocates; here they live in one file-scope __device__ array of fixed
// size that every GPU loading the library holds until the process exits.
#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace fi {

bool cache_ok(const fi_nvfp4_cache* c, int kv_format = 0);
bool aligned16(const void* p);

namespace {

// 2 MiB of scratch: status word (+ padding), qo_indptr, kv_indptr, work list.
constexpr int64_t kScratchWords = 1 << 19;
constexpr int64_t kStatusWords = 4;
constexpr int kMaxDevices = 64;
constexpr int kChunkItems = 1024;  // work-list items staged on the host stack per copy

static __device__ __align__(256) int32_t g_prefill_scratch[kScratchWords];

std::mutex g_setup_mutex;
int32_t* g_scratch_dev[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress, with that device current);
// in host code the array's name is only a host-side stand-in.
fi_status scratch_address(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FI_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || !p) return FI_ERR_CUDA;
    g_scratch_dev[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_dev[dev];
  return FI_OK;
}

int32_t kv_tiles_of(int32_t qt, int32_t qo_len, int32_t kv_len) {
  const int32_t last_row = std::min(qo_len, (qt + 1) * kTileQ) - 1;
  return (last_row + (kv_len - qo_len)) / kTileKV + 1;
}

}  // namespace
}  // namespace fi

extern "C" fi_status fi_prefill_noalloc(const int32_t* qo_indptr_host,
                                        const int32_t* kv_indptr_host, int32_t batch,
                                        const int32_t* page_table_dev,
                                        int32_t page_table_stride, int32_t num_qo_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t page_size, float sm_scale, const void* q_dev,
                                        const fi_nvfp4_cache* cache, void* out_dev,
                                        float* lse_dev, int32_t* status_dev, void* stream) {
  using namespace fi;
  // ---- arguments (the same rules as fi_prefill_plan and fi_prefill_run)
  if (batch < 0 || (batch > 0 && (!qo_indptr_host || !kv_indptr_host)))
    return FI_ERR_INVALID_ARGUMENT;
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return FI_ERR_INVALID_ARGUMENT;
  if (head_dim != 64 && head_dim != 128) return FI_ERR_UNSUPPORTED;
  if (page_size != 16 && page_size != 32 && page_size != 64 && page_size != 128)
    return FI_ERR_UNSUPPORTED;
  if (!cache_ok(cache) || !cache->k_scale || !cache->v_scale) return FI_ERR_INVALID_ARGUMENT;
  if (cache->head_dim != head_dim || cache->page_size != page_size ||
      cache->num_kv_heads != num_kv_heads)
    return FI_ERR_INVALID_ARGUMENT;
  if (batch > 0 && (qo_indptr_host[0] != 0 || kv_indptr_host[0] != 0))
    return FI_ERR_INVALID_ARGUMENT;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale))
    sm_scale = 1.0f / std::sqrt(static_cast<float>(head_dim));

  HostPlan P;  // its work vector stays empty: the list goes straight to scratch
  P.num_qo_heads = num_qo_heads;
  P.num_kv_heads = num_kv_heads;
  P.head_dim = head_dim;
  P.page_size = page_size;
  P.group = num_qo_heads / num_kv_heads;
  P.sm_scale = sm_scale;
  int32_t max_qo = 0, max_kv = 0;
  int64_t units_ragged = 0;
  fi_plan_info& I = P.info;
  I.heads_per_cta = (P.group % 2 == 0) ? 2 : 1;
  // groups of a multiple of 4 query heads on CTA pairs, as fi_prefill_plan
  // chooses by default
  P.pair = P.group % 4 == 0;
  I.ctas_per_unit = P.pair ? 2 : 1;
  P.units_per_kv_head = P.group / (I.heads_per_cta * I.ctas_per_unit);
  I.head_units = num_kv_heads * P.units_per_kv_head;
  for (int32_t b = 0; b < batch; ++b) {
    const int32_t qo = qo_indptr_host[b + 1] - qo_indptr_host[b];
    const int32_t kv = kv_indptr_host[b + 1] - kv_indptr_host[b];
    if (qo < 0 || kv < 0 || qo > kv) return FI_ERR_INVALID_ARGUMENT;
    max_qo = std::max(max_qo, qo);
    max_kv = std::max(max_kv, kv);
    units_ragged += static_cast<int64_t>((qo + kTileQ - 1) / kTileQ) * I.head_units;
  }
  I.batch = batch;
  I.max_qo_len = max_qo;
  I.max_kv_len = max_kv;
  I.total_qo_len = batch > 0 ? qo_indptr_host[batch] : 0;
  I.total_kv_len = batch > 0 ? kv_indptr_host[batch] : 0;
  I.is_uniform = (I.total_qo_len == static_cast<int64_t>(batch) * max_qo &&
                  I.total_kv_len == static_cast<int64_t>(batch) * max_kv)
                     ? 1
                     : 0;
  I.q_tiles = (max_qo + kTileQ - 1) / kTileQ;
  I.kv_bytes = I.total_kv_len * num_kv_heads * 2 * (head_dim / 2 + head_dim / 16);
  int dev = 0, l2 = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FI_ERR_CUDA;
  I.global_reverse = (I.is_uniform || 2 * I.kv_bytes <= l2) ? 1 : 0;  // as fi_prefill_plan
  if (I.is_uniform) {
    P.uniform_qo_len = max_qo;
    P.uniform_kv_len = max_kv;
    I.num_units = static_cast<int64_t>(batch) * I.head_units * I.q_tiles;
  } else {
    I.num_units = units_ragged;
  }
  I.num_ctas = static_cast<int32_t>(
      std::min<int64_t>(I.num_units * I.ctas_per_unit, std::max(sms, I.ctas_per_unit)));
  if (P.pair) I.num_ctas &= ~1;
  if (batch > 0 && (!page_table_dev || page_table_stride <= 0 ||
                    (max_kv + page_size - 1) / page_size > page_table_stride))
    return FI_ERR_INVALID_ARGUMENT;
  if (I.num_units == 0) return FI_OK;
  if (!q_dev || !out_dev || !aligned16(q_dev) || !aligned16(out_dev))
    return FI_ERR_INVALID_ARGUMENT;

  // ---- scratch layout: status | qo_indptr | kv_indptr | work list (16 B aligned)
  const int64_t nb = static_cast<int64_t>(batch) + 1;
  const int64_t off_qo = kStatusWords;
  const int64_t off_kv = off_qo + nb;
  const int64_t off_work = (off_kv + nb + 3) & ~static_cast<int64_t>(3);
  const int64_t words = off_work + (I.is_uniform ? 0 : 4 * (I.num_units / I.head_units));
  if (words > kScratchWords) return FI_ERR_SCRATCH_TOO_SMALL;

  int32_t* scratch = nullptr;
  fi_status st = scratch_address(&scratch);
  if (st != FI_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The copies and the kernel are enqueued on `stream`, so stream order puts
  // every copy after the stream's earlier work (an earlier call's kernel has
  // finished reading the scratch) and before this call's kernel.  The work
  // list is staged in a stack buffer: pageable memory, whose copy has read
  // the source when cudaMemcpyAsync returns, so the buffer may be refilled at
  // once.  The caller's indptr arrays are read when the stream reaches their
  // copies if they are page-locked (the header says so).
  if (!status_dev && cudaMemsetAsync(scratch, 0, kStatusWords * sizeof(int32_t), s) != cudaSuccess)
    return FI_ERR_CUDA;
  if (cudaMemcpyAsync(scratch + off_qo, qo_indptr_host, nb * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(scratch + off_kv, kv_indptr_host, nb * sizeof(int32_t),
                      cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FI_ERR_CUDA;
  if (!I.is_uniform) {
    // Ragged: one item per (sequence, q-tile), sequences in order, q-tiles
    // from the last (heaviest) to the first (the head units of an item are
    // consecutive units), staged through a fixed host buffer.
    int32_t chunk[4 * kChunkItems];
    int64_t done = 0;
    int n = 0;
    for (int32_t b = 0; b < batch; ++b) {
      const int32_t qo = qo_indptr_host[b + 1] - qo_indptr_host[b];
      const int32_t kv = kv_indptr_host[b + 1] - kv_indptr_host[b];
      const int32_t tiles = (qo + kTileQ - 1) / kTileQ;
      for (int32_t qt = tiles - 1; qt >= 0; --qt) {
        chunk[4 * n + 0] = b;
        chunk[4 * n + 1] = qt;
        chunk[4 * n + 2] = kv_tiles_of(qt, qo, kv);
        chunk[4 * n + 3] = 0;
        if (++n == kChunkItems) {
          if (cudaMemcpyAsync(scratch + off_work + 4 * done, chunk,
                              static_cast<size_t>(n) * 4 * sizeof(int32_t),
                              cudaMemcpyHostToDevice, s) != cudaSuccess)
            return FI_ERR_CUDA;
          done += n;
          n = 0;
        }
      }
    }
    if (n > 0 && cudaMemcpyAsync(scratch + off_work + 4 * done, chunk,
                                 static_cast<size_t>(n) * 4 * sizeof(int32_t),
                                 cudaMemcpyHostToDevice, s) != cudaSuccess)
      return FI_ERR_CUDA;
  }

  PrefillArgs a;
  a.plan = &P;
  a.qo_indptr_dev = scratch + off_qo;
  a.kv_indptr_dev = scratch + off_kv;
  a.work_dev = I.is_uniform ? nullptr : scratch + off_work;
  a.slot_units_dev = nullptr;  // units dealt round-robin
  a.slot_begin_dev = nullptr;
  a.num_slots = 0;
  a.page_table = page_table_dev;
  a.page_table_stride = page_table_stride;
  a.q = q_dev;
  a.cache = *cache;
  a.out = out_dev;
  a.lse = lse_dev;
  a.status = status_dev ? status_dev : scratch;
  return launch_prefill(a, s);
}
