// api.cu — the extern "C" entry points of libfi_nvfp4.so (declared and
// documented in include/fi_nvfp4.h): argument checks on the host, then the
// kernels on the caller's stream.  Nothing here reads device memory except
// fi_device_status().
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace fi {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool cache_ok(const fi_nvfp4_cache* c, int kv_format) {
  if (!c || !c->k_data || !c->v_data) return false;
  if (!aligned16(c->k_data) || !aligned16(c->v_data)) return false;
  if (kv_format == 0 &&
      (!c->k_sf || !c->v_sf || !aligned16(c->k_sf) || !aligned16(c->v_sf)))
    return false;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0) return false;
  return true;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

fi_status cache_supported(const fi_nvfp4_cache* c) {
  if (c->head_dim != 64 && c->head_dim != 128) return FI_ERR_UNSUPPORTED;
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64 && c->page_size != 128)
    return FI_ERR_UNSUPPORTED;
  return FI_OK;
}

// The FP8 cache as the common cache description (no block scales).
fi_nvfp4_cache fp8_view(const fi_fp8_cache* c) {
  fi_nvfp4_cache v{};
  v.k_data = c->k_data;
  v.v_data = c->v_data;
  v.k_sf = nullptr;
  v.v_sf = nullptr;
  v.k_scale = c->k_scale;
  v.v_scale = c->v_scale;
  v.num_pages = c->num_pages;
  v.page_size = c->page_size;
  v.num_kv_heads = c->num_kv_heads;
  v.head_dim = c->head_dim;
  return v;
}

fi_status append_common(fi_context* ctx, const void* k, const void* v, int64_t num_tokens,
                        int64_t ks, int64_t vs, const float* kd, const float* vd, float kh,
                        float vh, const int64_t* slots, const fi_nvfp4_cache* cache,
                        void* stream, int kv_format = 0) {
  if (!ctx || !cache_ok(cache, kv_format) || num_tokens < 0) return FI_ERR_INVALID_ARGUMENT;
  const fi_status sup = cache_supported(cache);
  if (sup != FI_OK) return sup;
  if (num_tokens == 0) return FI_OK;  // nothing launched, nothing checked
  if (!k || !v || !slots || !aligned16(k) || !aligned16(v)) return FI_ERR_INVALID_ARGUMENT;
  const int64_t row = static_cast<int64_t>(cache->num_kv_heads) * cache->head_dim;
  if (ks < row || vs < row || ks % 8 != 0 || vs % 8 != 0) return FI_ERR_INVALID_ARGUMENT;
  AppendArgs a;
  a.k = k;
  a.v = v;
  a.num_tokens = num_tokens;
  a.k_tok_stride = ks;
  a.v_tok_stride = vs;
  a.k_scale_dev = kd;
  a.v_scale_dev = vd;
  a.k_scale_host = kh;
  a.v_scale_host = vh;
  a.slot_mapping = slots;
  a.cache = *cache;
  a.kv_format = kv_format;
  a.status = ctx->status_dev;
  return launch_append(a, static_cast<cudaStream_t>(stream));
}

}  // namespace

bool encode_tensor_map_3d_bf16(void* map_out, const void* base, uint64_t dim0, uint64_t dim1,
                               uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                               uint32_t box0, uint32_t box1, uint32_t box2) {
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return false;
  cuuint64_t dims[3] = {dim0, dim1, dim2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(reinterpret_cast<CUtensorMap*>(map_out),
                              CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace fi

// ------------------------------------------------------------------ plans
struct fi_plan {
  fi_context* ctx = nullptr;
  fi::HostPlan host;
  bool planned = false;
  // device copies: qo_indptr, kv_indptr, work list (int32)
  int32_t* dev = nullptr;
  size_t dev_words = 0;
  // double-buffered pinned staging
  int32_t* pinned[2] = {nullptr, nullptr};
  size_t pinned_words[2] = {0, 0};
  cudaEvent_t copied[2] = {nullptr, nullptr};
  bool copy_pending[2] = {false, false};
  int next = 0;
  const int32_t* page_table = nullptr;
  int32_t page_table_stride = 0;
  size_t off_kv = 0, off_work = 0, off_slot_units = 0, off_slot_begin = 0;
  // decode plans: partial results of sequences split over several chunks
  float* part = nullptr;
  size_t part_floats = 0;
};

extern "C" {

fi_status fi_context_create(fi_context** out) {
  if (!out) return FI_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_CUDA;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FI_ERR_UNSUPPORTED;
  fi_context* c = new fi_context;
  c->device = dev;
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev);
  int l2 = 0;
  cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
  c->l2_bytes = l2;
  if (cudaMalloc(&c->status_dev, 64) != cudaSuccess) {
    delete c;
    return FI_ERR_OUT_OF_MEMORY;
  }
  if (cudaMemset(c->status_dev, 0, 64) != cudaSuccess) {
    cudaFree(c->status_dev);
    delete c;
    return FI_ERR_CUDA;
  }
  *out = c;
  return FI_OK;
}

fi_status fi_context_destroy(fi_context* ctx) {
  if (!ctx) return FI_ERR_INVALID_ARGUMENT;
  cudaDeviceSynchronize();
  cudaFree(ctx->status_dev);
  delete ctx;
  return FI_OK;
}

fi_status fi_nvfp4_append(fi_context* ctx, const void* k_dev, const void* v_dev,
                          int64_t num_tokens, int64_t k_tok_stride, int64_t v_tok_stride,
                          const float* k_scale_dev, const float* v_scale_dev,
                          const int64_t* slot_mapping_dev, const fi_nvfp4_cache* cache,
                          void* stream) {
  if (!k_scale_dev || !v_scale_dev) return FI_ERR_INVALID_ARGUMENT;
  return fi::append_common(ctx, k_dev, v_dev, num_tokens, k_tok_stride, v_tok_stride,
                           k_scale_dev, v_scale_dev, 0.0f, 0.0f, slot_mapping_dev, cache, stream);
}

fi_status fi_fp8_append(fi_context* ctx, const void* k_dev, const void* v_dev,
                        int64_t num_tokens, int64_t k_tok_stride, int64_t v_tok_stride,
                        const float* k_scale_dev, const float* v_scale_dev,
                        const int64_t* slot_mapping_dev, const fi_fp8_cache* cache,
                        void* stream) {
  if (!k_scale_dev || !v_scale_dev || !cache) return FI_ERR_INVALID_ARGUMENT;
  const fi_nvfp4_cache view = fi::fp8_view(cache);
  return fi::append_common(ctx, k_dev, v_dev, num_tokens, k_tok_stride, v_tok_stride,
                           k_scale_dev, v_scale_dev, 0.0f, 0.0f, slot_mapping_dev, &view, stream,
                           1);
}

fi_status fi_nvfp4_append_host_scale(fi_context* ctx, const void* k_dev, const void* v_dev,
                                     int64_t num_tokens, int64_t k_tok_stride,
                                     int64_t v_tok_stride, float k_scale, float v_scale,
                                     const int64_t* slot_mapping_dev,
                                     const fi_nvfp4_cache* cache, void* stream) {
  if (!(std::isfinite(k_scale) && k_scale > 0.0f) || !(std::isfinite(v_scale) && v_scale > 0.0f))
    return FI_ERR_BAD_SCALE;
  return fi::append_common(ctx, k_dev, v_dev, num_tokens, k_tok_stride, v_tok_stride, nullptr,
                           nullptr, k_scale, v_scale, slot_mapping_dev, cache, stream);
}

fi_status fi_plan_create(fi_context* ctx, fi_plan** out) {
  if (!ctx || !out) return FI_ERR_INVALID_ARGUMENT;
  fi_plan* p = new fi_plan;
  p->ctx = ctx;
  for (int i = 0; i < 2; ++i) {
    if (cudaEventCreateWithFlags(&p->copied[i], cudaEventDisableTiming) != cudaSuccess) {
      delete p;
      return FI_ERR_CUDA;
    }
  }
  *out = p;
  return FI_OK;
}

fi_status fi_plan_destroy(fi_plan* plan) {
  if (!plan) return FI_ERR_INVALID_ARGUMENT;
  cudaDeviceSynchronize();
  if (plan->dev) cudaFree(plan->dev);
  if (plan->part) cudaFree(plan->part);
  for (int i = 0; i < 2; ++i) {
    if (plan->pinned[i]) cudaFreeHost(plan->pinned[i]);
    if (plan->copied[i]) cudaEventDestroy(plan->copied[i]);
  }
  delete plan;
  return FI_OK;
}

}  // extern "C"

namespace {
// Copies qo_indptr | kv_indptr | work list | slot units | slot begins of the
// plan's host description to plan-owned device memory (see fi_prefill_plan).
fi_status upload_plan(fi_plan* plan, const int32_t* qo_indptr_host,
                      const int32_t* kv_indptr_host, int32_t batch, void* stream) {
  // Device copy: qo_indptr | kv_indptr | work list | slot units | slot begins.
  const size_t nb = static_cast<size_t>(batch) + 1;
  plan->off_kv = nb;
  plan->off_work = (2 * nb + 3) & ~static_cast<size_t>(3);  // 16-byte aligned work list
  plan->off_slot_units = plan->off_work + plan->host.work.size();
  plan->off_slot_begin = plan->off_slot_units + plan->host.slot_units.size();
  const size_t words = plan->off_slot_begin + plan->host.slot_begin.size();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (words > plan->dev_words) {
    if (plan->dev) cudaFree(plan->dev);  // growth only: amortized
    plan->dev = nullptr;
    plan->dev_words = 0;
    const size_t cap = std::max<size_t>(words, 1024) * 3 / 2;
    if (cudaMalloc(&plan->dev, cap * sizeof(int32_t)) != cudaSuccess) return FI_ERR_OUT_OF_MEMORY;
    plan->dev_words = cap;
  }
  const int b = plan->next;
  plan->next ^= 1;
  if (plan->copy_pending[b]) {
    // the copy issued from this staging buffer two plans ago
    if (cudaEventSynchronize(plan->copied[b]) != cudaSuccess) return FI_ERR_CUDA;
    plan->copy_pending[b] = false;
  }
  if (words > plan->pinned_words[b]) {
    if (plan->pinned[b]) cudaFreeHost(plan->pinned[b]);
    plan->pinned[b] = nullptr;
    plan->pinned_words[b] = 0;
    const size_t cap = std::max<size_t>(words, 1024) * 3 / 2;
    if (cudaMallocHost(&plan->pinned[b], cap * sizeof(int32_t)) != cudaSuccess)
      return FI_ERR_OUT_OF_MEMORY;
    plan->pinned_words[b] = cap;
  }
  int32_t* h = plan->pinned[b];
  if (batch >= 0) {
    std::memcpy(h, qo_indptr_host, nb * sizeof(int32_t));
    std::memcpy(h + plan->off_kv, kv_indptr_host, nb * sizeof(int32_t));
  }
  if (!plan->host.work.empty())
    std::memcpy(h + plan->off_work, plan->host.work.data(),
                plan->host.work.size() * sizeof(int32_t));
  if (!plan->host.slot_units.empty())
    std::memcpy(h + plan->off_slot_units, plan->host.slot_units.data(),
                plan->host.slot_units.size() * sizeof(int32_t));
  if (!plan->host.slot_begin.empty())
    std::memcpy(h + plan->off_slot_begin, plan->host.slot_begin.data(),
                plan->host.slot_begin.size() * sizeof(int32_t));
  if (cudaMemcpyAsync(plan->dev, h, words * sizeof(int32_t), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return FI_ERR_CUDA;
  if (cudaEventRecord(plan->copied[b], s) != cudaSuccess) return FI_ERR_CUDA;
  plan->copy_pending[b] = true;
  plan->planned = true;
  return FI_OK;
}
}  // namespace

extern "C" {

fi_status fi_prefill_plan(fi_plan* plan, const int32_t* qo_indptr_host,
                          const int32_t* kv_indptr_host, int32_t batch,
                          const int32_t* page_table_dev, int32_t page_table_stride,
                          int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t page_size, float sm_scale, const fi_plan_options* opts,
                          void* stream) {
  if (!plan) return FI_ERR_INVALID_ARGUMENT;
  plan->planned = false;
  if (batch > 0 && (!page_table_dev || page_table_stride <= 0)) return FI_ERR_INVALID_ARGUMENT;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale))
    sm_scale = 1.0f / std::sqrt(static_cast<float>(head_dim));
  const fi_context* ctx = plan->ctx;
  const int64_t l2 = (opts && opts->l2_bytes > 0) ? opts->l2_bytes : ctx->l2_bytes;
  fi_status st = fi::plan_host(qo_indptr_host, kv_indptr_host, batch, num_qo_heads, num_kv_heads,
                               head_dim, page_size, sm_scale, l2, ctx->num_sms, opts,
                               &plan->host);
  if (st != FI_OK) return st;
  // page table rows must cover every sequence's pages
  if (batch > 0 && (plan->host.info.max_kv_len + page_size - 1) / page_size > page_table_stride)
    return FI_ERR_INVALID_ARGUMENT;
  plan->page_table = page_table_dev;
  plan->page_table_stride = page_table_stride;

  return upload_plan(plan, qo_indptr_host, kv_indptr_host, batch, stream);
}

fi_status fi_decode_plan(fi_plan* plan, const int32_t* qo_indptr_host,
                         const int32_t* kv_indptr_host, int32_t batch,
                         const int32_t* page_table_dev, int32_t page_table_stride,
                         int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t page_size, float sm_scale, void* stream) {
  if (!plan) return FI_ERR_INVALID_ARGUMENT;
  plan->planned = false;
  if (batch > 0 && (!page_table_dev || page_table_stride <= 0)) return FI_ERR_INVALID_ARGUMENT;
  if (!(sm_scale > 0.0f) || !std::isfinite(sm_scale))
    sm_scale = 1.0f / std::sqrt(static_cast<float>(head_dim));
  fi::HostPlan& P = plan->host;
  fi_status st = fi::plan_decode_host(qo_indptr_host, kv_indptr_host, batch, num_qo_heads,
                                      num_kv_heads, head_dim, page_size, sm_scale,
                                      plan->ctx->num_sms, &P);
  if (st != FI_OK) return st;
  if (batch > 0 && (P.info.max_kv_len + page_size - 1) / page_size > page_table_stride)
    return FI_ERR_INVALID_ARGUMENT;
  plan->page_table = page_table_dev;
  plan->page_table_stride = page_table_stride;
  // the pieces, merges and warp offsets travel in the work-list, slot-unit
  // and slot-begin regions
  P.work.assign(P.dec_units.begin(), P.dec_units.end());
  P.slot_units.assign(P.dec_merges.begin(), P.dec_merges.end());
  P.slot_begin.assign(P.dec_warp_off.begin(), P.dec_warp_off.end());
  const size_t need = static_cast<size_t>(P.dec_parts) * P.dec_rows * (head_dim + 2);
  if (need > plan->part_floats) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return FI_ERR_CUDA;  // earlier runs use it
    if (plan->part) cudaFree(plan->part);
    plan->part = nullptr;
    plan->part_floats = 0;
    const size_t cap = need * 3 / 2;
    if (cudaMalloc(&plan->part, cap * sizeof(float)) != cudaSuccess) return FI_ERR_OUT_OF_MEMORY;
    plan->part_floats = cap;
  }
  return upload_plan(plan, qo_indptr_host, kv_indptr_host, batch, stream);
}

fi_status fi_decode_run(const fi_plan* plan, const void* q_dev, const fi_nvfp4_cache* cache,
                        void* out_dev, float* lse_dev, void* stream) {
  if (!plan || !plan->planned || !plan->host.decode || !fi::cache_ok(cache, 0) ||
      !cache->k_scale || !cache->v_scale)
    return FI_ERR_INVALID_ARGUMENT;
  const fi::HostPlan& P = plan->host;
  if (cache->head_dim != P.head_dim || cache->page_size != P.page_size ||
      cache->num_kv_heads != P.num_kv_heads)
    return FI_ERR_INVALID_ARGUMENT;
  if (P.info.num_units == 0) return FI_OK;
  if (!q_dev || !out_dev || !fi::aligned16(q_dev) || !fi::aligned16(out_dev))
    return FI_ERR_INVALID_ARGUMENT;
  fi::DecodeArgs a;
  a.plan = &P;
  a.qo_indptr_dev = plan->dev;
  a.kv_indptr_dev = plan->dev + plan->off_kv;
  a.units_dev = plan->dev + plan->off_work;
  a.merges_dev = plan->dev + plan->off_slot_units;
  a.warp_off_dev = plan->dev + plan->off_slot_begin;
  a.part = plan->part;
  a.page_table = plan->page_table;
  a.page_table_stride = plan->page_table_stride;
  a.q = q_dev;
  a.cache = *cache;
  a.out = out_dev;
  a.lse = lse_dev;
  a.status = plan->ctx->status_dev;
  return fi::launch_decode(a, static_cast<cudaStream_t>(stream));
}

fi_status fi_plan_get_info(const fi_plan* plan, fi_plan_info* info) {
  if (!plan || !info || !plan->planned) return FI_ERR_INVALID_ARGUMENT;
  *info = plan->host.info;
  return FI_OK;
}

namespace fi {
namespace {
fi_status run_common(const fi_plan* plan, const void* q_dev, const fi_nvfp4_cache* cache,
                     int kv_format, void* out_dev, float* lse_dev, void* stream);
}  // namespace
}  // namespace fi

fi_status fi_prefill_run(const fi_plan* plan, const void* q_dev, const fi_nvfp4_cache* cache,
                         void* out_dev, float* lse_dev, void* stream) {
  return fi::run_common(plan, q_dev, cache, 0, out_dev, lse_dev, stream);
}

fi_status fi_prefill_run_fp8(const fi_plan* plan, const void* q_dev, const fi_fp8_cache* cache,
                             void* out_dev, float* lse_dev, void* stream) {
  if (!cache) return FI_ERR_INVALID_ARGUMENT;
  const fi_nvfp4_cache view = fi::fp8_view(cache);
  return fi::run_common(plan, q_dev, &view, 1, out_dev, lse_dev, stream);
}

namespace fi {
namespace {
fi_status run_common(const fi_plan* plan, const void* q_dev, const fi_nvfp4_cache* cache,
                     int kv_format, void* out_dev, float* lse_dev, void* stream) {
  if (!plan || !plan->planned || !fi::cache_ok(cache, kv_format) || !cache->k_scale ||
      !cache->v_scale || plan->host.kv_format != kv_format || plan->host.decode)
    return FI_ERR_INVALID_ARGUMENT;
  const fi::HostPlan& P = plan->host;
  if (cache->head_dim != P.head_dim || cache->page_size != P.page_size ||
      cache->num_kv_heads != P.num_kv_heads)
    return FI_ERR_INVALID_ARGUMENT;
  if (P.info.num_units == 0) return FI_OK;
  if (!q_dev || !out_dev || !fi::aligned16(q_dev) || !fi::aligned16(out_dev))
    return FI_ERR_INVALID_ARGUMENT;
  fi::PrefillArgs a;
  a.plan = &P;
  a.qo_indptr_dev = plan->dev;
  a.kv_indptr_dev = plan->dev + plan->off_kv;
  a.work_dev = P.work.empty() ? nullptr : plan->dev + plan->off_work;
  const bool balanced = !P.slot_units.empty();
  a.slot_units_dev = balanced ? plan->dev + plan->off_slot_units : nullptr;
  a.slot_begin_dev = balanced ? plan->dev + plan->off_slot_begin : nullptr;
  a.num_slots = balanced ? static_cast<int32_t>(P.slot_begin.size()) - 1 : 0;
  a.page_table = plan->page_table;
  a.page_table_stride = plan->page_table_stride;
  a.q = q_dev;
  a.cache = *cache;
  a.out = out_dev;
  a.lse = lse_dev;
  a.status = plan->ctx->status_dev;
  return fi::launch_prefill(a, static_cast<cudaStream_t>(stream));
}
}  // namespace
}  // namespace fi

fi_status fi_device_status(fi_context* ctx, void* stream, int32_t* bits, int32_t reset) {
  if (!ctx || !bits) return FI_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FI_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, ctx->status_dev, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FI_ERR_CUDA;
  *bits = v;
  if (reset && cudaMemset(ctx->status_dev, 0, sizeof(int32_t)) != cudaSuccess) return FI_ERR_CUDA;
  return FI_OK;
}

const char* fi_status_string(fi_status status) {
  switch (status) {
    case FI_OK: return "ok";
    case FI_ERR_INVALID_ARGUMENT: return "invalid argument";
    case FI_ERR_BAD_SCALE: return "global decode scale must be positive and finite";
    case FI_ERR_UNSUPPORTED: return "unsupported head_dim, page_size or device";
    case FI_ERR_CUDA: return "CUDA runtime error";
    case FI_ERR_OUT_OF_MEMORY: return "out of memory";
    case FI_ERR_SCRATCH_TOO_SMALL:
      return "batch too large for the no-allocation prefill's fixed scratch";
    default: return "unknown status";
  }
}

int32_t fi_version(void) { return 201; }

}  // extern "C"
