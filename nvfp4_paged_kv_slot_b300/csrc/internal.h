// internal.h — declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "fi_nvfp4.h"

struct fi_context {
  int device = 0;
  int32_t* status_dev = nullptr;  // device status word (FI_DEV_* bits)
  int num_sms = 0;
  int64_t l2_bytes = 0;
};

namespace fi {

constexpr int kTileQ = 128;   // query rows per tile (MMA M)
constexpr int kTileKV = 128;  // keys per KV tile (MMA N of QK^T, K of PV)

// ---- append ----------------------------------------------------------------
struct AppendArgs {
  const void* k;
  const void* v;
  int64_t num_tokens;
  int64_t k_tok_stride;
  int64_t v_tok_stride;
  const float* k_scale_dev;  // null: use the host values below
  const float* v_scale_dev;
  float k_scale_host;
  float v_scale_host;
  const int64_t* slot_mapping;
  fi_nvfp4_cache cache;   // FP8: k_sf / v_sf null
  int32_t kv_format;      // 0 NVFP4, 1 FP8 (E4M3, one code per element)
  int32_t* status;
};
fi_status launch_append(const AppendArgs& a, cudaStream_t stream);

// Launches `kern` as a programmatic dependent of the stream's previous grid:
// it may start while that grid finishes and waits for it with
// griddepcontrol.wait before touching memory (extra attributes, e.g. a
// cluster shape, are added by the caller through `more`).
template <typename Params>
fi_status launch_pdl(void (*kern)(Params), dim3 grid, dim3 block, int smem, cudaStream_t stream,
                     const Params& p, const cudaLaunchAttribute* more = nullptr, int n_more = 0) {
  cudaLaunchAttribute attrs[4];
  int n = 0;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  for (int k = 0; k < n_more && n < 4; ++k) attrs[n++] = more[k];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = static_cast<unsigned>(n);
  if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return FI_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

// ---- planner ---------------------------------------------------------------
struct HostPlan {
  fi_plan_info info{};
  int32_t num_qo_heads = 0, num_kv_heads = 0, head_dim = 0, page_size = 0;
  int32_t group = 0;              // num_qo_heads / num_kv_heads
  int32_t units_per_kv_head = 0;  // group / heads_per_cta
  int32_t uniform_qo_len = 0, uniform_kv_len = 0;
  bool pair = false;              // units run on 2-CTA clusters sharing KV staging
  int32_t kv_format = 0;          // 0 NVFP4, 1 FP8
  float sm_scale = 0.0f;
  // Ragged batches: one item per (sequence, q-tile) with queries, 4 int32
  // each (sequence, q-tile, KV tiles, 0), in the kernel's order; unit u is
  // head unit u % head_units of item u / head_units.  Empty for uniform
  // batches, whose units the kernel decodes arithmetically.
  std::vector<int32_t> work;
  // Balanced plans (few units per CTA slot): the work-list indices of each
  // slot's units, heaviest first; slot s runs slot_units[slot_begin[s] ..
  // slot_begin[s + 1]).  Empty otherwise (units are dealt round-robin).
  std::vector<int32_t> slot_units;
  std::vector<int32_t> slot_begin;
  // decode plans (fi_decode_plan): pieces (sequence * H_kv + kv head, first
  // key, end key, partial slot or -1) and merges (sequence, kv head, first
  // slot, pieces), 4 int32 each; warp w runs pieces dec_warp_off[w] ..
  // dec_warp_off[w + 1] - 1; dec_rows = G * max qo_len rows per partial slot;
  // dec_steps = the most key steps a warp takes
  bool decode = false;
  int32_t dec_rows = 0, dec_warps = 0, dec_steps = 0;
  int64_t dec_parts = 0;
  std::vector<int32_t> dec_units;
  std::vector<int32_t> dec_merges;
  std::vector<int32_t> dec_warp_off;
};

// Plans a decode (qo_len <= kDecodeMaxQo per sequence, G * qo_len <= 32).
constexpr int kDecodeMaxQo = 8;
constexpr int kDecodeMaxRows = 32;
// Decode work split: keys go in steps of kDecodeStep (one warp-wide copy of
// raw rows); a warp takes at least kDecodeMinSteps steps unless the batch has
// fewer, and at most as many warps run as the decode kernels keep resident per
// SM for the plan's rows (their launch bounds and shared memory: 4 CTAs of 4
// warps up to 8 rows, 3 up to 16, 2 above).
constexpr int kDecodeStep = 32;
constexpr int kDecodeMinSteps = 8;
constexpr int decode_warps_per_sm(int rows) { return rows <= 8 ? 16 : rows <= 16 ? 12 : 8; }
fi_status plan_decode_host(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                           int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t page_size, float sm_scale, int32_t num_sms, HostPlan* out);

struct DecodeArgs {
  const HostPlan* plan;
  const int32_t* qo_indptr_dev;
  const int32_t* kv_indptr_dev;
  const int32_t* units_dev;
  const int32_t* merges_dev;
  const int32_t* warp_off_dev;
  float* part;
  const int32_t* page_table;
  int32_t page_table_stride;
  const void* q;
  fi_nvfp4_cache cache;
  void* out;
  float* lse;
  int32_t* status;
};
fi_status launch_decode(const DecodeArgs& a, cudaStream_t stream);

// Validates the arguments and plans on the host only (no CUDA calls).
fi_status plan_host(const int32_t* qo_indptr, const int32_t* kv_indptr, int32_t batch,
                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, float sm_scale, int64_t l2_bytes, int32_t default_ctas,
                    const fi_plan_options* opts, HostPlan* out);

// ---- prefill -----------------------------------------------------------------
struct PrefillArgs {
  const HostPlan* plan;
  const int32_t* qo_indptr_dev;
  const int32_t* kv_indptr_dev;
  const int32_t* work_dev;       // null for uniform batches without a work list
  const int32_t* slot_units_dev; // balanced plans only (else null)
  const int32_t* slot_begin_dev;
  int32_t num_slots;
  const int32_t* page_table;
  int32_t page_table_stride;
  const void* q;
  fi_nvfp4_cache cache;          // FP8 (plan kv_format 1): k_sf / v_sf null
  void* out;
  float* lse;
  int32_t* status;
};
fi_status launch_prefill(const PrefillArgs& a, cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
bool encode_tensor_map_3d_bf16(void* map_out, const void* base, uint64_t dim0, uint64_t dim1,
                               uint64_t dim2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                               uint32_t box0, uint32_t box1, uint32_t box2);

}  // namespace fi
