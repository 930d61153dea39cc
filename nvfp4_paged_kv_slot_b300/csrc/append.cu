// append.cu — NVFP4 quantize-append of bf16 K/V rows through a slot_mapping
// (FlashInfer PR #6204 analysis page, "FlashInfer: NVFP4 KV 캐시 어펜드 성능
// 최적화로 인한 동기화 제거": the append kernel checks the device scales itself
// instead of the host reading them back).
//
// One thread owns 8 consecutive head-dim elements of one (token, tensor, head)
// row: a 128-bit bf16 load, the per-16 amax shared with the neighbouring lane
// by one shuffle, native E4M3/E2M1 conversion, one 32-bit store of 8 codes and
// (even lanes) one scale byte.  The kernel is HBM-bound: per written token it
// reads 2*H*D*2 bytes and writes 2*H*(D/2 + D/16) bytes.
#include "internal.h"
#include "nvfp4.cuh"

namespace fi {

namespace {

constexpr int kAppendThreads = 256;

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
  int64_t num_rows;   // num_tokens * 2 * num_kv_heads
  int64_t num_slots;  // num_pages * page_size
  int32_t num_kv_heads, page_size;
  int32_t* status;
};

__device__ __forceinline__ bool scale_ok(float g) { return isfinite(g) && g > 0.0f; }

template <int D>
__global__ void __launch_bounds__(kAppendThreads) nvfp4_append_kernel(const AppendParams p) {
  constexpr int kChunks = D / 8;                     // threads per row
  constexpr int kRowsPerBlock = kAppendThreads / kChunks;

  // Scale check, once per CTA before any store: a bad scale means no CTA writes.
  const float ks = p.k_scale_dev ? __ldg(p.k_scale_dev) : p.k_scale_host;
  const float vs = p.v_scale_dev ? __ldg(p.v_scale_dev) : p.v_scale_host;
  if (!scale_ok(ks) || !scale_ok(vs)) {
    if (blockIdx.x == 0 && threadIdx.x == 0)
      atomicOr(p.status, (scale_ok(ks) ? 0 : FI_DEV_BAD_K_SCALE) |
                             (scale_ok(vs) ? 0 : FI_DEV_BAD_V_SCALE));
    return;  // uniform across the CTA
  }

  const int c = threadIdx.x % kChunks;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + threadIdx.x / kChunks;
  const int H = p.num_kv_heads;
  bool active = row < p.num_rows;
  int64_t tok = 0, slot = -1;
  int t = 0, h = 0;
  if (active) {
    tok = row / (2 * H);
    const int rem = static_cast<int>(row - tok * 2 * H);
    t = rem / H;  // 0 = K, 1 = V
    h = rem - t * H;
    slot = __ldg(p.slot_mapping + tok);
    if (slot < 0) {
      active = false;
    } else if (slot >= p.num_slots) {
      if (t == 0 && h == 0 && c == 0) atomicOr(p.status, FI_DEV_SLOT_OOB);
      active = false;
    }
  }
  float x[8];
  float amax = 0.0f;
  if (active) {
    const __nv_bfloat16* src =
        (t ? p.v + tok * p.v_tok_stride : p.k + tok * p.k_tok_stride) + h * D + c * 8;
    const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(src));
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.0f;
  }
  // lanes 2b and 2b+1 hold the two halves of 16-element block b
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  if (!active) return;

  const Quant8 q = quantize8(x, amax, t ? vs : ks);
  const int64_t page = slot / p.page_size;
  const int64_t off = slot - page * p.page_size;
  const int64_t cache_row = (page * H + h) * p.page_size + off;
  uint8_t* data = t ? p.v_data : p.k_data;
  uint8_t* sf = t ? p.v_sf : p.k_sf;
  *reinterpret_cast<uint32_t*>(data + cache_row * (D / 2) + c * 4) = q.codes;
  if ((c & 1) == 0) sf[cache_row * (D / 16) + c / 2] = static_cast<uint8_t>(q.s8);
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
  p.page_size = a.cache.page_size;
  p.num_rows = a.num_tokens * 2 * a.cache.num_kv_heads;
  p.num_slots = static_cast<int64_t>(a.cache.num_pages) * a.cache.page_size;
  p.status = a.status;
  const int D = a.cache.head_dim;
  const int rows_per_block = kAppendThreads / (D / 8);
  const int64_t blocks = (p.num_rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 0x7FFFFFFF) return FI_ERR_INVALID_ARGUMENT;
  if (D == 128) {
    nvfp4_append_kernel<128><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(p);
  } else {
    nvfp4_append_kernel<64><<<static_cast<unsigned>(blocks), kAppendThreads, 0, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

}  // namespace fi
