// append.cu — NVFP4 quantize-append of bf16 K/V rows through a slot_mapping
// (FlashInfer PR #6204 analysis page, "FlashInfer: NVFP4 KV 캐시 어펜드 성능
// 최적화로 인한 동기화 제거": the append kernel checks the device scales itself
// instead of the host reading them back).
//
// Grid: y = (tensor, kv head) = (K|V, h); x = persistent CTAs striding over
// groups of kTokPerCta tokens.  One thread owns one 16-element block of one
// (token, tensor, head) row per step: two 128-bit bf16 loads (issued one step
// ahead), the block amax in registers, native E4M3/E2M1 conversion, one
// 64-bit store of 16 codes and one scale byte.  All index
// arithmetic inside the kernel is 32-bit except the final byte offsets; the
// page size is a power of two (shift and mask).  The kernel is HBM-bound: per
// written token it reads 2*H*D*2 bytes and writes 2*H*(D/2 + D/16) bytes
// (the algorithmic count; the values of skipped tokens are read as well).
#include <algorithm>

#include "internal.h"
#include "nvfp4.cuh"

namespace fi {

namespace {

constexpr int kAppendThreads = 256;
constexpr int kCtasPerSm = 4;  // resident CTAs per SM the persistent grid aims for

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
};

__device__ __forceinline__ bool scale_ok(float g) { return isfinite(g) && g > 0.0f; }

// Loads of one work item: the token's slot and one 16-element bf16 block.
struct Item {
  int64_t slot;
  uint4 w0, w1;
};

template <int D>
__device__ __forceinline__ Item load_item(const AppendParams& p, int t, int h, int blk,
                                          int64_t tok) {
  Item it;
  it.slot = -1;
  it.w0 = it.w1 = make_uint4(0u, 0u, 0u, 0u);
  if (tok < p.num_tokens) {
    const __nv_bfloat16* src =
        (t ? p.v + tok * p.v_tok_stride : p.k + tok * p.k_tok_stride) + h * D + blk * 16;
    it.slot = __ldg(p.slot_mapping + tok);
    it.w0 = __ldcs(reinterpret_cast<const uint4*>(src));
    it.w1 = __ldcs(reinterpret_cast<const uint4*>(src) + 1);
  }
  return it;
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads) nvfp4_append_kernel(const AppendParams p) {
  constexpr int kBlocks = D / 16;                    // threads per row
  constexpr int kTokPerCta = kAppendThreads / kBlocks;

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
  const int blk = threadIdx.x % kBlocks;
  const float g = t ? vs : ks;
  uint8_t* data = t ? p.v_data : p.k_data;
  uint8_t* sf = t ? p.v_sf : p.k_sf;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kTokPerCta;
  int64_t tok = static_cast<int64_t>(blockIdx.x) * kTokPerCta + threadIdx.x / kBlocks;
  // Persistent over token groups: the next group's slot and values are
  // loaded before the current group is quantized and stored, so every thread
  // keeps a memory request in flight.
  Item cur = load_item<D>(p, t, h, blk, tok);
  while (tok < p.num_tokens) {
    const Item nxt = load_item<D>(p, t, h, blk, tok + stride);
    if (cur.slot >= p.num_slots) {
      if (t == 0 && h == 0 && blk == 0) atomicOr(p.status, FI_DEV_SLOT_OOB);
    } else if (cur.slot >= 0) {
      float x[16];
      bf16x8_to_f32(cur.w0, x);
      bf16x8_to_f32(cur.w1, x + 8);
      const Quant16 q = quantize16(x, g);
      const int64_t page = cur.slot >> p.log2_page_size;
      const int64_t off = cur.slot & ((1 << p.log2_page_size) - 1);
      const int64_t cache_row = ((page * H + h) << p.log2_page_size) + off;
      *reinterpret_cast<uint2*>(data + cache_row * (D / 2) + blk * 8) = make_uint2(q.lo, q.hi);
      sf[cache_row * kBlocks + blk] = static_cast<uint8_t>(q.s8);
    }
    cur = nxt;
    tok += stride;
  }
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
  const int tok_per_cta = kAppendThreads / (D / 16);
  const int64_t groups = (a.num_tokens + tok_per_cta - 1) / tok_per_cta;
  const int64_t gy = 2 * static_cast<int64_t>(a.cache.num_kv_heads);
  if (gy > 65535) return FI_ERR_INVALID_ARGUMENT;
  // Persistent grid: about kCtasPerSm resident CTAs on every SM in total,
  // spread over the gy (tensor, head) rows, each looping over token groups.
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FI_ERR_CUDA;
  const int64_t want = (static_cast<int64_t>(sms) * kCtasPerSm + gy - 1) / gy;
  const int64_t gx = std::max<int64_t>(1, std::min<int64_t>(groups, want));
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  if (D == 128) {
    nvfp4_append_kernel<128><<<grid, kAppendThreads, 0, stream>>>(p);
  } else {
    nvfp4_append_kernel<64><<<grid, kAppendThreads, 0, stream>>>(p);
  }
  return cudaGetLastError() == cudaSuccess ? FI_OK : FI_ERR_CUDA;
}

}  // namespace fi
