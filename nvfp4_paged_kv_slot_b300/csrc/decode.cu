// decode.cu — attention of the few newest query tokens of each sequence
// (decode steps and short speculative steps, qo_len <= 8) over the NVFP4
// paged cache.  The planner side follows FlashInfer PR #5043 ("FlashInfer의
// plan() 함수 최적화: Python max()에서 Tensor.max()로의 전환", decode.py:
// max_kv_len from one reduction over the lengths); the attention is the same
// causal GQA attention as the prefill's (query row t of a sequence sees keys
// j <= t + kv_len - qo_len).
//
// Decode rows are few (G * qo_len per KV head) and every key is read once, so
// the work is HBM-bound and runs on the CUDA cores, not the tensor cores.
// One warp owns one unit = (sequence, KV head, chunk of keys): each lane
// dequantizes its own key's K row (E2M1 x E4M3, exact in fp32) and forms the
// logits of every query row against it (Q rows in shared memory, prescaled
// by sm_scale * k_scale * log2 e); the online softmax takes warp-wide maxima;
// for P V every lane owns D/32 output columns of every row and reads its
// columns of each key's V row from the warp's shared-memory copy of the 32
// V rows (each lane loads its own key's K and V rows with 16-byte loads).  A
// sequence whose keys span several chunks writes unnormalized partial results
// (row max, row sum, O) that a merge kernel combines.
#include <algorithm>

#include "internal.h"
#include "nvfp4.cuh"

namespace fi {

namespace {

constexpr int kDecWarps = 4;  // warps (units) per CTA

struct DecodeParams {
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  float* lse;
  const uint8_t* k_data;
  const uint8_t* v_data;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
  const float* k_scale;
  const float* v_scale;
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* page_table;
  int64_t pt_stride;
  const int4* units;   // (sequence, kv head, chunk, partial slot or -1)
  const int4* merges;  // (sequence, kv head, first partial slot, chunks)
  float* part;         // partial slots: [slot][rows][D + 2] = O, then m, l
  int32_t num_units, num_merges, num_qo_heads, num_kv_heads, group, page_size, num_pages;
  int32_t chunk, rows;  // keys per chunk; partial rows per slot (G * max qo_len)
  float sm_scale;
  int32_t* status;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Exact fp32 values of 8 E2M1 codes (one word) times the block's E4M3 scale.
__device__ __forceinline__ void dequant8_f32(uint32_t w, float sv, float (&x)[8]) {
  uint32_t h[4];
  e2m1x8_to_f16x2(w, h);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[k]));
    x[2 * k] = f.x * sv;
    x[2 * k + 1] = f.y * sv;
  }
}

// Cache row of key `key` of sequence b, KV head hk (page checked).
__device__ __forceinline__ int64_t key_row(const DecodeParams& p, const int32_t* pt, int key,
                                           int hk) {
  int page = __ldg(pt + key / p.page_size);
  if (page < 0 || page >= p.num_pages) {
    atomicOr(p.status, FI_DEV_PAGE_OOB);
    page = 0;
  }
  return (static_cast<int64_t>(page) * p.num_kv_heads + hk) * p.page_size + key % p.page_size;
}

// RMAX: compile-time bound on the rows (G * qo_len) of a unit.
// Bytes of one staged V row (codes, then scales), padded to 16.
template <int D>
constexpr int kVRow = (D / 2 + D / 16 + 15) / 16 * 16;

template <int D, int RMAX>
__global__ void __launch_bounds__(32 * kDecWarps) nvfp4_decode_kernel(const DecodeParams p) {
  constexpr int kDpl = D / 32;  // output columns per lane
  extern __shared__ float dsm[];
  grid_dep_wait();  // Q and the cache may come from the previous grid
  grid_dep_launch();
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int u = blockIdx.x * kDecWarps + warp;
  if (u >= p.num_units) return;  // no block-wide barrier below
  const int4 w = __ldg(p.units + u);
  const int b = w.x, hk = w.y, c = w.z, slot = w.w;
  const int qo_start = __ldg(p.qo_indptr + b);
  const int qo_len = __ldg(p.qo_indptr + b + 1) - qo_start;
  const int kv_len = __ldg(p.kv_indptr + b + 1) - __ldg(p.kv_indptr + b);
  const int G = p.group;
  const int R = G * qo_len;  // <= RMAX (the planner guarantees it)
  const int delta = kv_len - qo_len;
  const int k0 = c * p.chunk;
  const int k1 = min(k0 + p.chunk, kv_len);
  const float ks = __ldg(p.k_scale), vs = __ldg(p.v_scale);
  // Q rows (row r = token r / G, head hk * G + r % G) prescaled to log2 units;
  // after all warps' Q rows: each warp's 32 V rows (codes, then scales)
  float* sq = dsm + warp * RMAX * D;
  uint8_t* svr = reinterpret_cast<uint8_t*>(dsm + kDecWarps * RMAX * D) +
                 warp * 32 * kVRow<D>;
  const float qs = p.sm_scale * ks * 1.4426950408889634f;
  for (int i = lane; i < R * (D / 8); i += 32) {
    const int r = i / (D / 8), ch = i % (D / 8);
    const int t = r / G, g = r % G;
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(
        p.q + (static_cast<int64_t>(qo_start + t) * p.num_qo_heads + hk * G + g) * D + ch * 8));
    float x[8];
    bf16x8_to_f32(v, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) sq[r * D + ch * 8 + e] = x[e] * qs;
  }
  __syncwarp();
  const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride;

  float m[RMAX], l[RMAX], o[RMAX][kDpl];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int e = 0; e < kDpl; ++e) o[r][e] = 0.0f;
  }
  for (int kb = k0; kb < k1; kb += 32) {
    const int key = kb + lane;
    const bool kvalid = key < k1;
    // ---- logits of every row against this lane's key
    float s[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) s[r] = 0.0f;
    // this lane's key: its K and V rows with 16-byte loads (one page lookup);
    // the V row goes to the warp's staging area for the P V step
    __syncwarp();  // the previous batch's V rows have been read
    if (kvalid) {
      const int64_t row = key_row(p, pt, key, hk);
      uint4 kc4[D / 32], vc4[D / 32];
      uint32_t ksf4[D / 64], vsf4[D / 64];
      const uint4* kg = reinterpret_cast<const uint4*>(p.k_data + row * (D / 2));
      const uint4* vg = reinterpret_cast<const uint4*>(p.v_data + row * (D / 2));
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        kc4[i] = __ldg(kg + i);
        vc4[i] = __ldg(vg + i);
      }
#pragma unroll
      for (int i = 0; i < D / 64; ++i) {
        ksf4[i] = __ldg(reinterpret_cast<const uint32_t*>(p.k_sf + row * (D / 16)) + i);
        vsf4[i] = __ldg(reinterpret_cast<const uint32_t*>(p.v_sf + row * (D / 16)) + i);
      }
      uint8_t* dst = svr + lane * kVRow<D>;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) reinterpret_cast<uint4*>(dst)[i] = vc4[i];
#pragma unroll
      for (int i = 0; i < D / 64; ++i) reinterpret_cast<uint32_t*>(dst + D / 2)[i] = vsf4[i];
      const uint32_t* kc = reinterpret_cast<const uint32_t*>(kc4);
#pragma unroll
      for (int blk = 0; blk < D / 16; ++blk) {
        const float sv = e4m3_value((ksf4[blk / 4] >> (8 * (blk % 4))) & 0xFFu);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float kx[8];
          dequant8_f32(kc[2 * blk + half], sv, kx);
          const int d0 = blk * 16 + half * 8;
#pragma unroll
          for (int r = 0; r < RMAX; ++r) {
            if (r < R) {
              const float4 qa = *reinterpret_cast<const float4*>(sq + r * D + d0);
              const float4 qb = *reinterpret_cast<const float4*>(sq + r * D + d0 + 4);
              s[r] = fmaf(qa.x, kx[0], s[r]);
              s[r] = fmaf(qa.y, kx[1], s[r]);
              s[r] = fmaf(qa.z, kx[2], s[r]);
              s[r] = fmaf(qa.w, kx[3], s[r]);
              s[r] = fmaf(qb.x, kx[4], s[r]);
              s[r] = fmaf(qb.y, kx[5], s[r]);
              s[r] = fmaf(qb.z, kx[6], s[r]);
              s[r] = fmaf(qb.w, kx[7], s[r]);
            }
          }
        }
      }
    }
    // ---- causal mask, online softmax (row statistics are warp-uniform)
    float pr[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      if (r < R) {
        const bool vis = kvalid && key <= delta + r / G;
        const float sr = vis ? s[r] : -INFINITY;
        const float m_new = fmaxf(m[r], warp_max(sr));
        const float alpha = m_new == -INFINITY ? 1.0f : ex2_approx(m[r] - m_new);
        pr[r] = vis ? ex2_approx(sr - m_new) : 0.0f;
        l[r] = l[r] * alpha + pr[r];
#pragma unroll
        for (int e = 0; e < kDpl; ++e) o[r][e] *= alpha;
        m[r] = m_new;
      } else {
        pr[r] = 0.0f;
      }
    }
    // ---- O += P V: this lane's columns of each key's V row
    __syncwarp();  // every lane's V row is staged
    const int nk = min(32, k1 - kb);
#pragma unroll 4
    for (int kk = 0; kk < nk; ++kk) {
      const uint8_t* vrow = svr + kk * kVRow<D>;
      const uint8_t* vc = vrow + lane * (kDpl / 2);
      const float sv = e4m3_value(vrow[D / 2 + (lane * kDpl) / 16]);
      float vx[kDpl];
      if constexpr (kDpl == 4) {
        const uint32_t two = *reinterpret_cast<const uint16_t*>(vc);
        uint32_t h[4];
        e2m1x8_to_f16x2(two, h);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h[0]));
        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&h[1]));
        vx[0] = f0.x * sv;
        vx[1] = f0.y * sv;
        vx[2] = f1.x * sv;
        vx[3] = f1.y * sv;
      } else {
        const uint32_t one = *vc;
        uint32_t h[4];
        e2m1x8_to_f16x2(one, h);
        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&h[0]));
        vx[0] = f0.x * sv;
        vx[1] = f0.y * sv;
      }
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r < R) {
          const float pk = __shfl_sync(0xFFFFFFFFu, pr[r], kk);
#pragma unroll
          for (int e = 0; e < kDpl; ++e) o[r][e] = fmaf(pk, vx[e], o[r][e]);
        }
      }
    }
  }
  // ---- results: the whole sequence in this unit, or a partial slot
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r < R) {
      const float lr = warp_sum(l[r]);
      const int t = r / G, g = r % G;
      if (slot < 0) {
        const int64_t orow = static_cast<int64_t>(qo_start + t) * p.num_qo_heads + hk * G + g;
        const float inv = vs / lr;
        __nv_bfloat16* dst = p.out + orow * D + lane * kDpl;
#pragma unroll
        for (int e = 0; e < kDpl; e += 2)
          *reinterpret_cast<__nv_bfloat162*>(dst + e) =
              __floats2bfloat162_rn(o[r][e] * inv, o[r][e + 1] * inv);
        if (p.lse && lane == 0) p.lse[orow] = (m[r] + log2f(lr)) * 0.6931471805599453f;
      } else {
        float* dst = p.part + (static_cast<int64_t>(slot) * p.rows + r) * (D + 2);
#pragma unroll
        for (int e = 0; e < kDpl; ++e) dst[lane * kDpl + e] = o[r][e];
        if (lane == 0) {
          dst[D] = m[r];
          dst[D + 1] = lr;
        }
      }
    }
  }
}

// One warp per (merge item, row): combines the item's partial slots
//   M = max m_i,  L = sum l_i 2^(m_i - M),  O = sum O_i 2^(m_i - M) / L,
// scaled by v_scale, and lse = (M + log2 L) ln 2.
template <int D>
__global__ void __launch_bounds__(128) nvfp4_decode_merge_kernel(const DecodeParams p) {
  constexpr int kDpl = D / 32;
  grid_dep_wait();
  grid_dep_launch();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int item = warp / p.rows, r = warp % p.rows;
  if (item >= p.num_merges) return;
  const int4 w = __ldg(p.merges + item);
  const int b = w.x, hk = w.y, first = w.z, n = w.w;
  const int qo_start = __ldg(p.qo_indptr + b);
  const int qo_len = __ldg(p.qo_indptr + b + 1) - qo_start;
  const int G = p.group;
  if (r >= G * qo_len) return;
  float M = -INFINITY;
  for (int i = 0; i < n; ++i)
    M = fmaxf(M, p.part[(static_cast<int64_t>(first + i) * p.rows + r) * (D + 2) + D]);
  float L = 0.0f, acc[kDpl];
#pragma unroll
  for (int e = 0; e < kDpl; ++e) acc[e] = 0.0f;
  for (int i = 0; i < n; ++i) {
    const float* src = p.part + (static_cast<int64_t>(first + i) * p.rows + r) * (D + 2);
    const float mi = src[D];
    const float wgt = mi == -INFINITY ? 0.0f : ex2_approx(mi - M);
    L += src[D + 1] * wgt;
#pragma unroll
    for (int e = 0; e < kDpl; ++e) acc[e] = fmaf(src[lane * kDpl + e], wgt, acc[e]);
  }
  const float vs = __ldg(p.v_scale);
  const int t = r / G, g = r % G;
  const int64_t orow = static_cast<int64_t>(qo_start + t) * p.num_qo_heads + hk * G + g;
  const float inv = vs / L;
  __nv_bfloat16* dst = p.out + orow * D + lane * kDpl;
#pragma unroll
  for (int e = 0; e < kDpl; e += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + e) =
        __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  if (p.lse && lane == 0) p.lse[orow] = (M + log2f(L)) * 0.6931471805599453f;
}

template <int D, int RMAX>
fi_status launch_decode_impl(const DecodeParams& p, cudaStream_t stream) {
  const int smem = kDecWarps * RMAX * D * static_cast<int>(sizeof(float)) +
                   kDecWarps * 32 * kVRow<D>;
  auto kern = nvfp4_decode_kernel<D, RMAX>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return FI_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>((p.num_units + kDecWarps - 1) / kDecWarps);
  fi_status st = launch_pdl(kern, dim3(grid), dim3(32 * kDecWarps), smem, stream, p);
  if (st != FI_OK || p.num_merges == 0) return st;
  const int64_t warps = static_cast<int64_t>(p.num_merges) * p.rows;
  const unsigned mgrid = static_cast<unsigned>((warps + 3) / 4);
  return launch_pdl(nvfp4_decode_merge_kernel<D>, dim3(mgrid), dim3(128), 0, stream, p);
}

}  // namespace

fi_status launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  const HostPlan& P = *a.plan;
  if (P.info.num_units == 0) return FI_OK;
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.k_data = a.cache.k_data;
  p.v_data = a.cache.v_data;
  p.k_sf = a.cache.k_sf;
  p.v_sf = a.cache.v_sf;
  p.k_scale = a.cache.k_scale;
  p.v_scale = a.cache.v_scale;
  p.qo_indptr = a.qo_indptr_dev;
  p.kv_indptr = a.kv_indptr_dev;
  p.page_table = a.page_table;
  p.pt_stride = a.page_table_stride;
  p.units = reinterpret_cast<const int4*>(a.units_dev);
  p.merges = reinterpret_cast<const int4*>(a.merges_dev);
  p.part = a.part;
  if (P.info.num_units > 0x7FFFFFFF) return FI_ERR_UNSUPPORTED;
  p.num_units = static_cast<int32_t>(P.info.num_units);
  p.num_merges = static_cast<int32_t>(P.dec_merges.size() / 4);
  p.num_qo_heads = P.num_qo_heads;
  p.num_kv_heads = P.num_kv_heads;
  p.group = P.group;
  p.page_size = P.page_size;
  p.num_pages = a.cache.num_pages;
  p.chunk = P.dec_chunk;
  p.rows = P.dec_rows;
  p.sm_scale = P.sm_scale;
  p.status = a.status;
  const int D = P.head_dim;
  if (P.dec_rows <= 8)
    return D == 128 ? launch_decode_impl<128, 8>(p, stream) : launch_decode_impl<64, 8>(p, stream);
  return D == 128 ? launch_decode_impl<128, 32>(p, stream) : launch_decode_impl<64, 32>(p, stream);
}

}  // namespace fi
