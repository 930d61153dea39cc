// diag.cu — probes that run the library's device code on small inputs
// (declared in include/fi_nvfp4_diag.h).
#include <cudaTypedefs.h>

#include <mutex>

#include "fi_nvfp4.h"
#include "fi_nvfp4_diag.h"
#include "nvfp4.cuh"

namespace fi {
namespace {

constexpr uint64_t kProbeTimeoutNs = 1000000000ull;

__global__ void codec_span_kernel(uint32_t first, uint64_t count, uint8_t* e4, uint8_t* e2) {
  const uint64_t i = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= count) return;
  const float x = __uint_as_float(first + static_cast<uint32_t>(i));
  e4[i] = static_cast<uint8_t>(e4m3_from_f32(x));
  e2[i] = static_cast<uint8_t>(e2m1x4_from_f32(x, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu);
}

__global__ void quantize_blocks_kernel(const __nv_bfloat16* x, int64_t n, float g, uint8_t* packed,
                                       uint8_t* s8) {
  const int64_t b = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (b >= n) return;
  float v[16];
  for (int j = 0; j < 16; ++j) v[j] = __bfloat162float(x[b * 16 + j]);
  const Quant16 q = quantize16(v, g);
  reinterpret_cast<uint32_t*>(packed + b * 8)[0] = q.lo;
  reinterpret_cast<uint32_t*>(packed + b * 8)[1] = q.hi;
  s8[b] = static_cast<uint8_t>(q.s8);
}

// For every bf16 bit pattern x (blockIdx.x, threadIdx.x) and every divisor
// d_values[blockIdx.y] that the quantizer would send through the Markstein
// path (markstein_range_ok(d, |x|)), compares div_markstein_x2 (as the
// quantizer calls it) with the IEEE quotient __fdiv_rn(x, d).
// counts[0] += checked pairs; counts[1] += pairs whose E2M1 codes differ;
// counts[2] += pairs with |x| >= 2^-100 and a normal IEEE quotient whose fp32
// bits differ (the range where the residual is exact); counts[3] += pairs
// with |x| < 2^-100 whose bits differ (allowed: the code is the same there).
// first_bad gets the (x bits, d index) of one pair counted in [1] or [2].
__global__ void div_check_kernel(const float* d_values, unsigned long long* counts,
                                 uint32_t* first_bad) {
  const uint32_t xb = blockIdx.x * blockDim.x + threadIdx.x;  // 0 .. 65535
  const float x = __uint_as_float(xb << 16);
  const float d = d_values[blockIdx.y];
  unsigned long long c[4] = {0, 0, 0, 0};
  if (isfinite(x) && markstein_range_ok(d, fabsf(x))) {
    c[0] = 1;
    const float r = __frcp_rn(d);
    float a = x, a1 = x;
    div_markstein_x2(a, a1, f2_pack(-d, -d), f2_pack(r, r));
    const float b = __fdiv_rn(x, d);
    const uint32_t ca = e2m1x4_from_f32(a, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu;
    const uint32_t cb = e2m1x4_from_f32(b, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu;
    const bool bits_differ = __float_as_uint(a) != __float_as_uint(b);
    const bool exact_range = fabsf(x) >= 0x1p-100f && fabsf(b) >= 0x1p-126f;
    // the block-scale division t = amax / RN(6 g) takes this path for
    // amax >= 2^-100; its E4M3 code must not change either
    const bool e4_differ =
        fabsf(x) >= 0x1p-100f && e4m3_from_f32(fabsf(a)) != e4m3_from_f32(fabsf(b));
    if (ca != cb || e4_differ) c[1] = 1;
    if (bits_differ && exact_range) c[2] = 1;
    if (bits_differ && fabsf(x) < 0x1p-100f) c[3] = 1;
    if (c[1] || c[2]) {
      first_bad[0] = xb;
      first_bad[1] = blockIdx.y;
    }
  }
  for (int k = 0; k < 4; ++k) {
    unsigned long long v = c[k];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if ((threadIdx.x & 31) == 0 && v) atomicAdd(counts + k, v);
  }
}

template <int D, bool IS_V>
__global__ void repack_probe_kernel(const uint8_t* raw, int valid, uint16_t* out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* rs = smem;                    // raw tile
  uint8_t* st = smem + 16384;            // staging tile (1 KB aligned)
  constexpr int kRaw = 128 * (D / 2 + D / 16);
  for (int i = threadIdx.x; i < kRaw; i += blockDim.x) rs[i] = raw[i];
  __syncthreads();
  repack_tile<D, IS_V, 128>(rs, st, valid, threadIdx.x);
  __syncthreads();
  for (int i = threadIdx.x; i < 128 * (D / 8); i += blockDim.x) {
    const int row = i / (D / 8), c = i % (D / 8);
    const uint4 v = *reinterpret_cast<const uint4*>(st + sw128_offset(row, c));
    *reinterpret_cast<uint4*>(out + row * D + c * 8) = v;
  }
}

struct UmmaProbeParams {
  CUtensorMap tmap_a;
  const uint16_t* a;
  const uint16_t* b;
  float* c;
  int32_t* status;
  int mode;
};

__global__ void __launch_bounds__(128, 1) umma_probe_kernel(const __grid_constant__ UmmaProbeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + 32768;
  uint64_t* bar_tma = reinterpret_cast<uint64_t*>(smem + 65536);
  uint64_t* bar_mma = bar_tma + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  int* abort_flag = reinterpret_cast<int*>(tslot + 1);
  const int tid = threadIdx.x;
  const int warp = tid / 32;
  if (tid == 0) {
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  // thread tid stages row tid of B (and of A in mode 3) in the swizzled layout
  for (int c = 0; c < 16; ++c)
    *reinterpret_cast<uint4*>(sb + sw128_offset(tid, c)) =
        *reinterpret_cast<const uint4*>(p.b + tid * 128 + c * 8);
  if (p.mode == 3)
    for (int c = 0; c < 16; ++c)
      *reinterpret_cast<uint4*>(sa + sw128_offset(tid, c)) =
          *reinterpret_cast<const uint4*>(p.a + tid * 128 + c * 8);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t lane_base = tbase + ((static_cast<uint32_t>(warp) * 32) << 16);
  if (p.mode == 1) {
    // row tid of A into columns 128..191: column c holds elements 2c (low
    // half) and 2c+1 (high half)
    const uint32_t* arow = reinterpret_cast<const uint32_t*>(p.a + tid * 128);
    uint32_t v[32];
    for (int k = 0; k < 32; ++k) v[k] = arow[k];
    tmem_st32(lane_base + 128, v);
    for (int k = 0; k < 32; ++k) v[k] = arow[32 + k];
    tmem_st32(lane_base + 160, v);
    tmem_st_wait();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const AbortState ab{abort_flag, p.status, kProbeTimeoutNs, 1 << 16};
  if (tid == 0) {
    bool ok = true;
    if (p.mode == 0) {
      mbar_arrive_expect_tx(bar_tma, 32768);
      tma_load_3d(sa, &p.tmap_a, bar_tma, 0, 0, 0);
      tma_load_3d(sa + 16384, &p.tmap_a, bar_tma, 64, 0, 0);
      ok = mbar_wait(bar_tma, 0, ab);
    }
    if (ok) {
      const uint32_t a_addr = smem_u32(sa), b_addr = smem_u32(sb);
      if (p.mode == 0) {
        constexpr uint32_t idesc = idesc_f16(1, 0, 0, 128, 128);
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_ss(tbase, smem_desc_sw128(a_addr + off, 16, 1024),
                 smem_desc_sw128(b_addr + off, 16, 1024), idesc, kk > 0);
        }
      } else {
        constexpr uint32_t idesc = idesc_f16(0, 0, 1, 128, 128);
        for (int s = 0; s < 8; ++s) {
          const uint64_t bd = smem_desc_sw128(b_addr + s * 2048, 16384, 1024);
          if (p.mode == 3) {
            const uint32_t off = (s >> 2) * 16384 + (s & 3) * 32;
            mma_ss(tbase, smem_desc_sw128(a_addr + off, 16, 1024), bd, idesc, s > 0);
          } else {
            mma_ts(tbase, tbase + 128 + s * 8, bd, idesc, s > 0);
          }
        }
      }
    }
    mma_commit(bar_mma);
  }
  __syncwarp();
  mbar_wait(bar_mma, 0, ab);
  tc_fence_after();
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tmem_ld32(lane_base + c * 32, v);
    for (int k = 0; k < 32; ++k) p.c[tid * 128 + c * 32 + k] = __uint_as_float(v[k]);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, 256);
}

// A pipeline that stops: the waits of the library's kernels (mbar_wait with
// an AbortState) on an mbarrier that nothing arrives at.  Warp 0 holds tensor
// memory and has a bulk copy in flight, as the prefill's roles do, and waits
// with the caller's limit; warp 1 (one thread) and warps 2-3 (every thread)
// wait on the same barrier with the prefill's own 2 s limit and must give up
// as soon as warp 0's wait has set the CTA's abort flag.  Then warp 0 drains
// its copy (a bounded wait on the copy's barrier, as the prefill's load warp
// does when it aborts), every thread meets, and the tensor memory is freed.
// report[0]: ns warp 0 waited; [1]: ns warp 1 waited; [2]: waits that gave up
// (66 expected: 1 + 1 + 64); [3]: 1 if the drained copy completed;
// copy_out: the copied bytes, read back from shared memory after the drain.
constexpr int kProbeCopyBytes = 4096;
constexpr uint64_t kPipelineTimeoutNs = 2000000000ull;  // the prefill's limit
constexpr uint64_t kDrainNs = 100000000ull;

__global__ void __launch_bounds__(128, 1)
    wait_timeout_probe_kernel(uint64_t timeout_ns, const uint8_t* copy_src, uint8_t* copy_out,
                              int32_t* status, unsigned long long* report) {
  __shared__ __align__(128) uint8_t buf[kProbeCopyBytes];
  __shared__ uint64_t never, copy_done;
  __shared__ uint32_t tslot;
  __shared__ int abort_flag;
  __shared__ unsigned gave_up;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    mbar_init(&never, 1);
    mbar_init(&copy_done, 1);
    abort_flag = 0;
    gave_up = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tslot, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = tslot;
  const AbortState ab_short{&abort_flag, status, timeout_ns, FI_DEV_WAIT_TIMEOUT};
  const AbortState ab_long{&abort_flag, status, kPipelineTimeoutNs, FI_DEV_WAIT_TIMEOUT};
  if (warp == 0) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&copy_done, kProbeCopyBytes);
      bulk_g2s(buf, copy_src, kProbeCopyBytes, &copy_done);
      const uint64_t t0 = global_timer_ns();
      const bool ok = mbar_wait(&never, 0, ab_short);
      report[0] = global_timer_ns() - t0;
      if (!ok) atomicAdd(&gave_up, 1u);
      volatile int drain_flag = 0;
      const AbortState drain_ab{&drain_flag, nullptr, kDrainNs, 0};
      report[3] = mbar_wait(&copy_done, 0, drain_ab) ? 1ull : 0ull;
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint64_t t0 = global_timer_ns();
      const bool ok = mbar_wait(&never, 0, ab_long);
      report[1] = global_timer_ns() - t0;
      if (!ok) atomicAdd(&gave_up, 1u);
    }
    __syncwarp();
  } else {
    if (!mbar_wait(&never, 0, ab_long)) atomicAdd(&gave_up, 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  for (int i = threadIdx.x; i < kProbeCopyBytes / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(copy_out)[i] = reinterpret_cast<const uint4*>(buf)[i];
  if (threadIdx.x == 0) report[2] = gave_up;
  if (warp == 0) tmem_dealloc(tbase, 32);
}

// One M=256 N=128 K=128 MMA over a CTA pair (cta_group::2), as the paired
// prefill issues them.  CTA r stages rows 128 r .. 128 r + 127 of A (K-major,
// bf16 in mode 0, fp16 in mode 1) and its half of B: mode 0 (S = Q K^T) rows
// 64 r .. 64 r + 63 of B [128 N][128 K] (K-major, 64-row column blocks of
// 8 KB); mode 1 (O = P V) columns 64 r .. 64 r + 63 of B [128 K][128 N]
// (MN-major, one 16 KB block).  The even CTA issues the MMAs and a commit to
// both CTAs' barriers; each CTA reads its 128 rows of D.  tmem_addrs[r]: the
// tensor-memory base each CTA was given.
struct UmmaPairParams {
  const uint16_t* a;
  const uint16_t* b;
  float* c;
  int32_t* status;
  uint32_t* tmem_addrs;
  int mode;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    umma_pair_probe_kernel(const __grid_constant__ UmmaPairParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + 32768;
  uint64_t* bar_mma = reinterpret_cast<uint64_t*>(smem + 49152);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  int* abort_flag = reinterpret_cast<int*>(tslot + 1);
  const uint32_t rank = cluster_ctarank();
  const int tid = threadIdx.x;
  const int warp = tid / 32;
  if (tid == 0) {
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(tslot, 256);
    tmem_relinquish_pair();
  }
  // row tid of this CTA's half of A
  const uint16_t* arow = p.a + (128 * rank + tid) * 128;
  for (int c = 0; c < 16; ++c)
    *reinterpret_cast<uint4*>(sa + sw128_offset(tid, c)) = *reinterpret_cast<const uint4*>(arow + 8 * c);
  if (p.mode == 0) {
    if (tid < 64) {
      const uint16_t* brow = p.b + (64 * rank + tid) * 128;
      for (int c = 0; c < 16; ++c)
        *reinterpret_cast<uint4*>(sb + (c >> 3) * 8192 + tid * 128 + (((c & 7) ^ (tid & 7)) << 4)) =
            *reinterpret_cast<const uint4*>(brow + 8 * c);
    }
  } else {
    const uint16_t* brow = p.b + tid * 128 + 64 * rank;
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(sb + sw128_offset(tid, c)) = *reinterpret_cast<const uint4*>(brow + 8 * c);
  }
  fence_proxy_async_cluster();
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  if (tid == 0) p.tmem_addrs[rank] = tbase;
  const AbortState ab{abort_flag, p.status, kProbeTimeoutNs, 1 << 16};
  if (rank == 0 && tid == 0) {
    const uint32_t a_addr = smem_u32(sa), b_addr = smem_u32(sb);
    if (p.mode == 0) {
      constexpr uint32_t idesc = idesc_f16(1, 0, 0, 256, 128);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t a_off = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t b_off = (kk >> 2) * 8192 + (kk & 3) * 32;
        mma_ss_pair(tbase, smem_desc_sw128(a_addr + a_off, 16, 1024),
                    smem_desc_sw128(b_addr + b_off, 16, 1024), idesc, kk > 0);
      }
    } else {
      constexpr uint32_t idesc = idesc_f16(0, 0, 1, 256, 128);
      for (int s = 0; s < 8; ++s) {
        const uint32_t a_off = (s >> 2) * 16384 + (s & 3) * 32;
        mma_ss_pair(tbase, smem_desc_sw128(a_addr + a_off, 16, 1024),
                    smem_desc_sw128(b_addr + s * 2048, 16384, 1024), idesc, s > 0);
      }
    }
    mma_commit_pair(bar_mma, 3);
  }
  __syncwarp();
  mbar_wait(bar_mma, 0, ab);
  tc_fence_after();
  const uint32_t lane_base = tbase + ((static_cast<uint32_t>(warp) * 32) << 16);
  for (int c = 0; c < 4; ++c) {
    uint32_t v[32];
    tmem_ld32(lane_base + c * 32, v);
    for (int k = 0; k < 32; ++k)
      p.c[(128 * rank + tid) * 128 + c * 32 + k] = __uint_as_float(v[k]);
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  if (warp == 0) tmem_dealloc_pair(tbase, 256);
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace fi

extern "C" {

int32_t fi_diag_codec_span(uint32_t first_bits, uint64_t count, uint8_t* e4m3_out,
                           uint8_t* e2m1_out, void* stream) {
  if (!e4m3_out || !e2m1_out || count > (1ull << 32)) return 1;
  if (count == 0) return 0;
  const unsigned blocks = static_cast<unsigned>((count + 255) / 256);
  fi::codec_span_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      first_bits, count, e4m3_out, e2m1_out);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int32_t fi_diag_quantize_blocks(const void* x, int64_t n_blocks, float g, uint8_t* packed_out,
                                uint8_t* s8_out, void* stream) {
  if (!x || !packed_out || !s8_out || n_blocks < 0 || !fi::a16(packed_out)) return 1;
  if (n_blocks == 0) return 0;
  const unsigned blocks = static_cast<unsigned>((n_blocks + 127) / 128);
  fi::quantize_blocks_kernel<<<blocks, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16*>(x), n_blocks, g, packed_out, s8_out);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int32_t fi_diag_div_check(const float* d_values, int32_t n_d, unsigned long long* counts,
                          uint32_t* first_bad, void* stream) {
  if (!d_values || !counts || !first_bad || n_d <= 0 || n_d > 65535) return 1;
  const dim3 grid(65536 / 256, static_cast<unsigned>(n_d));
  fi::div_check_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(d_values, counts,
                                                                           first_bad);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int32_t fi_diag_repack_tile(const uint8_t* raw, int32_t head_dim, int32_t is_v, int32_t valid,
                            uint16_t* out, void* stream) {
  if (!raw || !out || !fi::a16(out) || (head_dim != 64 && head_dim != 128)) return 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int smem = 16384 + 32768 + 1024;
  if (head_dim == 128) {
    if (is_v) {
      cudaFuncSetAttribute(fi::repack_probe_kernel<128, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      fi::repack_probe_kernel<128, true><<<1, 128, smem, s>>>(raw, valid, out);
    } else {
      cudaFuncSetAttribute(fi::repack_probe_kernel<128, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      fi::repack_probe_kernel<128, false><<<1, 128, smem, s>>>(raw, valid, out);
    }
  } else {
    if (is_v) {
      cudaFuncSetAttribute(fi::repack_probe_kernel<64, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      fi::repack_probe_kernel<64, true><<<1, 128, smem, s>>>(raw, valid, out);
    } else {
      cudaFuncSetAttribute(fi::repack_probe_kernel<64, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      fi::repack_probe_kernel<64, false><<<1, 128, smem, s>>>(raw, valid, out);
    }
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int32_t fi_diag_umma(int32_t mode, const void* a, const void* b, float* c, int32_t* status,
                     void* stream) {
  if ((mode != 0 && mode != 1 && mode != 3) || !a || !b || !c || !status || !fi::a16(a) || !fi::a16(b)) return 1;
  fi::UmmaProbeParams p;
  memset(&p, 0, sizeof(p));
  if (mode == 0) {
    std::call_once(fi::g_once, fi::load_encode);
    if (!fi::g_encode) return 4;
    cuuint64_t dims[3] = {128, 1, 128};
    cuuint64_t strides[2] = {256, 256};
    cuuint32_t box[3] = {64, 1, 128};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fi::g_encode(&p.tmap_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return 4;
  }
  p.a = static_cast<const uint16_t*>(a);
  p.b = static_cast<const uint16_t*>(b);
  p.c = c;
  p.status = status;
  p.mode = mode;
  const int smem = 65536 + 64 + 1024;
  if (cudaFuncSetAttribute(fi::umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return 4;
  fi::umma_probe_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int32_t fi_diag_umma_pair(int32_t mode, const void* a, const void* b, float* c, int32_t* status,
                          uint32_t* tmem_addrs, void* stream) {
  if ((mode != 0 && mode != 1) || !a || !b || !c || !status || !tmem_addrs || !fi::a16(a) ||
      !fi::a16(b))
    return 1;
  fi::UmmaPairParams p;
  p.a = static_cast<const uint16_t*>(a);
  p.b = static_cast<const uint16_t*>(b);
  p.c = c;
  p.status = status;
  p.tmem_addrs = tmem_addrs;
  p.mode = mode;
  const int smem = 49152 + 64 + 1024;
  if (cudaFuncSetAttribute(fi::umma_pair_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return 4;
  fi::umma_pair_probe_kernel<<<2, 128, smem, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

int32_t fi_diag_wait_timeout(uint64_t timeout_ns, const uint8_t* copy_src, uint8_t* copy_out,
                             int32_t* status, unsigned long long* report, void* stream) {
  if (!copy_src || !copy_out || !status || !report || !fi::a16(copy_src) || !fi::a16(copy_out) ||
      timeout_ns == 0 || timeout_ns > 1000000000ull)
    return 1;
  fi::wait_timeout_probe_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(
      timeout_ns, copy_src, copy_out, status, report);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

}  // extern "C"
