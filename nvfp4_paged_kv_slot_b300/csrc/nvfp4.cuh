// nvfp4.cuh — device-side NVFP4 quantization and the 16-bit staging layout.
//
// NVFP4 here: E2M1 codes with one E4M3 scale per 16 head-dim elements and one
// positive finite fp32 global decode scale g per tensor (FlashInfer PR #6204
// analysis page, "FlashInfer: NVFP4 KV 캐시 어펜드 성능 최적화로 인한 동기화 제거",
// k_scale/v_scale docstring).  Rounding: nearest, ties to even, saturating,
// sign kept — the native sm_100-family cvt instructions.
#pragma once

#include "ptx.cuh"

namespace fi {

// Value of an E4M3 byte as fp32 (exact; via the native fp16 conversion).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2 = e4m3_to_f16x2_dup(code);
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

struct Quant8 {
  uint32_t codes;  // 8 E2M1 codes, element 2c in the low nibble of byte c
  uint32_t s8;     // the block's E4M3 scale byte
};

// Quantizes 8 of the 16 elements of one NVFP4 block.  `amax` is the maximum
// magnitude over all 16 elements of the block, `g` the global decode scale.
// Each step is one fp32 IEEE operation (explicit _rn intrinsics: no fused
// multiply-add, IEEE division):
//   t = amax / (6 g), s8 = e4m3(t); d = e4m3(s8) g; code_j = e2m1(x_j / d);
// a block with amax == 0 or with s8 == 0 stores s8 = 0 and all-zero codes.
__device__ __forceinline__ Quant8 quantize8(const float (&x)[8], float amax, float g) {
  Quant8 q{0u, 0u};
  if (amax == 0.0f) return q;
  const float t = __fdiv_rn(amax, __fmul_rn(6.0f, g));
  const uint32_t s = e4m3_from_f32(t);
  const float sv = e4m3_value(s);
  if (sv == 0.0f) return q;
  const float d = __fmul_rn(sv, g);
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = __fdiv_rn(x[j], d);
  q.codes = e2m1x4_from_f32(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
  q.s8 = s;
  return q;
}

// --- 16-bit staging tile ------------------------------------------------------
// A [128 rows][D] tile of 16-bit values is stored as D/64 column blocks of
// [128 rows][64 elements] (16 KB each), rows 128 B apart, with the 128-byte
// swizzle the tensor cores expect: 16-byte chunk c of row r sits at chunk
// position c ^ (r % 8).  The same bytes serve as a K-major operand (rows = MMA
// N, 64-element column blocks = K blocks) and as an MN-major operand (rows =
// MMA K, column blocks = MN blocks 16 KB apart).  The tile base is 1024-byte
// aligned.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return (chunk >> 3) * (128u * 128u) + row * 128u + (((chunk & 7u) ^ (row & 7u)) << 4);
}

// Dequantizes 8 E2M1 codes sharing the E4M3 scale byte s8 to 8 bf16 values
// e2m1 * e4m3(s8), exactly: such a product has at most 6 significant bits and
// a magnitude in [2^-10, 2688], so bf16 holds it.  The codes are widened to
// fp16 natively, reinterpreted as bf16 * 2^-112, and multiplied by
// e4m3(s8) * 2^112 in bf16 (both factors and the product exact).
__device__ __forceinline__ uint4 dequant8_bf16(uint32_t w, uint32_t s8) {
  uint32_t h[4];
  e2m1x8_to_f16x2(w, h);
  const float m = e4m3_value(s8) * 0x1p112f;
  const __nv_bfloat162 mb = __floats2bfloat162_rn(m, m);
  const uint32_t mu = *reinterpret_cast<const uint32_t*>(&mb);
  uint4 o;
  o.x = bmul2_u32(f16x2_to_bf16x2_scaled(h[0]), mu);
  o.y = bmul2_u32(f16x2_to_bf16x2_scaled(h[1]), mu);
  o.z = bmul2_u32(f16x2_to_bf16x2_scaled(h[2]), mu);
  o.w = bmul2_u32(f16x2_to_bf16x2_scaled(h[3]), mu);
  return o;
}

// Same values as fp16 (exact for the same reason; fp16 covers [2^-14, 65504]).
__device__ __forceinline__ uint4 dequant8_f16(uint32_t w, uint32_t s8) {
  uint32_t h[4];
  e2m1x8_to_f16x2(w, h);
  const uint32_t s2 = e4m3_to_f16x2_dup(s8);
  uint4 o;
  o.x = hmul2_u32(h[0], s2);
  o.y = hmul2_u32(h[1], s2);
  o.z = hmul2_u32(h[2], s2);
  o.w = hmul2_u32(h[3], s2);
  return o;
}

// Repacks one raw NVFP4 KV tile (128 token rows of D/2 code bytes, then 128
// rows of D/16 scale bytes, as copied from the cache pages) into the 16-bit
// staging tile: K as bf16 (operand of QK^T), V as fp16 (operand of PV).  Rows
// at or beyond `valid` are written as zeros.  Thread `tid` of `nthreads`
// converts 8 elements per step: consecutive threads read consecutive 32-bit
// words and write distinct 16-byte chunk positions of one row, so neither the
// loads nor the swizzled stores conflict on shared-memory banks.
template <int D, bool IS_V>
__device__ __forceinline__ void repack_tile(const uint8_t* raw, uint8_t* dst, int valid, int tid,
                                            int nthreads) {
  const uint32_t* words = reinterpret_cast<const uint32_t*>(raw);
  const uint8_t* sf = raw + 128 * (D / 2);
#pragma unroll 4
  for (int task = tid; task < 128 * (D / 8); task += nthreads) {
    const int row = task / (D / 8);
    const int c = task % (D / 8);
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (row < valid) {
      const uint32_t w = words[task];
      const uint32_t s8 = sf[row * (D / 16) + c / 2];
      o = IS_V ? dequant8_f16(w, s8) : dequant8_bf16(w, s8);
    }
    *reinterpret_cast<uint4*>(dst + sw128_offset(row, c)) = o;
  }
}

}  // namespace fi
