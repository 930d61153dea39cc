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

struct Quant16 {
  uint32_t lo, hi;  // 16 E2M1 codes, element 2c in the low nibble of byte c
  uint32_t s8;      // the block's E4M3 scale byte
};

// Division by the block's decode scale d, correctly rounded, without an IEEE
// divide per element.  Markstein's theorem (P. W. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): if r is 1/d rounded to nearest and q0 = RN(x r) (within
// one ulp of x/d), the residual e = x - q0 d is exact when computed with one
// fused multiply-add, and RN(q0 + e r) is x/d rounded to nearest.  The
// hypotheses (no overflow, no underflow of q0 or e) hold for every element of
// a block when d is in [2^-98, 2^100] and amax <= 2^100 d: an element with
// |x| >= 2^-100 has an exact residual, and one with |x| < 2^-100 has
// |x/d| < 1/4, where every value within a few ulps encodes to the same E2M1
// code (0, or 8 for negative inputs).  Callers outside that range use the
// IEEE division itself.
// Signed zeros: the residual is computed rounding toward -infinity.  An exact
// residual does not depend on the rounding direction, except that an exact
// zero comes out as -0 (IEEE 754, section 6.3).  So a zero input x = s0
// gives q0 = s0, e = -0 and q1 = -0 * r + s0 = s0, the sign an IEEE division
// gives, and a nonzero input is unaffected (q0 + (-0) = q0).
__device__ __forceinline__ bool markstein_range_ok(float d, float amax) {
  return d >= 0x1p-98f && d <= 0x1p100f && amax <= d * 0x1p100f;
}

// Two elements with paired fp32 arithmetic (each lane one IEEE operation;
// fma(q0, -d, x) computes x - q0 d).
__device__ __forceinline__ void div_markstein_x2(float& x0, float& x1, uint64_t d2n,
                                                 uint64_t r2) {
  const uint64_t x2 = f2_pack(x0, x1);
  const uint64_t q0 = f2_mul(x2, r2);
  const uint64_t e = f2_fma_rm(q0, d2n, x2);
  f2_unpack(f2_fma(e, r2, q0), x0, x1);
}

// Quantizes one 16-element NVFP4 block with global decode scale g:
//   amax = max |x_j|, t = amax / RN(6 g), s8 = e4m3(t), d = RN(e4m3(s8) g),
//   code_j = e2m1(RN(x_j / d));
// every step rounds like one IEEE fp32 operation (no contraction).  A block
// with amax == 0, or whose s8 encodes 0, stores s8 = 0 and all-zero codes.
__device__ __forceinline__ Quant16 quantize16(const float (&x)[16], float g) {
  Quant16 q{0u, 0u, 0u};
  // elements 0..14 in seven three-input steps, then element 15
  float amax = fabsf(x[0]);
#pragma unroll
  for (int j = 1; j < 15; j += 2) amax = fmax3(amax, fabsf(x[j]), fabsf(x[j + 1]));
  amax = fmaxf(amax, fabsf(x[15]));
  if (amax == 0.0f) return q;
  const float t = __fdiv_rn(amax, __fmul_rn(6.0f, g));
  const uint32_t s = e4m3_from_f32(t);
  const float sv = e4m3_value(s);
  if (sv == 0.0f) return q;
  const float d = __fmul_rn(sv, g);
  float y[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) y[j] = x[j];
  if (markstein_range_ok(d, amax)) {
    const float r = __frcp_rn(d);
    const uint64_t r2 = f2_pack(r, r), d2n = f2_pack(-d, -d);
#pragma unroll
    for (int j = 0; j < 16; j += 2) div_markstein_x2(y[j], y[j + 1], d2n, r2);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) y[j] = __fdiv_rn(x[j], d);
  }
  q.lo = e2m1x4_from_f32(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
  q.hi = e2m1x4_from_f32(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
  q.s8 = s;
  return q;
}

// 8 bf16 values (one 128-bit word) -> fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* x) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = __uint_as_float(v[j] << 16);
    x[2 * j + 1] = __uint_as_float(v[j] & 0xFFFF0000u);
  }
}

// Per-tensor constants of the quantizer that depend only on g or on the scale
// byte, computed once per CTA instead of once per block:
//   d6 = RN(6 g), r6 = RN(1 / d6), lim6 = d6 * 2^100 when d6 is in the
//   Markstein range (else -1, which sends every block to the IEEE division);
//   per E4M3 code s in [0, 127]: d = RN(e4m3(s) g), r = RN(1 / d) and
//   lim = d * 2^100 when d is in range (else -1).
// quantize16_tab with these constants stores the same bytes as quantize16.
struct QuantConsts {
  float d6, r6, lim6;
};

__device__ __forceinline__ QuantConsts quant_consts(float g) {
  QuantConsts c;
  c.d6 = __fmul_rn(6.0f, g);
  c.r6 = __frcp_rn(c.d6);
  c.lim6 = (c.d6 >= 0x1p-98f && c.d6 <= 0x1p100f) ? c.d6 * 0x1p100f : -1.0f;
  return c;
}

__device__ __forceinline__ float4 quant_scale_entry(uint32_t s, float g) {
  const float d = __fmul_rn(e4m3_value(s), g);
  const float lim = (d >= 0x1p-98f && d <= 0x1p100f) ? d * 0x1p100f : -1.0f;
  return make_float4(d, __frcp_rn(d), lim, 0.0f);
}

// max |x| of 16 bf16 values (two 128-bit words) as fp32, computed on the
// packed halves: exact (a maximum), NaN halves ignored like fmaxf.
__device__ __forceinline__ float amax16_bf16(const uint4& w0, const uint4& w1) {
  const uint32_t m = bmax_abs2(bmax_abs2(bmax_abs2(w0.x, w0.y), bmax_abs2(w0.z, w0.w)),
                               bmax_abs2(bmax_abs2(w1.x, w1.y), bmax_abs2(w1.z, w1.w)));
  const uint32_t m2 = bmax_abs2(m, __byte_perm(m, 0u, 0x1032));
  return __uint_as_float((m2 & 0x7FFFu) << 16);
}

// quantize16 with the constants above.  The block scale t = amax / d6 is
// also divided by Markstein's method: amax >= 2^-100 makes its residual
// exact, and a quotient below the fp32 normal range rounds to the E4M3 code 0
// either way.  tab: the 128 entries of quant_scale_entry for this tensor.
// Input: the block's 16 bf16 values as two 128-bit words.
__device__ __forceinline__ Quant16 quantize16_tab(const uint4& w0, const uint4& w1,
                                                 const QuantConsts& c, const float4* tab) {
  Quant16 q{0u, 0u, 0u};
  const float amax = amax16_bf16(w0, w1);
  if (amax == 0.0f) return q;
  float t;
  if (amax >= 0x1p-100f && amax <= c.lim6) {
    const float q0 = __fmul_rn(amax, c.r6);
    t = __fmaf_rn(__fmaf_rn(-q0, c.d6, amax), c.r6, q0);
  } else {
    t = __fdiv_rn(amax, c.d6);
  }
  const uint32_t s = e4m3_from_f32(t);
  if (s == 0u) return q;  // t >= 0: code 0 is the only zero
  const float4 e = tab[s & 0x7Fu];
  float x[16];
  bf16x8_to_f32(w0, x);
  bf16x8_to_f32(w1, x + 8);
  float y[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) y[j] = x[j];
  if (amax <= e.z) {
    const uint64_t r2 = f2_pack(e.y, e.y), d2n = f2_pack(-e.x, -e.x);
#pragma unroll
    for (int j = 0; j < 16; j += 2) div_markstein_x2(y[j], y[j + 1], d2n, r2);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) y[j] = __fdiv_rn(x[j], e.x);
  }
  q.lo = e2m1x4_from_f32(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
  q.hi = e2m1x4_from_f32(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
  q.s8 = s;
  return q;
}

// --- FP8 (E4M3) per-element codes ---------------------------------------
// code = e4m3(RN(x / g)) for every element, one fp32 decode scale g per
// tensor.  The division is Markstein's (as above) when every element of the
// 16-element group is zero or has |x| in [2^-100, L), L = 2^100 g rounded
// down to bf16 (and g itself in [2^-98, 2^100]); otherwise the IEEE division.
// The group test runs on the packed bf16 magnitudes with 16-bit integer
// max/min (zeros are moved to the top of the range by subtracting one).
struct Fp8Consts {
  float g, r;      // decode scale and RN(1 / g)
  uint32_t lim16;  // bf16 bits of L rounded down (0: no fast path)
};

__device__ __forceinline__ Fp8Consts fp8_consts(float g) {
  Fp8Consts c;
  c.g = g;
  c.r = __frcp_rn(g);
  const bool ok = g >= 0x1p-98f && g <= 0x1p100f;
  c.lim16 = ok ? (__float_as_uint(g * 0x1p100f) >> 16) & 0x7FFFu : 0u;
  return c;
}

// Two bf16 words (16 values) -> 16 E4M3 codes, byte e = element e.
__device__ __forceinline__ uint4 fp8_quantize16(const uint4& w0, const uint4& w1,
                                               const Fp8Consts& c) {
  const uint32_t w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  uint32_t mx = 0u, mn = 0xFFFFFFFFu;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t a = w[k] & 0x7FFF7FFFu;
    mx = __vmaxu2(mx, a);
    mn = __vminu2(mn, __vsub2(a, 0x00010001u));
  }
  const uint32_t mx16 = max(mx & 0xFFFFu, mx >> 16);
  const uint32_t mn16 = min(mn & 0xFFFFu, mn >> 16);
  // 0x0D80: bf16 bits of 2^-100; zeros became 0xFFFF above.  lim16 is 0 when
  // g is outside [2^-98, 2^100] (its reciprocal may be infinite): then no
  // group, not even an all-zero one, takes the fast path.
  const bool fast = mx16 < c.lim16 && mn16 >= 0x0D7Fu;
  float x[16];
  bf16x8_to_f32(w0, x);
  bf16x8_to_f32(w1, x + 8);
  if (fast) {
    const uint64_t r2 = f2_pack(c.r, c.r), g2n = f2_pack(-c.g, -c.g);
#pragma unroll
    for (int j = 0; j < 16; j += 2) div_markstein_x2(x[j], x[j + 1], g2n, r2);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) x[j] = __fdiv_rn(x[j], c.g);
  }
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = e4m3x4_from_f32(x[4 * k], x[4 * k + 1], x[4 * k + 2], x[4 * k + 3]);
  return make_uint4(o[0], o[1], o[2], o[3]);
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
// at or beyond `valid` are written as zeros.  Thread `tid` of NT (NT a
// multiple of D/8 and of 64) converts 8 elements per task: task t is row
// t / (D/8), chunk t % (D/8); consecutive threads read consecutive 32-bit
// words and write distinct 16-byte chunk positions of one row, so neither the
// loads nor the swizzled stores conflict on shared-memory banks.  A thread's
// tasks keep its chunk and the row's phase in the swizzle, so its addresses
// advance by constant strides.  Full tiles take a branch-free path in batches
// of four tasks, the batch's loads issued before its conversions (the
// conversions of different tasks are independent, which keeps the warp busy
// within a small register budget).
template <int D, bool IS_V, int NT>
__device__ __forceinline__ void repack_tile(const uint8_t* raw, uint8_t* dst, int valid,
                                            int tid) {
  static_assert(NT % (D / 8) == 0 && NT % 64 == 0, "constant-stride tasks");
  constexpr int kPer = 128 * (D / 8) / NT;       // tasks per thread
  constexpr int kRowStep = NT / (D / 8);         // rows between a thread's tasks
  const uint32_t* words = reinterpret_cast<const uint32_t*>(raw);
  const uint8_t* sf = raw + 128 * (D / 2);
  const int c = tid % (D / 8);
  const int row0 = tid / (D / 8);
  const uint32_t off0 = sw128_offset(row0, c);
  if (valid >= 128) {
    // batches of kBatch tasks: the batch's loads, then its conversions
    constexpr int kBatch = kPer < 4 ? kPer : 4;
#pragma unroll 1
    for (int k0 = 0; k0 < kPer; k0 += kBatch) {
      uint32_t w[kBatch], s8[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        w[k] = words[tid + (k0 + k) * NT];
        s8[k] = sf[(row0 + (k0 + k) * kRowStep) * (D / 16) + c / 2];
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const uint4 o = IS_V ? dequant8_f16(w[k], s8[k]) : dequant8_bf16(w[k], s8[k]);
        *reinterpret_cast<uint4*>(dst + off0 + (k0 + k) * kRowStep * 128) = o;
      }
    }
  } else {
#pragma unroll 4
    for (int k = 0; k < kPer; ++k) {
      const int row = row0 + k * kRowStep;
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (row < valid) {
        const uint32_t s8 = sf[row * (D / 16) + c / 2];
        o = IS_V ? dequant8_f16(words[tid + k * NT], s8) : dequant8_bf16(words[tid + k * NT], s8);
      }
      *reinterpret_cast<uint4*>(dst + off0 + k * kRowStep * 128) = o;
    }
  }
}

// Repacks half a tile, for a pair of CTAs that share their staging tiles:
// `raw` holds 64 token rows (D/2 code bytes each, then 64 rows of D/16 scale
// bytes); they become rows row_base .. row_base+63 of the staging tile `dst`
// (the other CTA receives them by a bulk copy).  Rows at or beyond `valid`
// (of the 64) are written as zeros.  Same task layout and store order as
// repack_tile; row_base is a multiple of 8, so the swizzle phase is unchanged.
template <int D, bool IS_V, int NT>
__device__ __forceinline__ void repack_half(const uint8_t* raw, uint8_t* dst, int row_base,
                                            int valid, int tid) {
  static_assert(NT % (D / 8) == 0 && NT % 64 == 0, "constant-stride tasks");
  constexpr int kPer = 64 * (D / 8) / NT;        // tasks per thread
  constexpr int kRowStep = NT / (D / 8);
  constexpr int kBatch = kPer < 4 ? kPer : 4;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(raw);
  const uint8_t* sf = raw + 64 * (D / 2);
  const int c = tid % (D / 8);
  const int row0 = tid / (D / 8);
  const uint32_t off0 = sw128_offset(row_base + row0, c);
#pragma unroll 1
  for (int k0 = 0; k0 < kPer; k0 += kBatch) {
    uint32_t w[kBatch], s8[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      w[k] = words[tid + (k0 + k) * NT];
      s8[k] = sf[(row0 + (k0 + k) * kRowStep) * (D / 16) + c / 2];
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (row0 + (k0 + k) * kRowStep < valid)
        o = IS_V ? dequant8_f16(w[k], s8[k]) : dequant8_bf16(w[k], s8[k]);
      *reinterpret_cast<uint4*>(dst + off0 + (k0 + k) * kRowStep * 128) = o;
    }
  }
}

// --- FP8 (E4M3) tiles ------------------------------------------------------
// Eight E4M3 codes (8 bytes, element e in byte e) -> 8 fp16 values (exact:
// every E4M3 value is zero or an fp16 normal).
__device__ __forceinline__ uint4 fp8x8_to_f16(uint2 w) {
  uint4 o;
  o.x = e4m3x2_to_f16x2(w.x & 0xFFFFu);
  o.y = e4m3x2_to_f16x2(w.x >> 16);
  o.z = e4m3x2_to_f16x2(w.y & 0xFFFFu);
  o.w = e4m3x2_to_f16x2(w.y >> 16);
  return o;
}
// The same as bf16: the fp16 values are moved to bf16 bit patterns of
// value * 2^-112 (at most 4 significant bits, zero or normal) and multiplied
// by 2^112 in bf16 (both steps exact).
__device__ __forceinline__ uint4 fp8x8_to_bf16(uint2 w) {
  const uint4 h = fp8x8_to_f16(w);
  const uint32_t m = 0x77807780u;  // bf16x2 (2^112, 2^112)
  return make_uint4(bmul2_u32(f16x2_to_bf16x2_scaled(h.x), m),
                    bmul2_u32(f16x2_to_bf16x2_scaled(h.y), m),
                    bmul2_u32(f16x2_to_bf16x2_scaled(h.z), m),
                    bmul2_u32(f16x2_to_bf16x2_scaled(h.w), m));
}

// Repacks a raw FP8 KV tile (128 rows of D code bytes) into the 16-bit
// staging tile, as repack_tile does for NVFP4 (K as bf16, V as fp16; rows at
// or beyond `valid` written as zeros).  Task t (8 elements) is row t / (D/8),
// chunk t % (D/8), read as one 8-byte word.
template <int D, bool IS_V, int NT>
__device__ __forceinline__ void repack_tile_fp8(const uint8_t* raw, uint8_t* dst, int valid,
                                                int tid) {
  static_assert(NT % (D / 8) == 0 && NT % 64 == 0, "constant-stride tasks");
  constexpr int kPer = 128 * (D / 8) / NT;
  constexpr int kRowStep = NT / (D / 8);
  const uint2* words = reinterpret_cast<const uint2*>(raw);
  const int c = tid % (D / 8);
  const int row0 = tid / (D / 8);
  const uint32_t off0 = sw128_offset(row0, c);
#pragma unroll 4
  for (int k = 0; k < kPer; ++k) {
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (row0 + k * kRowStep < valid) {
      const uint2 w = words[tid + k * NT];
      o = IS_V ? fp8x8_to_f16(w) : fp8x8_to_bf16(w);
    }
    *reinterpret_cast<uint4*>(dst + off0 + k * kRowStep * 128) = o;
  }
}

// Half tile (64 raw rows) into rows row_base .. row_base+63 of the staging
// tile, as repack_half does for NVFP4.
template <int D, bool IS_V, int NT>
__device__ __forceinline__ void repack_half_fp8(const uint8_t* raw, uint8_t* dst, int row_base,
                                                int valid, int tid) {
  static_assert(NT % (D / 8) == 0 && NT % 64 == 0, "constant-stride tasks");
  constexpr int kPer = 64 * (D / 8) / NT;
  constexpr int kRowStep = NT / (D / 8);
  const uint2* words = reinterpret_cast<const uint2*>(raw);
  const int c = tid % (D / 8);
  const int row0 = tid / (D / 8);
  const uint32_t off0 = sw128_offset(row_base + row0, c);
#pragma unroll 4
  for (int k = 0; k < kPer; ++k) {
    uint4 o = make_uint4(0u, 0u, 0u, 0u);
    if (row0 + k * kRowStep < valid) {
      const uint2 w = words[tid + k * NT];
      o = IS_V ? fp8x8_to_f16(w) : fp8x8_to_bf16(w);
    }
    *reinterpret_cast<uint4*>(dst + off0 + k * kRowStep * 128) = o;
  }
}

}  // namespace fi
