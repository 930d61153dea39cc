// oracle.cpp — plain CPU reference.  TEST INFRASTRUCTURE ONLY (see oracle.h).
//
// Build flags matter: -O2 -ffp-contract=off, no -ffast-math, so that every fp32
// step below is one IEEE operation rounded to nearest even, in source order.
#include "oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

float bf16_to_float(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// E2M1 magnitude of the 3-bit code c (OCP MX v1.0, FP4 E2M1: bias 1,
// exponent 0 is subnormal with step 0.5).
double e2m1_magnitude(int c) {
  int e = (c >> 1) & 3;
  int m = c & 1;
  if (e == 0) return 0.5 * m;
  return std::ldexp(1.0 + m / 2.0, e - 1);
}

// E4M3 ("FN": no infinities, S.1111.111 is NaN) magnitude of the 7-bit code
// (OCP MX v1.0, FP8 E4M3: bias 7, exponent 0 is subnormal with step 2^-9).
double e4m3_magnitude(int c) {
  int e = (c >> 3) & 15;
  int m = c & 7;
  if (e == 15 && m == 7) return std::nan("");
  if (e == 0) return m * std::ldexp(1.0, -9);
  return std::ldexp(1.0 + m / 8.0, e - 7);
}

}  // namespace

extern "C" {

double orc_e2m1_value(uint8_t code) {
  double v = e2m1_magnitude(code & 7);
  return (code & 8) ? -v : v;
}

double orc_e4m3_value(uint8_t code) {
  double v = e4m3_magnitude(code & 0x7F);
  return (code & 0x80) ? -v : v;
}

// Nearest E2M1 value by exhaustive search over the 8 magnitudes, in double
// (every fp32 input and every E2M1 value is exact in double, so distances are
// exact).  Ties go to the even code; magnitudes above 6 saturate to 6; the
// sign bit of the input is kept, so negative inputs that round to zero give
// code 0x8.  NaN input is not specified by the format; this returns the
// saturated magnitude with the input's sign.
uint8_t orc_e2m1_encode(float y) {
  uint8_t sign = std::signbit(y) ? 0x8 : 0x0;
  if (std::isnan(y)) return sign | 0x7;
  double a = std::fabs(static_cast<double>(y));
  if (a > 6.0) return sign | 0x7;
  int best = 0;
  double best_dist = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double dist = std::fabs(e2m1_magnitude(c) - a);
    if (dist < best_dist || (dist == best_dist && (c & 1) == 0)) {
      best = c;
      best_dist = dist;
    }
  }
  return sign | static_cast<uint8_t>(best);
}

// Nearest E4M3 value by exhaustive search over the 127 finite magnitudes.
// Same tie, saturation (448) and sign rules; NaN input gives the NaN code.
uint8_t orc_e4m3_encode(float t) {
  uint8_t sign = std::signbit(t) ? 0x80 : 0x00;
  if (std::isnan(t)) return sign | 0x7F;
  double a = std::fabs(static_cast<double>(t));
  if (a > 448.0) return sign | 0x7E;
  int best = 0;
  double best_dist = INFINITY;
  for (int c = 0; c < 0x7F; ++c) {
    double dist = std::fabs(e4m3_magnitude(c) - a);
    if (dist < best_dist || (dist == best_dist && (c & 1) == 0)) {
      best = c;
      best_dist = dist;
    }
  }
  return sign | static_cast<uint8_t>(best);
}

// Bit-level version of orc_e4m3_encode: the same rule computed from the fp32
// bit pattern (rebias the exponent, round the 23-bit mantissa to 3 bits to
// nearest even; the subnormal range is an integer rounding of t * 2^9).
uint8_t orc_e4m3_encode_bits(float t) {
  uint32_t u;
  std::memcpy(&u, &t, 4);
  uint8_t sign = static_cast<uint8_t>((u >> 24) & 0x80);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return sign | 0x7F;          // NaN
  if (a > 0x43E00000u) return sign | 0x7E;          // above 448 (incl. inf)
  if (a < 0x3C800000u) {                            // below 2^-6: subnormal
    float s = std::fabs(t) * 512.0f;                // exact power-of-two scaling
    float r = std::nearbyint(s);                    // default mode: nearest even
    return sign | static_cast<uint8_t>(r);          // 0..8 (8 == 2^-6, code 0x08)
  }
  uint32_t x = a - ((127u - 7u) << 23);
  uint32_t lsb = (x >> 20) & 1u;
  x += 0x7FFFFu + lsb;
  uint32_t code = x >> 20;
  if (code > 0x7Eu) code = 0x7Eu;
  return sign | static_cast<uint8_t>(code);
}

// Bit-level version of orc_e2m1_encode (subnormal step 0.5 below 1.0).
uint8_t orc_e2m1_encode_bits(float y) {
  uint32_t u;
  std::memcpy(&u, &y, 4);
  uint8_t sign = static_cast<uint8_t>((u >> 28) & 0x8);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a > 0x7F800000u) return sign | 0x7;           // NaN
  if (a > 0x40C00000u) return sign | 0x7;           // above 6 (incl. inf)
  if (a < 0x3F800000u) {                            // below 1: subnormal
    float s = std::fabs(y) * 2.0f;
    float r = std::nearbyint(s);                    // 0, 1 or 2 (2 == 1.0)
    return sign | static_cast<uint8_t>(r);
  }
  uint32_t x = a - ((127u - 1u) << 23);
  uint32_t lsb = (x >> 22) & 1u;
  x += 0x1FFFFFu + lsb;
  uint32_t code = x >> 22;
  if (code > 0x7u) code = 0x7u;
  return sign | static_cast<uint8_t>(code);
}

void orc_e2m1_encode_span(uint32_t first_bits, uint64_t count, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < static_cast<int64_t>(count); ++i) {
    uint32_t b = first_bits + static_cast<uint32_t>(i);
    float y;
    std::memcpy(&y, &b, 4);
    out[i] = orc_e2m1_encode_bits(y);
  }
}

void orc_e4m3_encode_span(uint32_t first_bits, uint64_t count, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < static_cast<int64_t>(count); ++i) {
    uint32_t b = first_bits + static_cast<uint32_t>(i);
    float t;
    std::memcpy(&t, &b, 4);
    out[i] = orc_e4m3_encode_bits(t);
  }
}

void orc_e2m1_encode_array(const float* in, int64_t n, int32_t mode, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = mode ? orc_e2m1_encode_bits(in[i]) : orc_e2m1_encode(in[i]);
}

void orc_e4m3_encode_array(const float* in, int64_t n, int32_t mode, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = mode ? orc_e4m3_encode_bits(in[i]) : orc_e4m3_encode(in[i]);
}

// One NVFP4 block: 16 consecutive head-dim elements share one E4M3 scale s8,
// and the tensor's positive finite global decode scale g multiplies every
// element ([#6204] k_scale/v_scale docstring: "Positive finite global decode
// scale").  Steps, each an fp32 IEEE operation:
//   amax = max |x_j|
//   amax == 0            -> s8 = 0, every code 0
//   t = amax / (6 * g)   (6*g rounded first), s8 = e4m3(t)
//   e4m3(s8) == 0        -> s8 = 0, every code 0   (underflow; reading)
//   d = e4m3(s8) * g,  q_j = e2m1(x_j / d)
// Byte c of the packed output holds q_{2c} in its low nibble.
void orc_quantize_block16(const uint16_t* x, float g, uint8_t* packed, uint8_t* s8) {
  float xf[16];
  float amax = 0.0f;
  for (int j = 0; j < 16; ++j) {
    xf[j] = bf16_to_float(x[j]);
    amax = std::max(amax, std::fabs(xf[j]));
  }
  std::memset(packed, 0, 8);
  *s8 = 0;
  if (amax == 0.0f) return;
  float six_g = 6.0f * g;
  float t = amax / six_g;
  uint8_t s = orc_e4m3_encode(t);
  float s_val = static_cast<float>(orc_e4m3_value(s));
  if (s_val == 0.0f) return;
  float d = s_val * g;
  uint8_t q[16];
  for (int j = 0; j < 16; ++j) q[j] = orc_e2m1_encode(xf[j] / d);
  for (int c = 0; c < 8; ++c) packed[c] = static_cast<uint8_t>(q[2 * c] | (q[2 * c + 1] << 4));
  *s8 = s;
}

// The slot_mapping append ([#6204] "nvfp4_quantize_append_paged_kv_cache_with_
// slot_mapping"): token i goes to slot slot_mapping[i] = page * ps + offset of
// every kv head; a negative slot means "do not write".  A CUDA-tensor scale is
// checked where the rows are written: a scale that is not positive and finite
// is an error and, here, nothing is written.
int orc_append(const uint16_t* k, const uint16_t* v, int64_t num_tokens,
               int64_t k_tok_stride, int64_t v_tok_stride, int32_t num_kv_heads,
               int32_t head_dim, float k_scale, float v_scale,
               const int64_t* slot_mapping, uint8_t* k_data, uint8_t* v_data,
               uint8_t* k_sf, uint8_t* v_sf, int32_t num_pages, int32_t page_size) {
  int status = 0;
  if (!(std::isfinite(k_scale) && k_scale > 0.0f)) status |= ORC_BAD_K_SCALE;
  if (!(std::isfinite(v_scale) && v_scale > 0.0f)) status |= ORC_BAD_V_SCALE;
  if (status != 0) return status;
  const int64_t num_slots = static_cast<int64_t>(num_pages) * page_size;
  const int32_t blocks = head_dim / 16;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      status |= ORC_SLOT_OOB;
      continue;
    }
    int64_t page = slot / page_size;
    int64_t off = slot % page_size;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      int64_t row = (page * num_kv_heads + h) * page_size + off;
      for (int32_t b = 0; b < blocks; ++b) {
        orc_quantize_block16(k + i * k_tok_stride + h * head_dim + b * 16, k_scale,
                             k_data + row * (head_dim / 2) + b * 8, k_sf + row * blocks + b);
        orc_quantize_block16(v + i * v_tok_stride + h * head_dim + b * 16, v_scale,
                             v_data + row * (head_dim / 2) + b * 8, v_sf + row * blocks + b);
      }
    }
  }
  return status;
}

void orc_dequant_row(const uint8_t* data, const uint8_t* sf, int32_t num_kv_heads,
                     int32_t head_dim, int32_t page_size, int64_t slot, int32_t head,
                     double g, double* out) {
  int64_t page = slot / page_size;
  int64_t off = slot % page_size;
  int64_t row = (page * num_kv_heads + head) * page_size + off;
  const uint8_t* d = data + row * (head_dim / 2);
  const uint8_t* s = sf + row * (head_dim / 16);
  for (int32_t e = 0; e < head_dim; ++e) {
    uint8_t byte = d[e / 2];
    uint8_t code = (e % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    out[e] = orc_e2m1_value(code) * orc_e4m3_value(s[e / 16]) * g;
  }
}

// FP8 (E4M3) paged KV: every element is divided by the tensor's decode scale
// (one fp32 IEEE division) and rounded to the nearest E4M3 value by the
// exhaustive encoder above (ties to even, saturating at 448, sign kept).
uint8_t orc_fp8_quantize(float x, float g) { return orc_e4m3_encode(x / g); }

int orc_fp8_append(const uint16_t* k, const uint16_t* v, int64_t num_tokens,
                   int64_t k_tok_stride, int64_t v_tok_stride, int32_t num_kv_heads,
                   int32_t head_dim, float k_scale, float v_scale,
                   const int64_t* slot_mapping, uint8_t* k_data, uint8_t* v_data,
                   int32_t num_pages, int32_t page_size) {
  int status = 0;
  if (!(std::isfinite(k_scale) && k_scale > 0.0f)) status |= ORC_BAD_K_SCALE;
  if (!(std::isfinite(v_scale) && v_scale > 0.0f)) status |= ORC_BAD_V_SCALE;
  if (status != 0) return status;
  const int64_t num_slots = static_cast<int64_t>(num_pages) * page_size;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      status |= ORC_SLOT_OOB;
      continue;
    }
    int64_t page = slot / page_size;
    int64_t off = slot % page_size;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      int64_t row = (page * num_kv_heads + h) * page_size + off;
      for (int32_t e = 0; e < head_dim; ++e) {
        k_data[row * head_dim + e] =
            orc_fp8_quantize(bf16_to_float(k[i * k_tok_stride + h * head_dim + e]), k_scale);
        v_data[row * head_dim + e] =
            orc_fp8_quantize(bf16_to_float(v[i * v_tok_stride + h * head_dim + e]), v_scale);
      }
    }
  }
  return status;
}

void orc_fp8_dequant_row(const uint8_t* data, int32_t num_kv_heads, int32_t head_dim,
                         int32_t page_size, int64_t slot, int32_t head, double g, double* out) {
  int64_t page = slot / page_size;
  int64_t off = slot % page_size;
  int64_t row = (page * num_kv_heads + head) * page_size + off;
  for (int32_t e = 0; e < head_dim; ++e) out[e] = orc_e4m3_value(data[row * head_dim + e]) * g;
}

void orc_dense_causal(const double* q, const double* k, const double* v, int32_t L_q,
                      int32_t L_kv, int32_t head_dim, double sm_scale, double* out,
                      double* lse) {
  std::vector<double> s(L_kv);
  for (int32_t i = 0; i < L_q; ++i) {
    int32_t last = i + L_kv - L_q;
    double m = -INFINITY;
    for (int32_t j = 0; j <= last; ++j) {
      double dot = 0.0;
      for (int32_t e = 0; e < head_dim; ++e) dot += q[i * head_dim + e] * k[j * head_dim + e];
      s[j] = sm_scale * dot;
      m = std::max(m, s[j]);
    }
    double l = 0.0;
    for (int32_t e = 0; e < head_dim; ++e) out[i * head_dim + e] = 0.0;
    for (int32_t j = 0; j <= last; ++j) {
      double p = std::exp(s[j] - m);
      l += p;
      for (int32_t e = 0; e < head_dim; ++e) out[i * head_dim + e] += p * v[j * head_dim + e];
    }
    for (int32_t e = 0; e < head_dim; ++e) out[i * head_dim + e] /= l;
    lse[i] = m + std::log(l);
  }
}

// Causal batched prefill over the paged NVFP4 cache ([#3575] "들어가며": causal
// attention where a query row sees a key range that grows with its position;
// GQA: kv head = q head / (H_q / H_kv)).  K and V are dequantized to doubles
// ([#4769]: dequantize the tile once, then attend) and attention is the
// textbook softmax in fp64:
//   s_j = sm_scale * <q, K_j>,  j <= i + kv_len - qo_len
//   o = sum_j exp(s_j - m) V_j / sum_j exp(s_j - m),  lse = m + ln(sum_j exp(s_j - m))
int orc_prefill(const uint16_t* q, int32_t batch, const int32_t* qo_indptr,
                const int32_t* kv_indptr, const int32_t* page_table, int32_t pt_stride,
                int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                int32_t page_size, const uint8_t* k_data, const uint8_t* v_data,
                const uint8_t* k_sf, const uint8_t* v_sf, double k_scale, double v_scale,
                double sm_scale, const int64_t* rows, int64_t n_rows, double* out,
                double* lse, int32_t threads) {
  return orc_prefill_fmt(q, batch, qo_indptr, kv_indptr, page_table, pt_stride, num_qo_heads,
                         num_kv_heads, head_dim, page_size, 0, k_data, v_data, k_sf, v_sf,
                         k_scale, v_scale, sm_scale, rows, n_rows, out, lse, threads);
}

int orc_prefill_fmt(const uint16_t* q, int32_t batch, const int32_t* qo_indptr,
                    const int32_t* kv_indptr, const int32_t* page_table, int32_t pt_stride,
                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, int32_t kv_format, const uint8_t* k_data,
                    const uint8_t* v_data, const uint8_t* k_sf, const uint8_t* v_sf,
                    double k_scale, double v_scale, double sm_scale, const int64_t* rows,
                    int64_t n_rows, double* out, double* lse, int32_t threads) {
  if (kv_format != 0 && kv_format != 1) return -1;
  if (batch < 0 || num_kv_heads <= 0 || num_qo_heads % num_kv_heads != 0) return -1;
  for (int32_t b = 0; b < batch; ++b) {
    int32_t qo_len = qo_indptr[b + 1] - qo_indptr[b];
    int32_t kv_len = kv_indptr[b + 1] - kv_indptr[b];
    if (qo_len < 0 || kv_len < 0 || qo_len > kv_len) return -1;
  }
  const int32_t group = num_qo_heads / num_kv_heads;
  const int64_t total_q = qo_indptr[batch];
  const int64_t n = rows ? n_rows : total_q * num_qo_heads;
  // Row r -> (global q token, q head).
  std::vector<int64_t> tok(n), head(n);
  for (int64_t r = 0; r < n; ++r) {
    tok[r] = rows ? rows[2 * r] : r / num_qo_heads;
    head[r] = rows ? rows[2 * r + 1] : r % num_qo_heads;
    if (tok[r] < 0 || tok[r] >= total_q || head[r] < 0 || head[r] >= num_qo_heads) return -1;
  }
  // Group rows by (sequence, kv head) so that each sequence's K/V is
  // dequantized once per group.
  std::vector<int32_t> seq(n);
  for (int64_t r = 0; r < n; ++r)
    seq[r] = static_cast<int32_t>(std::upper_bound(qo_indptr, qo_indptr + batch + 1, tok[r]) -
                                  qo_indptr) - 1;
  std::vector<int64_t> order(n);
  for (int64_t r = 0; r < n; ++r) order[r] = r;
  std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    int64_t ka = static_cast<int64_t>(seq[a]) * num_kv_heads + head[a] / group;
    int64_t kb = static_cast<int64_t>(seq[b]) * num_kv_heads + head[b] / group;
    return ka < kb;
  });
#ifdef _OPENMP
  if (threads > 0) omp_set_num_threads(threads);
#endif
  std::vector<double> kd, vd;
  int64_t start = 0;
  while (start < n) {
    int32_t b = seq[order[start]];
    int32_t hk = static_cast<int32_t>(head[order[start]] / group);
    int64_t end = start;
    while (end < n && seq[order[end]] == b && head[order[end]] / group == hk) ++end;
    const int32_t qo_len = qo_indptr[b + 1] - qo_indptr[b];
    const int32_t kv_len = kv_indptr[b + 1] - kv_indptr[b];
    kd.assign(static_cast<size_t>(kv_len) * head_dim, 0.0);
    vd.assign(static_cast<size_t>(kv_len) * head_dim, 0.0);
#pragma omp parallel for schedule(static)
    for (int32_t j = 0; j < kv_len; ++j) {
      int64_t page = page_table[static_cast<int64_t>(b) * pt_stride + j / page_size];
      int64_t slot = page * page_size + j % page_size;
      if (kv_format == 1) {
        orc_fp8_dequant_row(k_data, num_kv_heads, head_dim, page_size, slot, hk, k_scale,
                            &kd[static_cast<size_t>(j) * head_dim]);
        orc_fp8_dequant_row(v_data, num_kv_heads, head_dim, page_size, slot, hk, v_scale,
                            &vd[static_cast<size_t>(j) * head_dim]);
      } else {
        orc_dequant_row(k_data, k_sf, num_kv_heads, head_dim, page_size, slot, hk, k_scale,
                        &kd[static_cast<size_t>(j) * head_dim]);
        orc_dequant_row(v_data, v_sf, num_kv_heads, head_dim, page_size, slot, hk, v_scale,
                        &vd[static_cast<size_t>(j) * head_dim]);
      }
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t idx = start; idx < end; ++idx) {
      const int64_t r = order[idx];
      const int64_t i = tok[r] - qo_indptr[b];
      const int64_t last = i + kv_len - qo_len;
      std::vector<double> qv(head_dim), s(last + 1);
      for (int32_t e = 0; e < head_dim; ++e)
        qv[e] = bf16_to_float(q[(tok[r] * num_qo_heads + head[r]) * head_dim + e]);
      double m = -INFINITY;
      for (int64_t j = 0; j <= last; ++j) {
        double dot = 0.0;
        for (int32_t e = 0; e < head_dim; ++e) dot += qv[e] * kd[j * head_dim + e];
        s[j] = sm_scale * dot;
        m = std::max(m, s[j]);
      }
      double l = 0.0;
      double* o = out + r * head_dim;
      for (int32_t e = 0; e < head_dim; ++e) o[e] = 0.0;
      for (int64_t j = 0; j <= last; ++j) {
        double p = std::exp(s[j] - m);
        l += p;
        for (int32_t e = 0; e < head_dim; ++e) o[e] += p * vd[j * head_dim + e];
      }
      for (int32_t e = 0; e < head_dim; ++e) o[e] /= l;
      lse[r] = m + std::log(l);
    }
    start = end;
  }
  return 0;
}

int32_t orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

}  // extern "C"
