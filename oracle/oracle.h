/*
 * oracle.h — plain, slow CPU reference for the NVFP4 paged-KV append and the
 * causal prefill that reads the cache back.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this code; only the tests, the smoke check and the benchmark's CPU
 * baseline load it.  It shares no source with the CUDA path.
 *
 * Sources followed (analysis pages of merged FlashInfer PRs, cited by PR number
 * and title):
 *   [#6204] "FlashInfer: NVFP4 KV 캐시 어펜드 성능 최적화로 인한 동기화 제거"
 *           — the append API, its positive-finite global decode scale and the
 *             slot_mapping scatter (sections "코드 분석" and the k_scale/v_scale
 *             docstring).
 *   [#4769] "FlashInfer NVFP4 KV 타일 리팩(Repack)을 통한 성능 최적화"
 *           — prefill dequantizes each NVFP4 KV tile once to 16 bits ("들어가며").
 *   [#3575] "FlashInfer FP8 Causal Attention 최적화: O(1) 디코딩과 글로벌 스케줄링의 힘"
 *           — causal batched prefill with GQA heads h_kv ("들어가며", §1).
 *   OCP Microscaling Formats (MX) v1.0 — the bit formats of E2M1 and E4M3 (the
 *           pages name NVFP4 but never spell out its bits).
 *
 * The FP8 (E4M3) paged-KV variant (the pages measure FP8 attention but give
 * no FP8 cache format): one E4M3 code per element, code = e4m3(x / g) with one
 * fp32 decode scale g per tensor, pages [P][H_kv][ps][D] bytes (a reading).
 *
 * Readings where the pages are silent (all listed in the design notes):
 *   - codes and scales are rounded to nearest, ties to the even code, with
 *     saturation to the largest finite magnitude and the sign kept (-0.2 -> -0);
 *   - s8 = e4m3(amax / (6 g)), q = e2m1(x / (e4m3(s8) g)), all in fp32 with IEEE
 *     division; an all-zero block, or one whose s8 underflows to 0, stores s8 = 0
 *     and all codes 0;
 *   - cache layout HND: data [P][H_kv][ps][D/2] bytes, element 2c in the low
 *     nibble of byte c; scales [P][H_kv][ps][D/16] bytes;
 *   - slot = page * ps + offset, negative slots are skipped;
 *   - key j is visible to query row i iff j <= i + kv_len - qo_len;
 *   - lse is the natural-log log-sum-exp of the scaled logits.
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status bits, same meaning as the library's device status word. */
#define ORC_BAD_K_SCALE 1
#define ORC_BAD_V_SCALE 2
#define ORC_SLOT_OOB 4

/* --- element codecs (OCP MX v1.0) ------------------------------------- */
double orc_e2m1_value(uint8_t code);            /* code & 15 */
double orc_e4m3_value(uint8_t code);            /* NaN for 0x7F / 0xFF */
uint8_t orc_e2m1_encode(float y);               /* brute-force nearest */
uint8_t orc_e4m3_encode(float t);               /* brute-force nearest */
uint8_t orc_e2m1_encode_bits(float y);          /* bit-level RNE, same rule */
uint8_t orc_e4m3_encode_bits(float t);          /* bit-level RNE, same rule */
/* Bit-level encoders over `count` consecutive fp32 bit patterns starting at
 * `first_bits` (wrapping at 2^32).  Used by the exhaustive hardware check. */
void orc_e2m1_encode_span(uint32_t first_bits, uint64_t count, uint8_t* out);
void orc_e4m3_encode_span(uint32_t first_bits, uint64_t count, uint8_t* out);
/* Array forms: mode 0 = brute-force nearest, mode 1 = bit-level. */
void orc_e2m1_encode_array(const float* in, int64_t n, int32_t mode, uint8_t* out);
void orc_e4m3_encode_array(const float* in, int64_t n, int32_t mode, uint8_t* out);

/* --- quantize one 16-element block ----------------------------------- */
/* x: 16 bf16 bit patterns; g: global decode scale.  Writes 8 packed bytes
 * and the E4M3 scale byte. */
void orc_quantize_block16(const uint16_t* x, float g, uint8_t* packed, uint8_t* s8);

/* --- append with slot_mapping ---------------------------------------- */
/* k, v: bf16 bit patterns, token i / head h / element d at
 * [i*tok_stride + h*D + d].  Returns ORC_* status bits.  If either scale is
 * not a positive finite number nothing is written.  Slots >= P*ps are skipped
 * and flagged.  Bytes that are not written keep their value. */
int orc_append(const uint16_t* k, const uint16_t* v, int64_t num_tokens,
               int64_t k_tok_stride, int64_t v_tok_stride, int32_t num_kv_heads,
               int32_t head_dim, float k_scale, float v_scale,
               const int64_t* slot_mapping, uint8_t* k_data, uint8_t* v_data,
               uint8_t* k_sf, uint8_t* v_sf, int32_t num_pages, int32_t page_size);

/* Dequantize the cache row for (slot, head) to doubles: e2m1 * e4m3 * g. */
void orc_dequant_row(const uint8_t* data, const uint8_t* sf, int32_t num_kv_heads,
                     int32_t head_dim, int32_t page_size, int64_t slot, int32_t head,
                     double g, double* out);

/* --- FP8 (E4M3) paged KV variant ------------------------------------- */
/* One E4M3 code per head-dim element, HND pages [P][H_kv][ps][D] bytes, and
 * one positive finite fp32 decode scale g per tensor (k_scale / v_scale):
 *   code = e4m3(x / g)   (fp32 IEEE division, then nearest even, saturating
 *                         to +-448, sign kept; NaN gives the NaN code)
 *   value = e4m3(code) * g. */
uint8_t orc_fp8_quantize(float x, float g);
int orc_fp8_append(const uint16_t* k, const uint16_t* v, int64_t num_tokens,
                   int64_t k_tok_stride, int64_t v_tok_stride, int32_t num_kv_heads,
                   int32_t head_dim, float k_scale, float v_scale,
                   const int64_t* slot_mapping, uint8_t* k_data, uint8_t* v_data,
                   int32_t num_pages, int32_t page_size);
void orc_fp8_dequant_row(const uint8_t* data, int32_t num_kv_heads, int32_t head_dim,
                         int32_t page_size, int64_t slot, int32_t head, double g, double* out);

/* --- causal batched prefill over the paged cache (fp64) --------------- */
/* q: bf16 bits [total_q][H_q][D].  page_table: [B][pt_stride] int32.
 * rows == NULL: every (token, q head) row; else n_rows pairs
 * (global q token, q head) given as rows[2r], rows[2r+1].
 * out: [n][D] doubles (n = total_q*H_q or n_rows), lse: [n].
 * threads <= 0 means all available.  Returns 0, or -1 on invalid
 * arguments (qo_len > kv_len, head counts not divisible, bad row). */
int orc_prefill(const uint16_t* q, int32_t batch, const int32_t* qo_indptr,
                const int32_t* kv_indptr, const int32_t* page_table, int32_t pt_stride,
                int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                int32_t page_size, const uint8_t* k_data, const uint8_t* v_data,
                const uint8_t* k_sf, const uint8_t* v_sf, double k_scale, double v_scale,
                double sm_scale, const int64_t* rows, int64_t n_rows, double* out,
                double* lse, int32_t threads);

/* The same over either cache format: kv_format 0 = NVFP4 (k_sf, v_sf used),
 * 1 = FP8 (k_sf, v_sf ignored). */
int orc_prefill_fmt(const uint16_t* q, int32_t batch, const int32_t* qo_indptr,
                    const int32_t* kv_indptr, const int32_t* page_table, int32_t pt_stride,
                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, int32_t kv_format, const uint8_t* k_data,
                    const uint8_t* v_data, const uint8_t* k_sf, const uint8_t* v_sf,
                    double k_scale, double v_scale, double sm_scale, const int64_t* rows,
                    int64_t n_rows, double* out, double* lse, int32_t threads);

/* Dense causal attention on already-dequantized K/V (no pages), one head:
 * q [L_q][D] (double), k/v [L_kv][D] (double).  Used to pin the paged path. */
void orc_dense_causal(const double* q, const double* k, const double* v, int32_t L_q,
                      int32_t L_kv, int32_t head_dim, double sm_scale, double* out,
                      double* lse);

int32_t orc_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
