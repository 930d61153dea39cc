/*
 * fi_nvfp4.h — C ABI of libfi_nvfp4.so: quantize-append bf16 K/V into an NVFP4
 * paged KV cache through a slot_mapping, plan a causal batched prefill over that
 * cache, and run it.  Built for NVIDIA B300 (sm_103a) only.
 *
 * Sources (analysis pages of merged FlashInfer PRs, cited by PR number and title):
 *   [#6204] "FlashInfer: NVFP4 KV 캐시 어펜드 성능 최적화로 인한 동기화 제거"
 *   [#4769] "FlashInfer NVFP4 KV 타일 리팩(Repack)을 통한 성능 최적화"
 *   [#3575] "FlashInfer FP8 Causal Attention 최적화: O(1) 디코딩과 글로벌 스케줄링의 힘"
 *   [#5043] "FlashInfer의 plan() 함수 최적화: Python max()에서 Tensor.max()로의 전환"
 *
 * Conventions of every call below
 *   - Pointers named *_dev are device pointers on the current CUDA device;
 *     *_host are host pointers.  `stream` is a cudaStream_t (NULL = legacy
 *     default stream).  The library never frees caller memory.
 *   - Every argument error is detected on the host and returned as a status;
 *     such a call enqueues nothing.
 *   - Errors that only the device can see (a bad device scale, a slot or page
 *     id out of range, a pipeline wait that ran out of time) set bits of the
 *     context's device status word with atomicOr.  Kernels never trap.  The
 *     word is read (and optionally cleared) only by fi_device_status().
 *   - No call synchronizes the host with the device except fi_device_status()
 *     and fi_context_destroy(); fi_nvfp4_append and fi_prefill_run read no
 *     device memory on the host and may be captured in a CUDA graph.
 *
 * NVFP4 cache format (readings of the pages, which name the format but not
 * its bits or layout):
 *   value = e2m1(code) * e4m3(s8) * g, one E4M3 scale s8 per 16 consecutive
 *   head-dim elements, one positive finite fp32 global decode scale g per tensor
 *   ([#6204] k_scale/v_scale docstring).  Bit formats: OCP MX v1.0 E2M1 and
 *   E4M3 ("FN": no inf, max 448).  Layout, per tensor (K and V alike), HND:
 *     data  uint8 [num_pages][num_kv_heads][page_size][head_dim/2]
 *           byte c of a row holds element 2c in its low nibble, 2c+1 in its high
 *     scale uint8 [num_pages][num_kv_heads][page_size][head_dim/16]
 *   Token slot s lives in page s / page_size at offset s % page_size.
 *   Quantization (round to nearest, ties to the even code, saturating, sign
 *   kept): s8 = e4m3(amax / (6 g)); code_j = e2m1(x_j / (e4m3(s8) g)); a block
 *   whose amax is 0, or whose s8 rounds to 0, stores s8 = 0 and codes 0.  All
 *   steps are single fp32 IEEE operations, so the bytes are deterministic.
 */
#ifndef FI_NVFP4_H
#define FI_NVFP4_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t fi_status;

/* Host-side return codes. */
#define FI_OK 0
#define FI_ERR_INVALID_ARGUMENT 1 /* null pointer, bad size, misaligned, ... */
#define FI_ERR_BAD_SCALE 2        /* host scale not positive and finite     */
#define FI_ERR_UNSUPPORTED 3      /* head_dim / page_size / device not supported */
#define FI_ERR_CUDA 4             /* a CUDA runtime call failed             */
#define FI_ERR_OUT_OF_MEMORY 5    /* plan or context allocation failed      */
#define FI_ERR_SCRATCH_TOO_SMALL 6 /* batch too large for fi_prefill_noalloc's fixed scratch */

/* Bits of the device status word (fi_device_status). */
#define FI_DEV_BAD_K_SCALE 1   /* device k_scale not positive finite: nothing written */
#define FI_DEV_BAD_V_SCALE 2   /* device v_scale not positive finite: nothing written */
#define FI_DEV_SLOT_OOB 4      /* slot_mapping entry >= num_pages*page_size: token skipped */
#define FI_DEV_PAGE_OOB 8      /* page_table entry outside [0, num_pages): page read as zeros */
#define FI_DEV_WAIT_TIMEOUT 16 /* a pipeline wait ran out of time; the kernel returned early */

typedef struct fi_context fi_context;
typedef struct fi_plan fi_plan;

/* The paged NVFP4 cache, described by caller-owned device memory.  All four
 * arrays must be 16-byte aligned.  k_scale / v_scale are device fp32 scalars
 * holding the global decode scales the prefill dequantizes with. */
typedef struct {
  uint8_t* k_data;
  uint8_t* v_data;
  uint8_t* k_sf;
  uint8_t* v_sf;
  const float* k_scale;
  const float* v_scale;
  int32_t num_pages;
  int32_t page_size;    /* 16, 32, 64 or 128 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* 64 or 128 */
} fi_nvfp4_cache;

/* Creates a context on the current device: it owns the device status word
 * (cleared at creation).  Returns FI_ERR_UNSUPPORTED if the current device is
 * not compute capability 10.3. */
fi_status fi_context_create(fi_context** out);
/* Synchronizes the device, then frees the context. */
fi_status fi_context_destroy(fi_context* ctx);

/* Quantize-append with device scales ([#6204], nvfp4_quantize_append_paged_
 * kv_cache_with_slot_mapping and its k_scale/v_scale docstring).
 *   k_dev, v_dev: bf16, token i / head h / element d at
 *       [i*tok_stride + h*head_dim + d]; 16-byte aligned, tok_stride a
 *       multiple of 8 elements.
 *   slot_mapping_dev: int64 [num_tokens]; a negative slot skips the token.
 *   k_scale_dev, v_scale_dev: device fp32 scalars (the global decode scales).
 *       They are checked by the kernel, never read on the host: if either is
 *       not positive and finite the kernel writes nothing and sets
 *       FI_DEV_BAD_K_SCALE / FI_DEV_BAD_V_SCALE.
 *   num_tokens == 0 launches nothing and checks nothing (as on the page, a
 *   scale is only checked when there are rows to write).
 * Duplicate non-negative slots within one call are undefined. */
fi_status fi_nvfp4_append(fi_context* ctx, const void* k_dev, const void* v_dev,
                          int64_t num_tokens, int64_t k_tok_stride, int64_t v_tok_stride,
                          const float* k_scale_dev, const float* v_scale_dev,
                          const int64_t* slot_mapping_dev, const fi_nvfp4_cache* cache,
                          void* stream);

/* Same append with host scales: they are checked on the host and a scale that
 * is not positive and finite returns FI_ERR_BAD_SCALE without enqueueing
 * anything ([#6204]: "A float or CPU tensor is checked on the host and raises
 * ValueError"). */
fi_status fi_nvfp4_append_host_scale(fi_context* ctx, const void* k_dev, const void* v_dev,
                                     int64_t num_tokens, int64_t k_tok_stride,
                                     int64_t v_tok_stride, float k_scale, float v_scale,
                                     const int64_t* slot_mapping_dev,
                                     const fi_nvfp4_cache* cache, void* stream);

/* Plan options (all zero = defaults). */
typedef struct {
  int32_t schedule; /* 0: default (uniform batches: global reverse-Q-tile order;
                       ragged batches: decided by the L2 gate, global order iff
                       2 * KV bytes <= L2); 1: global reverse-Q-tile order;
                       2: per-(sequence, head) reverse order */
  int32_t num_ctas; /* persistent CTAs; 0 = number of SMs */
  int64_t l2_bytes; /* L2 size for the gate; 0 = the device's */
  int32_t cta_pairs; /* 0: GQA groups of a multiple of 4 query heads run on 2-CTA
                        clusters that share their KV staging tiles; 1: never */
  int32_t kv_format; /* cache the runs read: 0 NVFP4 (fi_prefill_run), 1 FP8
                        (fi_prefill_run_fp8); sets the KV bytes of the L2 gate */
} fi_plan_options;

/* What the planner decided (host values). */
typedef struct {
  int32_t batch;
  int32_t max_qo_len;
  int32_t max_kv_len;
  int64_t total_qo_len;
  int64_t total_kv_len;
  int32_t is_uniform;     /* every qo_len equal and every kv_len equal */
  int32_t global_reverse; /* heaviest q-tiles of all sequences and heads first */
  int32_t q_tiles;        /* ceil(max_qo_len / 128) */
  int32_t heads_per_cta;  /* q heads per CTA sharing each staged KV tile */
  int32_t head_units;     /* num_kv_heads * group / (heads_per_cta * ctas_per_unit) */
  int64_t num_units;      /* work units (sequence, head unit, q-tile) */
  int64_t kv_bytes;       /* NVFP4 bytes of K and V the batch reads */
  int32_t num_ctas;       /* CTAs the run launches (at most; pairs may be fewer) */
  int32_t ctas_per_unit;  /* 2 when units run on CTA pairs, else 1 */
  int32_t balanced;       /* 1: fewer than 16 units per CTA (pair); each unit,
                             heaviest first, is assigned to the least-loaded one
                             (longest-processing-time first); 0: round-robin */
  int32_t max_slot_tiles; /* balanced plans: KV tiles (plus one per unit) of the
                             most loaded CTA (pair); 0 otherwise */
} fi_plan_info;

/* Creates an empty, reusable plan bound to `ctx`. */
fi_status fi_plan_create(fi_context* ctx, fi_plan** out);
/* Synchronizes the device, then frees the plan's device and pinned memory. */
fi_status fi_plan_destroy(fi_plan* plan);

/* Plans a causal batched prefill ([#5043]: one reduction gives max_qo_len and
 * max_kv_len; [#3575] §1-§3: the uniform-length flag for O(1) tile decoding,
 * global reverse-Q-tile scheduling and the L2 gate).
 *   qo_indptr_host, kv_indptr_host: int32 [batch+1], non-decreasing, from 0;
 *       sequence b has qo_len = qo_indptr[b+1]-qo_indptr[b] query rows and
 *       kv_len likewise (kv_len >= qo_len; query row i sees keys
 *       j <= i + kv_len - qo_len).
 *   page_table_dev: int32 [batch][page_table_stride]; key j of sequence b is
 *       in page page_table[b][j / page_size].  Only the pointer is kept: it
 *       must stay valid until every run of this plan has finished.
 *   sm_scale: logit scale; <= 0 selects 1/sqrt(head_dim).
 * The plan reads host memory only.  It copies its work description to plan-
 * owned device memory with cudaMemcpyAsync on `stream` from pinned staging;
 * the staging is double-buffered and a buffer is reused only after the copy
 * issued from it two plans earlier has finished, so steady-state planning does
 * not wait on the device.  Runs of this plan must be enqueued on `stream`
 * (or ordered after it). */
fi_status fi_prefill_plan(fi_plan* plan, const int32_t* qo_indptr_host,
                          const int32_t* kv_indptr_host, int32_t batch,
                          const int32_t* page_table_dev, int32_t page_table_stride,
                          int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t page_size, float sm_scale, const fi_plan_options* opts,
                          void* stream);

fi_status fi_plan_get_info(const fi_plan* plan, fi_plan_info* info);

/* Runs the planned prefill ([#4769]: each NVFP4 KV tile is dequantized once
 * into a 16-bit staging tile outside the MMA loop; [#3575]: causal, GQA).
 *   q_dev: bf16 [total_qo][num_qo_heads][head_dim], 16-byte aligned.
 *   cache: the NVFP4 cache (its k_scale/v_scale device scalars are used).
 *   out_dev: bf16 [total_qo][num_qo_heads][head_dim] (written for every row).
 *   lse_dev: fp32 [total_qo][num_qo_heads] natural-log log-sum-exp of the
 *       scaled logits, or NULL.
 * Head counts, head_dim and page_size must match the plan. */
fi_status fi_prefill_run(const fi_plan* plan, const void* q_dev, const fi_nvfp4_cache* cache,
                         void* out_dev, float* lse_dev, void* stream);

/* ---- decode ----------------------------------------------------------------
 * Plans attention for the newest query tokens of each sequence (decode and
 * short speculative steps) over the NVFP4 cache ([#5043] decode.py: max_kv_len
 * comes from one reduction over the lengths).  Same arguments and causal rule
 * as fi_prefill_plan; every sequence has qo_len <= 8 and
 * (num_qo_heads / num_kv_heads) * qo_len <= 32, else FI_ERR_UNSUPPORTED.  The
 * keys of all (sequence, KV head) pairs are split evenly over the warps the
 * decode kernel keeps resident (fi_decode_plan_host gives the rule); a pair
 * split across warps is merged by a second kernel.  The plan owns a device
 * buffer for the pieces' partial results, grown (after synchronizing
 * `stream`) when a plan needs more; otherwise it behaves as fi_prefill_plan.
 * fi_plan_get_info reports the pieces in num_units. */
fi_status fi_decode_plan(fi_plan* plan, const int32_t* qo_indptr_host,
                         const int32_t* kv_indptr_host, int32_t batch,
                         const int32_t* page_table_dev, int32_t page_table_stride,
                         int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t page_size, float sm_scale, void* stream);

/* Runs a decode plan: arguments, layouts and output as fi_prefill_run.  A
 * prefill plan passed here, or a decode plan passed to fi_prefill_run,
 * returns FI_ERR_INVALID_ARGUMENT. */
fi_status fi_decode_run(const fi_plan* plan, const void* q_dev, const fi_nvfp4_cache* cache,
                        void* out_dev, float* lse_dev, void* stream);

/* ---- FP8 (E4M3) paged KV variant --------------------------------------
 * The same paged layout with one E4M3 code per element and no block scales
 * (a reading: the pages measure FP8 attention ([#3575]) but give no FP8
 * cache format):
 *   data uint8 [num_pages][num_kv_heads][page_size][head_dim], per tensor;
 *   value = e4m3(code) * g, code = e4m3(x / g) (one fp32 IEEE division, then
 *   nearest even, saturating to +-448, sign kept), g the tensor's positive
 *   finite fp32 decode scale.  Both arrays 16-byte aligned. */
typedef struct {
  uint8_t* k_data;
  uint8_t* v_data;
  const float* k_scale;
  const float* v_scale;
  int32_t num_pages;
  int32_t page_size;    /* 16, 32, 64 or 128 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* 64 or 128 */
} fi_fp8_cache;

/* Quantize-append into the FP8 cache; arguments, scale checks, status bits
 * and error behaviour as fi_nvfp4_append. */
fi_status fi_fp8_append(fi_context* ctx, const void* k_dev, const void* v_dev,
                        int64_t num_tokens, int64_t k_tok_stride, int64_t v_tok_stride,
                        const float* k_scale_dev, const float* v_scale_dev,
                        const int64_t* slot_mapping_dev, const fi_fp8_cache* cache,
                        void* stream);

/* Runs a plan made with kv_format = 1 over the FP8 cache: each KV tile is
 * converted once into the same 16-bit staging tiles; everything else as
 * fi_prefill_run.  A plan made for the other format returns
 * FI_ERR_INVALID_ARGUMENT. */
fi_status fi_prefill_run_fp8(const fi_plan* plan, const void* q_dev, const fi_fp8_cache* cache,
                             void* out_dev, float* lse_dev, void* stream);

/* Host-only planning, for inspection and tests: fills `info` and, if
 * `work_out` is non-NULL, up to `work_capacity` work units as 4 int32 each
 * (sequence, head unit, q-tile, KV tiles the unit reads) in the order the
 * kernel numbers them.  (The device plan of a ragged batch holds one entry
 * per (sequence, q-tile), whose head units are consecutive units; uniform
 * batches are decoded arithmetically and need no list.)  Makes no CUDA call.
 * `l2_bytes` is the L2 size for the gate. */
fi_status fi_prefill_plan_host(const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                               int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t page_size, int64_t l2_bytes,
                               const fi_plan_options* opts, fi_plan_info* info,
                               int32_t* work_out, int64_t work_capacity);

/* Host-only decode planning, for inspection and tests (the decision
 * fi_decode_plan makes for the same arguments on a GPU with `num_sms` SMs).
 * The keys of every (sequence, KV head) pair with queries are taken in steps
 * of 32, laid end to end in (sequence, head) order and cut into W runs of
 * equal length (to one step), one per warp of the decode kernel: W is the
 * number of warps the kernel keeps resident on num_sms SMs (16 per SM up to 8
 * rows G * max qo_len, 12 up to 16, 8 above), or fewer so that a warp takes at
 * least 8 steps.  A run becomes one piece per pair it touches; a pair cut into
 * several pieces writes one partial result per piece and is merged.
 *   Fills `info` (num_units = pieces, num_ctas = ceil(W / 4)), *num_warps_out
 * = W and *num_merges_out, and, when the pointers are non-NULL: up to
 * `unit_capacity` pieces as 4 int32 each (sequence * num_kv_heads + KV head,
 * first key, end key (exclusive), partial slot or -1 for a pair in one piece)
 * in (sequence, head, key) order; up to `merge_capacity` merge items as 4
 * int32 each (sequence, KV head, first partial slot, pieces); up to
 * `warp_off_capacity` of the W + 1 offsets, warp w running pieces
 * warp_off[w] .. warp_off[w + 1] - 1.  Makes no CUDA call.  Errors as
 * fi_decode_plan. */
fi_status fi_decode_plan_host(const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                              int32_t batch, int32_t num_qo_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t page_size, int32_t num_sms,
                              fi_plan_info* info, int32_t* num_warps_out, int64_t* num_merges_out,
                              int32_t* units_out, int64_t unit_capacity, int32_t* merges_out,
                              int64_t merge_capacity, int32_t* warp_off_out,
                              int64_t warp_off_capacity);

/* Plans and runs the causal prefill in one call without allocating memory
 * (no cudaMalloc, no host heap), for callers that cannot allocate while they
 * run — a serving engine that reserves all device memory for its KV cache up
 * front, or a plugin whose enqueue callback must not allocate.  The pages have
 * no counterpart of this entry point.
 *   Arguments as in fi_prefill_plan and fi_prefill_run (no context, no plan).
 *   status_dev: caller-owned device int32 that receives FI_DEV_* bits with
 *       atomicOr (not cleared by the call), or NULL to discard them.
 * Scratch: the indptr copies and, for ragged batches, the work-unit list are
 * kept in one fixed device array of 2 MiB (524288 int32 words) inside the
 * library, held by every GPU that loads it until the process exits.  A call
 * needs 4 + 2 (batch + 1) words, plus 4 per (sequence, q-tile) for ragged
 * batches (sum over sequences of ceil(qo_len / 128) entries, each standing for
 * all head units of its q-tile); larger calls return FI_ERR_SCRATCH_TOO_SMALL
 * and enqueue nothing.  Every
 * call shares the array: calls that overlap on the GPU (on different streams)
 * race; calls on one stream are ordered by the stream (each call's copies into
 * the array run after the previous call's kernel).  The indptr arrays are
 * copied with cudaMemcpyAsync: from pageable memory they have been read when
 * the call returns; page-locked ones are read when the stream reaches the
 * copy, so they must stay unchanged until then.  The first call on a device
 * looks up the array's device address; make that first call before any stream
 * capture.  Ragged work units are taken in sequence order with the heaviest
 * q-tile of each sequence first, the head units of a q-tile together (dealt
 * round-robin to the CTAs: no balanced
 * slot lists); groups of a multiple of 4 query heads run on CTA pairs, as
 * fi_prefill_plan chooses by default. */
fi_status fi_prefill_noalloc(const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                             int32_t batch, const int32_t* page_table_dev,
                             int32_t page_table_stride, int32_t num_qo_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                             float sm_scale, const void* q_dev, const fi_nvfp4_cache* cache,
                             void* out_dev, float* lse_dev, int32_t* status_dev, void* stream);

/* Reads the context's device status word after synchronizing `stream`; if
 * `reset` is non-zero the word is cleared afterwards.  The only call that
 * waits for the device. */
fi_status fi_device_status(fi_context* ctx, void* stream, int32_t* bits, int32_t reset);

const char* fi_status_string(fi_status status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int32_t fi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FI_NVFP4_H */
