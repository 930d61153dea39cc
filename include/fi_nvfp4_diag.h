/*
 * fi_nvfp4_diag.h — diagnostic probes of libfi_nvfp4_diag.so.  They run the
 * exact device code of libfi_nvfp4.so (the same headers) on small inputs so
 * that tests can pin each building block separately:
 *   - the native NVFP4 / FP8 conversions against the CPU codec over all 2^32
 *     fp32 bit patterns,
 *   - the per-16 block quantizer (the append's arithmetic),
 *   - the tile repack (FP4 codes + E4M3 scales -> exact 16-bit staging tile),
 *   - the tcgen05 operand layouts and descriptors used by the prefill.
 * The pages have no counterpart of these probes; they exist to test the
 * library.  All pointers are device pointers; `stream` is a cudaStream_t.
 * Every call returns 0 on success, 1 on a bad argument, 4 on a CUDA error.
 */
#ifndef FI_NVFP4_DIAG_H
#define FI_NVFP4_DIAG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* For the `count` fp32 bit patterns first_bits, first_bits+1, ... (mod 2^32):
 * e4m3_out[i] = E4M3 code (cvt.rn.satfinite.e4m3x2.f32),
 * e2m1_out[i] = E2M1 code (cvt.rn.satfinite.e2m1x2.f32) in the low nibble. */
int32_t fi_diag_codec_span(uint32_t first_bits, uint64_t count, uint8_t* e4m3_out,
                           uint8_t* e2m1_out, void* stream);

/* Quantizes n_blocks blocks of 16 bf16 values (x: [n_blocks][16]) with global
 * decode scale g, exactly as the append kernel does: packed_out [n_blocks][8]
 * code bytes, s8_out [n_blocks] scale bytes. */
int32_t fi_diag_quantize_blocks(const void* x, int64_t n_blocks, float g, uint8_t* packed_out,
                                uint8_t* s8_out, void* stream);

/* Checks the append's division by the block decode scale: for all 65536 bf16
 * inputs x and each of the n_d fp32 divisors d_values[i] (device array), where
 * the quantizer takes its Markstein path (d in [2^-98, 2^100], |x| <= 2^100 d),
 * compares its quotient with the IEEE quotient x / d.  counts (device, 4 x
 * uint64, zeroed by the caller): [0] checked pairs, [1] pairs whose E2M1 codes
 * differ, [2] pairs with |x| >= 2^-100 and a normal IEEE quotient whose bits
 * differ, [3] pairs with |x| < 2^-100 whose bits differ (the code is the same
 * there by construction).  first_bad (device, 2 x uint32): x bits and divisor
 * index of a pair counted in [1] or [2].  n_d <= 65535. */
int32_t fi_diag_div_check(const float* d_values, int32_t n_d, unsigned long long* counts,
                          uint32_t* first_bad, void* stream);

/* Repacks one raw tile (raw: 128*(D/2) code bytes then 128*(D/16) scale bytes)
 * as the prefill does (is_v = 0: bf16, 1: fp16; rows >= valid become 0) and
 * writes the unswizzled 16-bit values to out [128][D] (uint16 bit patterns). */
int32_t fi_diag_repack_tile(const uint8_t* raw, int32_t head_dim, int32_t is_v, int32_t valid,
                            uint16_t* out, void* stream);

/* One 128x128x128 tcgen05 MMA product, fp32 result c [128][128]:
 *   mode 0: c = A * B^T, A bf16 [128][128] loaded by TMA (128B swizzle,
 *           K-major), B bf16 [128][128] staged K-major by threads (as K tiles);
 *   mode 1: c = A * B, A fp16 [128][128] stored into tensor memory (as P),
 *           B fp16 [128 k][128 n] staged MN-major (as V tiles), leading byte
 *           offset 16384 (between 64-column blocks) and stride byte offset
 *           1024 (between groups of 8 k rows), the prefill's choice;
 *   mode 3: as mode 1 with A fp16 staged K-major in shared memory.
 * Any other mode returns 1.
 * `status` (device int32) gets bit 16 if a wait ran out of time. */
int32_t fi_diag_umma(int32_t mode, const void* a, const void* b, float* c, int32_t* status,
                     void* stream);

/* One M=256 x N=128 x K=128 tcgen05 MMA issued for a pair of CTAs (one
 * 2-CTA cluster, cta_group::2), fp32 result c [256][128]:
 *   mode 0: c = A * B^T, A bf16 [256][128] K-major (CTA r holds rows
 *           128r..128r+127), B bf16 [128 N][128 K] K-major, N rows split
 *           64 per CTA (as the paired prefill's S = Q K^T);
 *   mode 1: c = A * B, A fp16 [256][128 K] K-major, B fp16 [128 K][128 N]
 *           MN-major, N columns split 64 per CTA (as its O = P V).
 * tmem_addrs (device, 2 x uint32): the tensor-memory base address each CTA
 * was allocated.  `status` gets bit 16 if a wait ran out of time. */
int32_t fi_diag_umma_pair(int32_t mode, const void* a, const void* b, float* c, int32_t* status,
                          uint32_t* tmem_addrs, void* stream);

/* Makes a bounded pipeline wait run out, with the library's own wait code: a
 * one-CTA kernel whose warps wait on an mbarrier that nothing arrives at.
 * Warp 0 holds tensor memory, has a 4096-byte bulk copy (copy_src -> shared
 * memory) in flight and waits with the limit `timeout_ns` (1 ns .. 1 s); the
 * other warps wait with the prefill's 2 s limit and give up through the CTA's
 * abort flag as soon as warp 0's wait has run out.  Warp 0 then waits
 * (bounded) for its copy, every thread meets, the tensor memory is freed and
 * the kernel returns.  Effects: `status` (device int32) gets FI_DEV_WAIT_TIMEOUT
 * (16) with atomicOr; copy_out (device, 4096 bytes) receives the copied bytes;
 * report (device, 4 x uint64): [0] ns warp 0 waited, [1] ns warp 1 waited,
 * [2] waits that gave up (66), [3] 1 if the copy completed.  copy_src and
 * copy_out 16-byte aligned. */
int32_t fi_diag_wait_timeout(uint64_t timeout_ns, const uint8_t* copy_src, uint8_t* copy_out,
                             int32_t* status, unsigned long long* report, void* stream);

#ifdef __cplusplus
}
#endif
#endif
