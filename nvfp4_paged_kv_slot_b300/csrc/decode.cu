// decode.cu — attention of the few newest query tokens of each sequence
// (decode steps and short speculative steps, qo_len <= 8) over the NVFP4
// paged cache.  The planner side follows FlashInfer PR #5043 ("FlashInfer의
// plan() 함수 최적화: Python max()에서 Tensor.max()로의 전환", decode.py:
// max_kv_len from one reduction over the lengths); the attention is the same
// causal GQA attention as the prefill's (query row t of a sequence sees keys
// j <= t + kv_len - qo_len).
//
// Decode rows are few (G * qo_len per KV head) and every key is read once, so
// the work is HBM-bound and runs on warp-level m16n8k16 MMAs (fp16 in, fp32
// accumulators) fed straight from the raw NVFP4 rows, with the rows on the
// MMA's n side (below).  The keys of all (sequence, KV head) pairs are split
// evenly over the resident warps in steps of 32; a warp runs its pieces one
// after another, copying each step's raw K and V rows (codes and block
// scales) into a two-stage ring in shared memory one step ahead (cp.async),
// converting its MMA fragments from the raw codes (E2M1 x E4M3 is exact in
// fp16) and running the online softmax on the accumulator fragments.  A pair
// split over several warps writes unnormalized partials (O, row max, row
// sum) per piece, which a second kernel merges.

#include <algorithm>
#include <atomic>

#include "internal.h"
#include "nvfp4.cuh"

namespace fi {

namespace {

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
  const int4* units;   // pieces (sequence * H_kv + kv head, first key, end key, slot or -1)
  const int4* merges;  // (sequence, kv head, first partial slot, chunks)
  float* part;         // partial slots: [slot][rows][D + 2] = O, then m, l
  const int32_t* warp_off;  // warp w runs pieces warp_off[w] .. warp_off[w + 1] - 1
  int32_t num_warps, num_merges, num_qo_heads, num_kv_heads, group, page_size, num_pages;
  int32_t rows;      // partial rows per slot (G * max qo_len)
  int32_t ps_shift;  // log2 of page_size (a power of two)
  float sm_scale;
  int32_t* status;
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// m16n8k16 MMA with fp16 inputs and fp32 accumulators (the warp-level tensor
// core path: decode is HBM-bound, so its rate is ample).
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// ---- the decode kernel: rows on the MMA's n side ------------------------
// With few rows the row dimension is better placed on the MMA's n side (8
// rows per n-tile) than on its 16-row m side: S^T = K Q^T takes keys as m,
// O^T = V^T P^T takes head dimensions as m.  With up to 8 rows that halves
// the MMAs and the accumulators of the row-major form (S = Q K^T, O += P V),
// and both K and V fragments come straight from the raw codes, so no
// dequantized copy of V is staged.
//
// The contraction index of each MMA may be permuted freely as long as both
// operands agree, and the m index of O^T may be permuted as long as the
// epilogue undoes it; both are chosen so that every lane converts contiguous
// code bytes:
//  * S^T, k-step s, lane (g = lane/4, t = lane%4): the A fragment's column
//    pairs are code bytes t*D/8 + 2s (k = 2t, 2t+1) and t*D/8 + 2s + 1 (k =
//    2t+8, 2t+9) of keys g and g+8 of the m-tile; Q's B fragment takes the
//    same head dimensions, d = t*D/4 + 4s .. t*D/4 + 4s + 3, of row g.
//  * O^T, m-tile i: row g of the tile is head dimension 2(g*D/16 + i), row
//    g+8 the one after it, so a lane converts code bytes g*D/16 .. g*D/16 +
//    D/16 - 1 of each key it touches; a pair of keys is merged nibble-wise
//    into E2M1 pairs that hold one dimension of both keys.
//  * The keys of the PV k-step are the S^T m-tile's rows in order; P^T's B
//    fragment is the S^T accumulator packed to fp16 and transposed 8x8 by
//    movmatrix.
// Raw stage of one warp (32 keys, row r = key kb + r): K codes (D/2
// bytes a key: a quarter-warp reads 128 contiguous bytes), K scales (D/16
// bytes a key), V codes and scales (D/2 and D/16 bytes a key).  V rows
// padded to 80 or 48 bytes put the 8- or 4-byte reads of a half-warp or warp
// on distinct banks; unpadded (two-way conflicts) they leave room for a
// third stage, which pays with 2 n-tiles (12 warps per SM) only.
constexpr int kDecMaxDevices = 64;  // per-device launch attributes cached
constexpr int kTWarps = 4;          // warps per CTA

// The planner sizes the warp count to what is resident per SM: 4 CTAs up to
// 8 rows, 3 up to 16, 2 up to 32 (the launch bounds below).
static_assert(kTWarps * 4 == decode_warps_per_sm(8) && kTWarps * 3 == decode_warps_per_sm(16) &&
                  kTWarps * 2 == decode_warps_per_sm(32),
              "decode occupancy and plan disagree");

// Raw stages per warp and their layout by n-tiles: with 2 n-tiles (3 CTAs
// per SM) three stages in unpadded rows, V scales in their own rows; else
// two stages with V rows (codes, then scales) padded to 80 or 48 bytes.
template <int NT>
constexpr int kTStagesOf = NT == 2 ? 3 : 2;
template <int D, int NT>
constexpr bool kTSepSf = NT == 2;
template <int D, int NT>
constexpr int kTVRowOf = kTSepSf<D, NT> ? D / 2 : (D == 128 ? 80 : 48);
template <int D, int NT>
constexpr int kTStageOf = 32 * (D / 2 + D / 16 + kTVRowOf<D, NT> + (kTSepSf<D, NT> ? D / 16 : 0));
template <int D, int NT>
constexpr int decode_t_smem_bytes() {
  return kTWarps * (kTStagesOf<NT> * kTStageOf<D, NT> + (NT >= 2 ? NT * (D / 16) * 32 * 8 : 0));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// NT: 8-row n-tiles (rows G * qo_len <= 8 NT); one warp runs its pieces in turn.
template <int D, int NT>
__global__ void __launch_bounds__(32 * kTWarps, NT == 1 ? 4 : NT == 2 ? 3 : 2)
    nvfp4_decode_t_kernel(const DecodeParams p) {
  constexpr int kTStages = kTStagesOf<NT>;
  constexpr int kStage = kTStageOf<D, NT>;
  constexpr int kVR = kTVRowOf<D, NT>;
  constexpr int kKsf = 32 * (D / 2);         // K scales within a stage
  constexpr int kV = 32 * (D / 2 + D / 16);  // V rows within a stage
  // V scale byte of block b of row r: kVsf + r * kVsfS + b
  constexpr int kVsf = kTSepSf<D, NT> ? kV + 32 * kVR : kV + D / 2;
  constexpr int kVsfS = kTSepSf<D, NT> ? D / 16 : kVR;
  constexpr int kKW = D / 32;                // code words of a key a lane converts for S^T
  constexpr int kVW = D / 64;                // code words of a key a lane converts for O^T
  constexpr bool kQs = NT >= 2;              // Q^T fragments in shared memory
  extern __shared__ __align__(16) uint8_t dsm[];
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int g = lane / 4, t = lane % 4;
  const int wid = blockIdx.x * kTWarps + warp;
  // The plan's memory (the warp's pieces) is written by no kernel (its copy
  // completed before the previous grid started): read it while the previous
  // grid finishes.  Q and the cache may come from the previous grid: after
  // the wait.
  int u_begin = 0, u_end = 0;
  int4 w_first = make_int4(0, 0, 0, 0);
  if (wid < p.num_warps) {
    u_begin = __ldg(p.warp_off + wid);
    u_end = __ldg(p.warp_off + wid + 1);
    if (u_begin < u_end) w_first = __ldg(p.units + u_begin);
  }
  grid_dep_wait();
  grid_dep_launch();
  if (wid >= p.num_warps) return;  // no block-wide barrier below
  for (int u = u_begin; u < u_end; ++u) {
    __syncwarp();  // every lane is done with the previous piece's ring
    const int4 w = u == u_begin ? w_first : __ldg(p.units + u);
    const int b = w.x / p.num_kv_heads, hk = w.x - b * p.num_kv_heads, slot = w.w;
    const int qo_start = __ldg(p.qo_indptr + b);
    const int qo_len = __ldg(p.qo_indptr + b + 1) - qo_start;
    const int kv_len = __ldg(p.kv_indptr + b + 1) - __ldg(p.kv_indptr + b);
    const int G = p.group;
    const int R = G * qo_len;  // <= 8 NT (the dispatch guarantees it)
    const int delta = kv_len - qo_len;
    const int k0 = w.y;  // the piece's keys: k0 .. k1 - 1
    const int k1 = w.z;
    const float ks = __ldg(p.k_scale), vs = __ldg(p.v_scale);
    uint8_t* ring = dsm + warp * kTStages * kStage;
    uint2* qsm = reinterpret_cast<uint2*>(dsm + kTWarps * kTStages * kStage) +
                 warp * (kQs ? NT * (D / 16) * 32 : 0);
    const int32_t* pt = p.page_table + static_cast<int64_t>(b) * p.pt_stride;
    auto q_ptr = [&](int r) {  // row r = token r / G, head hk * G + r % G
      return p.q + (static_cast<int64_t>(qo_start + r / G) * p.num_qo_heads + hk * G + r % G) * D;
    };

    // Q^T as fp16 B fragments: Q * sm_scale * k_scale * log2 e * 2^-e with e
    // chosen so that every |value| < 2^14 (a power of two: exact); the logits
    // are multiplied back by 2^e.
    const float qs = p.sm_scale * ks * 1.4426950408889634f;
    float qmax = 0.0f;
    for (int i = lane; i < R * (D / 8); i += 32) {
      float x[8];
      bf16x8_to_f32(
          __ldg(reinterpret_cast<const uint4*>(q_ptr(i / (D / 8)) + (i % (D / 8)) * 8)), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) qmax = fmaxf(qmax, fabsf(x[e]));
    }
    qmax = warp_max(qmax) * qs;
    const int qe = qmax > 0.0f ? ilogbf(qmax) - 13 : 0;
    const float qsc = ldexpf(qs, -qe);
    const float ssc = ldexpf(1.0f, qe);
    // With 2 or 4 n-tiles the fragments live in shared memory (this warp's slice,
    // fragment (nt, k-step s) of lane l at [nt][s][l]: conflict-free 8-byte
    // reads), which keeps the kernel within its registers; else in registers.
    uint32_t qb[NT][D / 16][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = 8 * nt + g;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = 0.0f;
        if (r < R)
          bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(q_ptr(r) + t * (D / 4)) + i), x);
        const uint2 f0 =
            make_uint2(f16x2_of(x[0] * qsc, x[1] * qsc), f16x2_of(x[2] * qsc, x[3] * qsc));
        const uint2 f1 =
            make_uint2(f16x2_of(x[4] * qsc, x[5] * qsc), f16x2_of(x[6] * qsc, x[7] * qsc));
        if constexpr (kQs) {
          qsm[(nt * (D / 16) + 2 * i) * 32 + lane] = f0;
          qsm[(nt * (D / 16) + 2 * i + 1) * 32 + lane] = f1;
        } else {
          qb[nt][2 * i][0] = f0.x;
          qb[nt][2 * i][1] = f0.y;
          qb[nt][2 * i + 1][0] = f1.x;
          qb[nt][2 * i + 1][1] = f1.y;
        }
      }
    }
    if constexpr (kQs) __syncwarp();  // every lane's fragments are stored
    auto qfrag = [&](int nt, int ks) {
      if constexpr (kQs)
        return qsm[(nt * (D / 16) + ks) * 32 + lane];
      else
        return make_uint2(qb[nt][ks][0], qb[nt][ks][1]);
    };

    // O^T accumulators (m-tile i, n-tile nt), and per lane the running max and
    // sum of rows 8 nt + 2t + e.  The max is raised lazily: only when a step's
    // max exceeds it by more than 8 (in log2 units), so exponentials stay at
    // most 2^8 and the rescale of O is rare.
    float o[D / 16][NT][4];
    float mrun[NT][2], lrun[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mrun[nt][e] = -INFINITY;
        lrun[nt][e] = 0.0f;
      }
#pragma unroll
      for (int i = 0; i < D / 16; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[i][nt][e] = 0.0f;
    }

    // Raw rows of keys kbs .. kbs+31 into stage st (one commit group per
    // call).  Lane l owns key kbs + l: its page id (read one step ahead) and
    // its two scale rows.  The code rows are copied by the whole warp, so that
    // each instruction reads 512 contiguous bytes of one page (8 rows of 64
    // bytes or 16 of 32): instruction i copies rows kRpi*i .. kRpi*i + kRpi-1
    // in 16-byte chunks.  A key past the piece gets zero V scales, so its
    // stale V codes weigh 0.
    constexpr int kChunks = D / 32;      // 16-byte chunks per code row
    constexpr int kRpi = 32 / kChunks;   // code rows per warp instruction
    const int ps_mask = p.page_size - 1;
    auto page_of = [&](int key) { return key < k1 ? __ldg(pt + (key >> p.ps_shift)) : 0; };
    int page_next = page_of(k0 + lane);
    auto row_of = [&](int page, int key) {
      return (static_cast<int64_t>(page) * p.num_kv_heads + hk) * p.page_size + (key & ps_mask);
    };
    auto issue = [&](int kbs, int st) {
      const int key = kbs + lane;
      int page = page_next;
      page_next = page_of(key + 32);
      uint8_t* s = ring + st * kStage;
      if (key < k1 && (page < 0 || page >= p.num_pages)) {
        atomicOr(p.status, FI_DEV_PAGE_OOB);
        page = 0;
      }
      // each half step (16 keys, 16-aligned) lies in one page: the cache row
      // of its first key, from the page id of the lane that owns that key
      const int64_t row_h0 = row_of(__shfl_sync(0xFFFFFFFFu, page, 0), kbs);
      const int64_t row_h1 = row_of(__shfl_sync(0xFFFFFFFFu, page, 16), kbs + 16);
#pragma unroll
      for (int i = 0; i < kChunks; ++i) {
        const int kr = kRpi * i + lane / kChunks;  // the step's row this lane copies
        const int ch = lane % kChunks;
        if (kbs + kr < k1) {
          const int64_t row = (kr < 16 ? row_h0 : row_h1) + (kr & 15);
          cp_async16(s + kr * (D / 2) + 16 * ch, p.k_data + row * (D / 2) + 16 * ch);
          cp_async16(s + kV + kr * kVR + 16 * ch, p.v_data + row * (D / 2) + 16 * ch);
        }
      }
      if (key < k1) {
        const int64_t row = (lane < 16 ? row_h0 : row_h1) + (lane & 15);
        if constexpr (D == 128) {
          cp_async8(s + kKsf + lane * 8, p.k_sf + row * 8);
          cp_async8(s + kVsf + lane * kVsfS, p.v_sf + row * 8);
        } else {
          cp_async4(s + kKsf + lane * 4, p.k_sf + row * 4);
          cp_async4(s + kVsf + lane * kVsfS, p.v_sf + row * 4);
        }
      } else {
        if constexpr (D == 128)
          *reinterpret_cast<uint2*>(s + kVsf + lane * kVsfS) = make_uint2(0u, 0u);
        else
          *reinterpret_cast<uint32_t*>(s + kVsf + lane * kVsfS) = 0u;
      }
      cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < kTStages - 1; ++i) issue(k0 + 32 * i, i);

    int st = 0;
    for (int kb = k0; kb < k1; kb += 32) {
      __syncwarp();  // every lane is done with the stage read in the previous step
      issue(kb + 32 * (kTStages - 1), st == 0 ? kTStages - 1 : st - 1);
      cp_async_wait<kTStages - 1>();  // this lane's rows of this step have landed
      __syncwarp();                   // ... and every lane's
      const uint8_t* sb = ring + st * kStage;

      // ---- S^T = K Q^T: m-tiles of keys 0-15 and 16-31.  Keys past k1 read
      // stale bytes; their logits are replaced by -inf below.  A lane converts
      // its code words of keys g, g+8 (m-tile 0) and 16+g, 24+g (m-tile 1).
      float sacc[2][NT][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.0f;
      // code words and scale bytes of key 16 mt + 8 z + g
      auto load_k = [&](int mt, int z, uint32_t (&cw)[kKW], uint32_t& sf) {
        const int key = 16 * mt + 8 * z + g;
        if constexpr (D == 128) {
          const uint4 x = *reinterpret_cast<const uint4*>(sb + key * 64 + 16 * t);
          cw[0] = x.x;
          cw[1] = x.y;
          cw[2] = x.z;
          cw[3] = x.w;
          sf = *reinterpret_cast<const uint16_t*>(sb + kKsf + key * 8 + 2 * t);
        } else {
          const uint2 x = *reinterpret_cast<const uint2*>(sb + key * 32 + 8 * t);
          cw[0] = x.x;
          cw[1] = x.y;
          sf = sb[kKsf + key * 4 + t];
        }
      };
      // code word i holds bytes 4i .. 4i+3 of the lane's range = k-steps 2i and
      // 2i+1; its scale block is the lane's first (bytes 0-7) or second (8-15)
      auto kscale = [&](uint32_t sf, int i) {
        return e4m3x2_to_f16x2(__byte_perm(sf, 0u, i / 2 ? 0x1111u : 0x0000u));
      };
      if constexpr (kQs) {
        // Q fragments from shared memory: each is read once and used for both
        // m-tiles, so the words of all four keys are converted together
        uint32_t cw[2][2][kKW], sfb[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int z = 0; z < 2; ++z) load_k(mt, z, cw[mt][z], sfb[mt][z]);
#pragma unroll
        for (int i = 0; i < kKW; ++i) {
          uint32_t hc[2][2][4], sc[2][2];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int z = 0; z < 2; ++z) {
              sc[mt][z] = kscale(sfb[mt][z], i);
              e2m1x8_to_f16x2(cw[mt][z][i], hc[mt][z]);
            }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              a[mt][0] = hmul2_u32(hc[mt][0][2 * h], sc[mt][0]);
              a[mt][1] = hmul2_u32(hc[mt][1][2 * h], sc[mt][1]);
              a[mt][2] = hmul2_u32(hc[mt][0][2 * h + 1], sc[mt][0]);
              a[mt][3] = hmul2_u32(hc[mt][1][2 * h + 1], sc[mt][1]);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint2 q = qfrag(nt, 2 * i + h);
              mma16816(sacc[0][nt], a[0], q.x, q.y);
              mma16816(sacc[1][nt], a[1], q.x, q.y);
            }
          }
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t ca[kKW], cz[kKW], sfa, sfz;
          load_k(mt, 0, ca, sfa);
          load_k(mt, 1, cz, sfz);
#pragma unroll
          for (int i = 0; i < kKW; ++i) {
            const uint32_t sa = kscale(sfa, i), sz = kscale(sfz, i);
            uint32_t ha[4], hz[4];
            e2m1x8_to_f16x2(ca[i], ha);
            e2m1x8_to_f16x2(cz[i], hz);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t a[4];
              a[0] = hmul2_u32(ha[2 * h], sa);
              a[1] = hmul2_u32(hz[2 * h], sz);
              a[2] = hmul2_u32(ha[2 * h + 1], sa);
              a[3] = hmul2_u32(hz[2 * h + 1], sz);
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const uint2 q = qfrag(nt, 2 * i + h);
                mma16816(sacc[mt][nt], a, q.x, q.y);
              }
            }
          }
        }
      }

      // ---- causal mask and online softmax; lane holds rows 8 nt + 2t + e of
      // keys kb + 16 mt + g + 8 h (accumulator element 2h + e).  A step whose
      // 32 keys every row sees (row 0 sees the fewest) takes no mask; rows past
      // R then run on zero logits, finite and never written out.
      const bool full = kb + 31 <= min(k1 - 1, delta);
      // This lane's maximum of each row over its four keys; the row maximum
      // (three shuffles) is taken only when some lane's exceeds the running
      // maximum by more than 8, which the lazy rescale needs to move it.
      float mxl[NT][2];
      bool grow = false;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float mx;
          if (full) {
            mx = fmaxf(fmaxf(sacc[0][nt][e], sacc[0][nt][2 + e]),
                       fmaxf(sacc[1][nt][e], sacc[1][nt][2 + e])) * ssc;
          } else {
            const int r = 8 * nt + 2 * t + e;
            const int lim = r < R ? min(k1 - 1, delta + r / G) : -1;  // last visible key
            mx = -INFINITY;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int key = kb + 16 * mt + g + 8 * h;
                const float x = key <= lim ? sacc[mt][nt][2 * h + e] * ssc : -INFINITY;
                sacc[mt][nt][2 * h + e] = x;
                mx = fmaxf(mx, x);
              }
          }
          mxl[nt][e] = mx;
          grow |= mx > mrun[nt][e] + 8.0f;
        }
      }
      if (__any_sync(0xFFFFFFFFu, grow)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float mx = mxl[nt][e];
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
            if (mx > mrun[nt][e] + 8.0f) {
              const float alpha = ex2_approx(mrun[nt][e] - mx);  // 0 while mrun is -inf
              lrun[nt][e] *= alpha;
#pragma unroll
              for (int i = 0; i < D / 16; ++i) {
                o[i][nt][e] *= alpha;
                o[i][nt][2 + e] *= alpha;
              }
              mrun[nt][e] = mx;
            }
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float m = mrun[nt][e];
          float psum = 0.0f;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const float x = sacc[mt][nt][2 * h + e];
              float pv;
              if (full)
                pv = ex2_approx(fmaf(x, ssc, -m));  // x is the unscaled logit here
              else
                pv = x == -INFINITY ? 0.0f : ex2_approx(x - m);
              sacc[mt][nt][2 * h + e] = pv;
              psum += pv;
            }
          lrun[nt][e] += psum;
        }
      }

      // ---- O^T += V^T P^T, k-steps of keys 0-15 and 16-31
      const uint8_t* vb = sb + kV;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          pb[nt][0] = movmatrix_t(f16x2_of(sacc[kk][nt][0], sacc[kk][nt][1]));
          pb[nt][1] = movmatrix_t(f16x2_of(sacc[kk][nt][2], sacc[kk][nt][3]));
        }
        const int kA = 16 * kk + 2 * t;  // keys kA, kA+1 (k = 2t, 2t+1) and kA+8, kA+9
        uint32_t va[kVW], vb1[kVW], vc[kVW], vd[kVW];
        uint32_t sab, scd;
        if constexpr (D == 128) {
          const uint2 x0 = *reinterpret_cast<const uint2*>(vb + kA * kVR + 8 * g);
          const uint2 x1 = *reinterpret_cast<const uint2*>(vb + (kA + 1) * kVR + 8 * g);
          const uint2 x2 = *reinterpret_cast<const uint2*>(vb + (kA + 8) * kVR + 8 * g);
          const uint2 x3 = *reinterpret_cast<const uint2*>(vb + (kA + 9) * kVR + 8 * g);
          va[0] = x0.x; va[1] = x0.y; vb1[0] = x1.x; vb1[1] = x1.y;
          vc[0] = x2.x; vc[1] = x2.y; vd[0] = x3.x; vd[1] = x3.y;
          sab = sb[kVsf + kA * kVsfS + g] | (sb[kVsf + (kA + 1) * kVsfS + g] << 8);
          scd = sb[kVsf + (kA + 8) * kVsfS + g] | (sb[kVsf + (kA + 9) * kVsfS + g] << 8);
        } else {
          va[0] = *reinterpret_cast<const uint32_t*>(vb + kA * kVR + 4 * g);
          vb1[0] = *reinterpret_cast<const uint32_t*>(vb + (kA + 1) * kVR + 4 * g);
          vc[0] = *reinterpret_cast<const uint32_t*>(vb + (kA + 8) * kVR + 4 * g);
          vd[0] = *reinterpret_cast<const uint32_t*>(vb + (kA + 9) * kVR + 4 * g);
          sab = sb[kVsf + kA * kVsfS + g / 2] | (sb[kVsf + (kA + 1) * kVsfS + g / 2] << 8);
          scd = sb[kVsf + (kA + 8) * kVsfS + g / 2] | (sb[kVsf + (kA + 9) * kVsfS + g / 2] << 8);
        }
        const uint32_t s01 = e4m3x2_to_f16x2(sab), s89 = e4m3x2_to_f16x2(scd);
#pragma unroll
        for (int j = 0; j < kVW; ++j) {
          // byte i of a word: low nibbles of the two keys (head dimension
          // 2(g D/16 + 4j + i)), then their high nibbles (the next dimension)
          const uint32_t lo01 = (va[j] & 0x0F0F0F0Fu) | ((vb1[j] << 4) & 0xF0F0F0F0u);
          const uint32_t hi01 = ((va[j] >> 4) & 0x0F0F0F0Fu) | (vb1[j] & 0xF0F0F0F0u);
          const uint32_t lo89 = (vc[j] & 0x0F0F0F0Fu) | ((vd[j] << 4) & 0xF0F0F0F0u);
          const uint32_t hi89 = ((vc[j] >> 4) & 0x0F0F0F0Fu) | (vd[j] & 0xF0F0F0F0u);
          uint32_t l01[4], h01[4], l89[4], h89[4];
          e2m1x8_to_f16x2(lo01, l01);
          e2m1x8_to_f16x2(hi01, h01);
          e2m1x8_to_f16x2(lo89, l89);
          e2m1x8_to_f16x2(hi89, h89);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t a[4];
            a[0] = hmul2_u32(l01[i], s01);
            a[1] = hmul2_u32(h01[i], s01);
            a[2] = hmul2_u32(l89[i], s89);
            a[3] = hmul2_u32(h89[i], s89);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma16816(o[4 * j + i][nt], a, pb[nt][0], pb[nt][1]);
          }
        }
      }
      st = st == kTStages - 1 ? 0 : st + 1;
    }

    cp_async_wait<0>();  // (the copies past the chunk are empty groups; none is left in flight)

    // ---- results: lane holds head dimensions g D/8 .. g D/8 + D/8 - 1 of rows
    // 8 nt + 2t + e (m-tile i gives dimensions g D/8 + 2i and the one after)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float lsum = lrun[nt][e];
        lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 4);
        lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 8);
        lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 16);
        const int r = 8 * nt + 2 * t + e;
        if (r >= R) continue;
        const int d0 = g * (D / 8);
        if (slot < 0) {
          const int64_t orow =
              static_cast<int64_t>(qo_start + r / G) * p.num_qo_heads + hk * G + r % G;
          const float inv = vs / lsum;
          uint32_t packed[D / 16];
#pragma unroll
          for (int i = 0; i < D / 16; ++i) {
            const __nv_bfloat162 v2 =
                __floats2bfloat162_rn(o[i][nt][e] * inv, o[i][nt][2 + e] * inv);
            packed[i] = *reinterpret_cast<const uint32_t*>(&v2);
          }
          uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D + d0);
#pragma unroll
          for (int i = 0; i < D / 64; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                packed[4 * i + 3]);
          if (p.lse && g == 0) p.lse[orow] = (mrun[nt][e] + log2f(lsum)) * 0.6931471805599453f;
        } else {
          float* dst = p.part + (static_cast<int64_t>(slot) * p.rows + r) * (D + 2);
#pragma unroll
          for (int i = 0; i < D / 16; ++i)
            *reinterpret_cast<float2*>(dst + d0 + 2 * i) =
                make_float2(o[i][nt][e], o[i][nt][2 + e]);
          if (g == 0) {
            dst[D] = mrun[nt][e];
            dst[D + 1] = lsum;
          }
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
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32;
  const int item = warp / p.rows, r = warp % p.rows;
  // the merge item and the lengths are plan memory (no kernel writes it):
  // read while the decode kernel finishes; its partial results after the wait
  int4 w = make_int4(0, 0, 0, 0);
  int qo_start = 0, qo_len = 0;
  if (item < p.num_merges) {
    w = __ldg(p.merges + item);
    qo_start = __ldg(p.qo_indptr + w.x);
    qo_len = __ldg(p.qo_indptr + w.x + 1) - qo_start;
  }
  grid_dep_wait();
  grid_dep_launch();
  if (item >= p.num_merges) return;
  const int b = w.x, hk = w.y, first = w.z, n = w.w;
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

template <int D, int NT>
fi_status launch_decode_t_impl(const DecodeParams& p, cudaStream_t stream) {
  const int smem = decode_t_smem_bytes<D, NT>();
  auto kern = nvfp4_decode_t_kernel<D, NT>;
  // the shared-memory attribute is set once per device (a race between host
  // threads only sets it twice)
  static std::atomic<int> attr_set[kDecMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FI_ERR_CUDA;
  if (dev < 0 || dev >= kDecMaxDevices) return FI_ERR_UNSUPPORTED;
  if (attr_set[dev].load(std::memory_order_relaxed) == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return FI_ERR_CUDA;
    attr_set[dev].store(1, std::memory_order_relaxed);
  }
  const unsigned grid = static_cast<unsigned>((p.num_warps + kTWarps - 1) / kTWarps);
  fi_status st = launch_pdl(kern, dim3(grid), dim3(32 * kTWarps), smem, stream, p);
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

  p.num_merges = static_cast<int32_t>(P.dec_merges.size() / 4);
  p.num_qo_heads = P.num_qo_heads;
  p.num_kv_heads = P.num_kv_heads;
  p.group = P.group;
  p.page_size = P.page_size;
  p.ps_shift = 0;
  while ((1 << p.ps_shift) < P.page_size) ++p.ps_shift;
  p.num_pages = a.cache.num_pages;
  p.warp_off = a.warp_off_dev;
  p.num_warps = P.dec_warps;
  p.rows = P.dec_rows;
  p.sm_scale = P.sm_scale;
  p.status = a.status;
  const int D = P.head_dim;
  if (P.dec_rows <= 8)
    return D == 128 ? launch_decode_t_impl<128, 1>(p, stream)
                    : launch_decode_t_impl<64, 1>(p, stream);
  if (P.dec_rows <= 16)
    return D == 128 ? launch_decode_t_impl<128, 2>(p, stream)
                    : launch_decode_t_impl<64, 2>(p, stream);
  return D == 128 ? launch_decode_t_impl<128, 4>(p, stream)
                  : launch_decode_t_impl<64, 4>(p, stream);
}

}  // namespace fi
