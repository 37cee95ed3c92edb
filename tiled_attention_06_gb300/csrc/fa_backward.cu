// FlashAttention backward for sm_103a: the gradients of O = softmax(scale Q K^T + mask) V,
// recomputing the scores from the saved LSE instead of storing them (the reason the
// pages give for re-reading the scores in the backward pass; "zwxr.cn article on
// ops-transformer", section 3.1, and the ops-transformer overview, section 二.1).
// Per (batch, head), with D_i = dO_i . O_i:
//   P = exp(scale Q K^T - LSE), dV = P^T dO, dP = dO V^T, dS = P (dP - D),
//   dQ = scale dS K, dK = scale dS^T Q.
//
// Three kernels, each step on the tensor cores where it is a contraction:
//   bwd_prep_kernel   D_i, one FP32 per query row (HBM-bound), and zeros the FP32 dQ
//                     accumulator.
//   bwd_dkdv_kernel   one CTA per (batch*head, block of 128 keys), dispatched in groups of
//                     heads, key block by key block within a group (bwd_item); TMEM lane = key. For
//                     each block of 128 queries that sees these keys, in two halves of 64
//                     queries: S^T = K Q^T and dP^T = V dO^T (tcgen05, A and B from shared
//                     memory); P^T and dS^T = P^T (dP^T - D) by the elementwise warps, P^T
//                     rounded to 16 bits over its own TMEM columns and dS^T into shared
//                     memory; then dV += P^T dO (A from TMEM), dK += dS^T Q and
//                     dQ^T = K^T dS^T (A and B from shared memory; TMEM lane = element of
//                     d), the last added by the elementwise warps into an FP32 dQ
//                     accumulator in global memory laid out [B*H][ceil(Sq/4)][d][4] (query
//                     q, element c at ((q/4) d + c) 4 + q%4), so that one thread adds four
//                     consecutive queries of its element in one 16-byte reduction and one
//                     warp instruction covers 512 contiguous bytes.
//   bwd_dq_convert_kernel  dq = scale * accumulator, rounded to 16 bits (HBM-bound).
// Each visible (query block, key block) pair is visited once: five products over the
// visible pairs, none recomputed.
//
// Roles of the dK/dV kernel (576 threads): four elementwise warpgroups, two per 64-wide
// half of every tile (warps 0-7 the first half, 8-15 the second; in each pair the first
// warpgroup takes the half's first 32 columns, the second the last 32; one TMEM lane per
// thread; all four share the epilogue), warp 16 TMA, warp 17 MMA (warp-wide, one elected
// lane issues). Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cstdint>
#include <type_traits>

#include "fa_bwd_tiles.h"
#include "fa_internal.h"
#include "fa_mma.cuh"
#include "fa_plan.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kBT = 128;  // rows of a query or key tile
constexpr int kBwdThreads = 576;
constexpr int kBwdTmaWarp = 16;
constexpr int kBwdMmaWarp = 17;
constexpr int kBwdEwPerHalf = 256;  // elementwise threads per half (two warpgroups)

// The streamed side moves in halves of 64 rows (kBwdBoxRows, the tensor maps' box height):
// stage h holds one half of each of the two streamed tiles, and is released as soon as the
// MMAs of that half are done, so the next loads start half a tile earlier than whole-tile
// stages would let them.
constexpr int kHalf = kBwdBoxRows;
constexpr int kStages = 4;
static_assert(kHalf * 2 == kBT, "two halves per tile");

template <int D>
struct BwdCfg {
  static constexpr int TILE = kBT * D * 2;   // one 128-row 16-bit tile (resident)
  static constexpr int HTILE = kHalf * D * 2;  // one 64-row half (streamed)
  static constexpr int DS = kBT * kHalf * 2;   // dS^T of one half: 128 keys x 64 queries
  static constexpr int STATS = 2 * kHalf * 4;  // per stage: LSE * log2(e) and D of 64 queries
  static constexpr int BARS = 256;             // BwdBars, rounded up
  // From a 1024-byte aligned base: K, V (resident), four stages of two streamed halves,
  // dS^T of both halves, statistics, barriers.
  static constexpr int BODY = 2 * TILE + kStages * 2 * HTILE + 2 * DS + kStages * STATS + BARS;
  // The allocation leaves room to align the base when the device's dynamic shared memory
  // does not start 1024-byte aligned, up to the per-block limit; the kernel checks that its
  // base fits (at d = 128 it does when the allocation starts at most 768 bytes short of a
  // 1024-byte boundary, and the usual start is on one).
  static constexpr int WANT = BODY + 1023;
  static constexpr int SMEM = WANT < 232448 ? WANT : 232448;
  static_assert(BODY + 768 <= SMEM, "shared memory over budget");
  // over half the SM's shared memory: one CTA (which takes all 512 TMEM columns) per SM
  static_assert(BODY > 116 * 1024, "two CTAs would share an SM");
};

struct BwdBars {
  uint64_t res_full;              // the CTA's resident tiles landed
  uint64_t st_full[kStages];      // streamed halves of stage h landed
  uint64_t st_empty[kStages];     // MMAs done with stage h
  uint64_t s_full[2];             // S^T and dP^T of half u of the current tile in TMEM
  uint64_t p_full[2];             // P^T (TMEM) and dS^T (shared memory) of half u written
  uint64_t dq_full[2];            // dQ^T of half u in TMEM (over the dP^T columns)
  uint64_t dq_read[2];            // the elementwise warps of half u have read dQ^T
  uint64_t acc_full;              // every MMA of the CTA complete
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(BwdBars) <= 256, "barrier block over its reserve");

// 32 lanes x 16 columns of 32-bit TMEM -> 16 registers per thread, and 8 registers -> 8
// columns: the elementwise step works on 16 queries at a time.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// Half g = 2 t + u of the stream (tile t, half u) lives in stage g % kStages; its fills and
// releases alternate parity every kStages halves.
__device__ __forceinline__ int stage_of(int g) { return g % kStages; }
__device__ __forceinline__ uint32_t stage_parity(int g) { return (g / kStages) & 1; }

// Key positions are the query index plus delta = Sk - Sq (queries aligned to the last
// Sq keys), as in the forward.

// Queries that see key j, as the interval [lo, hi] of columns of the query tile at m0
// (the transpose of the same masks); empty when lo > hi.
struct RowSpan {
  int lo, hi;
};
__device__ __forceinline__ RowSpan query_cols(int j, int m0, int sk, const PrefillParams& p) {
  const long long delta = static_cast<long long>(sk) - p.Sq;
  long long lo = 0, hi = static_cast<long long>(p.Sq) - 1;  // query indices
  if (j >= sk) return RowSpan{1, 0};
  switch (p.mask_mode) {
    case FA_MASK_CAUSAL:  // pos >= j
      lo = j - delta;
      break;
    case FA_MASK_CAUSAL_WINDOW:  // pos >= j and (pos - j < w or j < g)
      lo = j - delta;
      if (j >= p.n_global) hi = min(hi, j - delta + p.window - 1);
      break;
    case FA_MASK_BAND:  // |pos - j| <= w
      lo = j - delta - p.window;
      hi = min(hi, j - delta + p.window);
      break;
    case FA_MASK_PREFIX_LM:  // pos >= j or j < g
      if (j >= p.n_global) lo = j - delta;
      break;
    default:
      break;
  }
  if (lo < 0) lo = 0;
  lo -= m0;
  hi -= m0;
  return RowSpan{static_cast<int>(lo < -1 ? -1 : (lo > kBT ? kBT : lo)),
                 static_cast<int>(hi < -1 ? -1 : (hi > kBT ? kBT : hi))};
}

__device__ __forceinline__ void wait_quiet_b(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  volatile uint32_t zero = 0;
  WaitCtx w2 = wc;
  w2.abort = &zero;
  mbar_wait(bar, parity, w2);
}

// D_i = sum_c dO_ic O_ic in FP32: d/8 lanes per row, one 16-byte load of each per lane,
// xor-shuffle reduction inside the row's lanes. The grid also zeros the n4 float4s of the
// FP32 dQ accumulator.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint4* __restrict__ o,
                                                       const uint4* __restrict__ dout,
                                                       float* __restrict__ dsum,
                                                       float4* __restrict__ dqacc, int64_t rows,
                                                       int64_t n4) {
  {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride)
      dqacc[i] = z;
  }
  constexpr int LPR = D / 8;  // lanes per row
  constexpr int RPW = 32 / LPR;
  const int lane = threadIdx.x % 32;
  const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * blockDim.x / 32;
  for (int64_t r0 = warp * RPW; r0 < rows; r0 += nwarps * RPW) {
    const int64_t row = r0 + lane / LPR;
    float acc = 0.f;
    if (row < rows) {
      const uint4 a = o[row * LPR + lane % LPR], b = dout[row * LPR + lane % LPR];
      const uint32_t* ap = reinterpret_cast<const uint32_t*>(&a);
      const uint32_t* bp = reinterpret_cast<const uint32_t*>(&b);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float2 x, y;
        if (BF16) {
          x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(ap + e));
          y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(bp + e));
        } else {
          x = __half22float2(*reinterpret_cast<const __half2*>(ap + e));
          y = __half22float2(*reinterpret_cast<const __half2*>(bp + e));
        }
        acc += x.x * y.x + x.y * y.y;
      }
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off /= 2) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && lane % LPR == 0) dsum[row] = acc;
  }
}

// dq = scale * accumulator, rounded to 16 bits. A block takes 32 queries of one (batch,
// head): it loads their [8 groups][D][4] accumulator floats as contiguous float4s, transposes
// them through shared memory (one padded row per query) and writes each query's row as
// 16-byte chunks of 8 elements, consecutive threads on consecutive chunks.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                             uint4* __restrict__ dq, float scale,
                                                             int Sq, int64_t nblk) {
  constexpr int G = 8;  // groups of four queries per block
  __shared__ __align__(16) float tile[G * 4][D + 4];  // rows of (D + 4) * 4 bytes: 16-byte aligned
  const int sq4 = (Sq + 3) / 4;
  const int per_bh = (sq4 + G - 1) / G;
  for (int64_t blk = blockIdx.x; blk < nblk; blk += gridDim.x) {
    const int64_t bh = blk / per_bh;
    const int g0 = static_cast<int>(blk % per_bh) * G;
    const int ng = min(G, sq4 - g0);
    const float4* src = acc + (bh * sq4 + g0) * D;
    for (int i = threadIdx.x; i < ng * D; i += blockDim.x) {
      const float4 v = src[i];
      const int g = i / D, c = i % D;
      tile[4 * g][c] = v.x;
      tile[4 * g + 1][c] = v.y;
      tile[4 * g + 2][c] = v.z;
      tile[4 * g + 3][c] = v.w;
    }
    __syncthreads();
    const int nq = min(G * 4, Sq - g0 * 4);
    for (int i = threadIdx.x; i < nq * (D / 8); i += blockDim.x) {
      const int qq = i / (D / 8), c8 = i % (D / 8);
      const float4 lo = *reinterpret_cast<const float4*>(&tile[qq][8 * c8]);
      const float4 hi = *reinterpret_cast<const float4*>(&tile[qq][8 * c8 + 4]);
      const uint32_t p0 = BF16 ? cvt_pack_bf16(lo.x * scale, lo.y * scale) : cvt_pack_f16(lo.x * scale, lo.y * scale);
      const uint32_t p1 = BF16 ? cvt_pack_bf16(lo.z * scale, lo.w * scale) : cvt_pack_f16(lo.z * scale, lo.w * scale);
      const uint32_t p2 = BF16 ? cvt_pack_bf16(hi.x * scale, hi.y * scale) : cvt_pack_f16(hi.x * scale, hi.y * scale);
      const uint32_t p3 = BF16 ? cvt_pack_bf16(hi.z * scale, hi.w * scale) : cvt_pack_f16(hi.z * scale, hi.w * scale);
      dq[((bh * Sq + g0 * 4 + qq) * D) / 8 + c8] = make_uint4(p0, p1, p2, p3);
    }
    __syncthreads();
  }
}

// Half-tile MMAs: every tile of 128 queries (or keys) is processed as two halves u of 64,
// so that the tensor core works on one half while the elementwise warps work on the other.
// X_u = A B_u^T: A a resident 128-row tile (regions of 64 elements of d 16 KB apart), B_u a
// streamed 64-row half (regions 8 KB apart), both K-major and 128-byte swizzled; M = 128,
// N = 64.
template <int D, bool BF16>
__device__ __forceinline__ void issue_s_half(uint32_t d_tmem, uint32_t a_smem, uint32_t b_half) {
  constexpr uint32_t id = idesc_f16(BF16, kBT, kHalf, false);
  const uint64_t a0 = smem_desc_sw128(a_smem, 16, 1024);
  const uint64_t b0 = smem_desc_sw128(b_half, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t a_off = static_cast<uint64_t>((kk / 4) * (kBT * 128 / 16) + (kk % 4) * 2);
    const uint64_t b_off = static_cast<uint64_t>((kk / 4) * (kHalf * 128 / 16) + (kk % 4) * 2);
    umma_ss(d_tmem, a0 + a_off, b0 + b_off, id, kk > 0 ? 1u : 0u);
  }
}

// Y (+)= A_u B_u: A_u the half's 64 elements of K as packed 16-bit values in TMEM, written
// by the two elementwise warpgroups of the half over their own columns: K-elements 0-31 in
// columns [a, a+16), 32-63 in [a+32, a+48); B_u a streamed 64-row half used MN-major (N = D,
// its second 64 elements of d 8 KB on; 16 rows = 2048 bytes per MMA).
template <int D, bool BF16>
__device__ __forceinline__ void issue_pv_half(uint32_t y_tmem, uint32_t a_tmem, uint32_t b_half,
                                              bool accumulate) {
  constexpr uint32_t id = idesc_f16(BF16, kBT, D, true);
  const uint64_t b0 = smem_desc_sw128(b_half, kHalf * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < kHalf / 16; ++kk)
    umma_ts(y_tmem, a_tmem + (kk / 2) * 32 + (kk % 2) * 8, b0 + static_cast<uint64_t>(kk * 128),
            id, (accumulate || kk > 0) ? 1u : 0u);
}

// dK (+)= dS^T_u Q_u: A = dS^T_u in shared memory (128 keys x 64 queries, K-major, one
// 128-byte swizzled region), B = Q_u, the streamed 64-row half used MN-major as in
// issue_pv_half.
template <int D, bool BF16>
__device__ __forceinline__ void issue_dk_half(uint32_t y_tmem, uint32_t ds, uint32_t b_half,
                                              bool accumulate) {
  constexpr uint32_t id = idesc_f16(BF16, kBT, D, true);
  const uint64_t a0 = smem_desc_sw128(ds, 16, 1024);
  const uint64_t b0 = smem_desc_sw128(b_half, kHalf * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < kHalf / 16; ++kk)
    umma_ss(y_tmem, a0 + static_cast<uint64_t>(kk * 2), b0 + static_cast<uint64_t>(kk * 128), id,
            (accumulate || kk > 0) ? 1u : 0u);
}

// dQ^T_u = K^T dS^T_u (M = D elements of d, N = 64 queries, K = 128 keys): A = the resident
// K tile read MN-major (its 64-element regions of d 16 KB apart), B = dS^T_u read MN-major
// (keys are its rows); 16 keys = 2048 bytes per MMA in both. With D = 64 the accumulator
// takes the M = 64 layout: row r of dQ^T in TMEM lane 32 (r / 16) + r % 16.
template <int D, bool BF16>
__device__ __forceinline__ void issue_dq_half(uint32_t y_tmem, uint32_t k_smem, uint32_t ds) {
  constexpr uint32_t id = idesc_f16(BF16, D, kHalf, true, true);
  const uint64_t a0 = smem_desc_sw128(k_smem, kBT * 128, 1024);
  const uint64_t b0 = smem_desc_sw128(ds, kBT * 128, 1024);
#pragma unroll
  for (int kk = 0; kk < kBT / 16; ++kk)
    umma_ss(y_tmem, a0 + static_cast<uint64_t>(kk * 128), b0 + static_cast<uint64_t>(kk * 128), id,
            kk > 0 ? 1u : 0u);
}

// A resident 128-row tile as two 64-row boxes per 64-element region of d (the region's
// second box 8 KB after the first, which is the 128-row box's layout).
template <int D>
__device__ __forceinline__ void load_resident(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                              int row0, int bh) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c)
#pragma unroll
    for (int r = 0; r < 2; ++r)
      tma_load_3d(dst + c * (kBT * 128) + r * (kHalf * 128), map, bar, c * 64, row0 + r * kHalf,
                  bh);
}

// A streamed 64-row half: one box per 64-element region of d, regions 8 KB apart.
template <int D>
__device__ __forceinline__ void load_half(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                          int row0, int bh) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * (kHalf * 128), map, bar, c * 64, row0, bh);
}

// Does the query block qb see any key of key block kb (the forward's key ranges; for a
// block layout, its 128 x 128 block, which is then seen whole)?
__device__ __forceinline__ bool tile_visited(int qb, int kb, int bh, const PrefillParams& p) {
  if (p.mask_mode == FA_MASK_BLOCK_SPARSE)
    return p.layout[(static_cast<size_t>(bh % p.H) * p.lnqb + qb) * p.lnkb + kb] != 0;
  const Range r = key_range(qb * kBT, min(qb * kBT + kBT, p.Sq), kBT, p.Sk, p, bh);
  return range_has(r, kb);
}

// The (batch*head, key block) of CTA x. Heads go in groups of G (the last group may be
// smaller); within a group the order is key block-major: key block 0 of every head of the
// group, then key block 1, and so on. Under the causal, window and prefix masks the low key
// blocks are seen by the most query blocks, so a group's longest CTAs start first and its
// last CTAs are short, which evens out the end of the launch; and the CTAs running at one
// time belong to a few groups, whose streamed Q and dO and whose dQ accumulators stay in L2.
// With G = 1 this is the plain head-major order.
__device__ __forceinline__ void bwd_item(int x, int BH, int nkb, int G, int& bh, int& kb) {
  const int per = G * nkb;
  const int grp = x / per, w = x - grp * per;
  const int gs = min(G, BH - grp * G);
  kb = w / gs;
  bh = grp * G + (w - kb * gs);
}

// The next query block after qb that sees key block kb, or nqb.
__device__ __forceinline__ int next_qb(int qb, int kb, int bh, const PrefillParams& p, int nqb) {
  do {
    ++qb;
  } while (qb < nqb && !tile_visited(qb, kb, bh, p));
  return qb;
}

template <int D, bool BF16>
__device__ __forceinline__ void store_tile_row(void* out, size_t row, const uint32_t* v,
                                               float mul, int c0) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float a = __uint_as_float(v[2 * e]) * mul, b = __uint_as_float(v[2 * e + 1]) * mul;
    pk[e] = BF16 ? cvt_pack_bf16(a, b) : cvt_pack_f16(a, b);
  }
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + row * D + c0);
#pragma unroll
  for (int e = 0; e < 4; ++e) dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
}

// Common CTA setup: barriers, TMEM, descriptor prefetch. Returns the TMEM base.
__device__ __forceinline__ uint32_t bwd_setup(BwdBars* bars, const CUtensorMap* m0,
                                              const CUtensorMap* m1, const CUtensorMap* m2,
                                              const CUtensorMap* m3) {
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars->res_full), 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->st_full[i]), 1);
      mbar_init(smem_u32(&bars->st_empty[i]), 1);
    }
    for (int u = 0; u < 2; ++u) {
      mbar_init(smem_u32(&bars->s_full[u]), 1);
      mbar_init(smem_u32(&bars->p_full[u]), kBwdEwPerHalf);
      mbar_init(smem_u32(&bars->dq_full[u]), 1);
      mbar_init(smem_u32(&bars->dq_read[u]), kBwdEwPerHalf);
    }
    mbar_init(smem_u32(&bars->acc_full), 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == kBwdTmaWarp && threadIdx.x % 32 == 0) {
    tma_prefetch_desc(m0);
    tma_prefetch_desc(m1);
    tma_prefetch_desc(m2);
    tma_prefetch_desc(m3);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return bars->tmem_base;
}

__device__ __forceinline__ void bwd_teardown(uint32_t tmem) {
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x / 32 == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// dK, dV and the dQ contributions of one block of 128 keys. TMEM: S^T [0,128) (P^T packed
// over the first 16 of every 32 columns), dP^T [128,256) (dQ^T of half u over [128+64u,
// 192+64u) once dP^T has been read), dV [256,256+D), dK [256+D,256+2D). Shared memory
// from a 1024-byte aligned base: K, V (resident), (Q, dO) halves of 64 queries in four
// stages, dS^T of each half, the stages' statistics, the barriers.
template <int D, bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmdO, const PrefillParams p,
                    const BwdParams b) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  if (base - raw + C::BODY > static_cast<uint32_t>(C::SMEM)) {  // uniform over the CTA
    if (threadIdx.x == 0) atomicOr(p.status, FA_DEV_SMEM_BASE);
    return;
  }
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sK = base, sV = base + C::TILE;
  const uint32_t sSt = base + 2 * C::TILE;  // stage h: Q half at sSt + 2h HTILE, dO half one on
  auto sQh = [&](int h) { return sSt + 2 * h * C::HTILE; };
  auto sdOh = [&](int h) { return sSt + (2 * h + 1) * C::HTILE; };
  const uint32_t sDS = sSt + kStages * 2 * C::HTILE;  // dS^T of half u at sDS + u DS
  // [stage][-LSE2 | -D][64]
  float* stats = reinterpret_cast<float*>(smem + 2 * C::TILE + kStages * 2 * C::HTILE + 2 * C::DS);
  BwdBars* bars = reinterpret_cast<BwdBars*>(reinterpret_cast<uint8_t*>(stats) + kStages * C::STATS);
  auto B = [&](uint64_t& x) { return smem_u32(&x); };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nkb = (p.Sk + kBT - 1) / kBT, nqb = (p.Sq + kBT - 1) / kBT;
  int bh, kb;
  bwd_item(blockIdx.x, p.BH, nkb, b.head_group, bh, kb);
  const uint32_t tmem = bwd_setup(bars, &tmQ, &tmK, &tmV, &tmdO);
  const WaitCtx wc{&bars->abort, p.status, p.timeout_ns};

  if (warp == kBwdTmaWarp) {
    // ------------------------------------------------------------ TMA
    const bool leader = elect_one();
    bool ok = true;
    uint32_t fills[kStages] = {0, 0, 0, 0};
    if (leader) {
      mbar_arrive_expect_tx(B(bars->res_full), 2 * C::TILE);
      load_resident<D>(sK, &tmK, B(bars->res_full), kb * kBT, bh);
      load_resident<D>(sV, &tmV, B(bars->res_full), kb * kBT, bh);
    }
    int g = 0;  // half index of the stream
    for (int qb = next_qb(-1, kb, bh, p, nqb); qb < nqb && ok; qb = next_qb(qb, kb, bh, p, nqb)) {
      for (int u = 0; u < 2 && ok; ++u, ++g) {
        const int h = stage_of(g);
        // LSE and D of the half's 64 queries, 2 per lane (0 past Sq), loaded before the
        // wait for the stage so that their latency overlaps it
        float lv[2], dv[2];
        const size_t r0 = static_cast<size_t>(bh) * p.Sq;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = qb * kBT + u * kHalf + lane * 2 + e;
          lv[e] = i < p.Sq ? __ldg(b.lse + r0 + i) : 0.f;
          dv[e] = i < p.Sq ? __ldg(b.dsum + r0 + i) : 0.f;
        }
        if (g >= kStages && !(ok = mbar_wait(B(bars->st_empty[h]), stage_parity(g - kStages), wc)))
          break;
        {  // the stage's statistics, negated: -LSE * log2(e) and -D
          float* st = stats + h * 2 * kHalf;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            st[lane * 2 + e] = -lv[e] * 1.4426950408889634f;
            st[kHalf + lane * 2 + e] = -dv[e];
          }
          __syncwarp();  // the leader's arrive below releases every lane's writes
        }
        if (leader) {
          mbar_arrive_expect_tx(B(bars->st_full[h]), 2 * C::HTILE);
          load_half<D>(sQh(h), &tmQ, B(bars->st_full[h]), qb * kBT + u * kHalf, bh);
          load_half<D>(sdOh(h), &tmdO, B(bars->st_full[h]), qb * kBT + u * kHalf, bh);
        }
        fills[h] = g / kStages + 1;
      }
    }
    if (!ok) {  // every load issued lands before the CTA exits
      wait_quiet_b(B(bars->res_full), 0, wc);
      for (int h = 0; h < kStages; ++h)
        if (fills[h] > 0) wait_quiet_b(B(bars->st_full[h]), (fills[h] - 1) & 1, wc);
    }
    __syncwarp();
  } else if (warp == kBwdMmaWarp) {
    // ------------------------------------------------------------ MMA
    const bool leader = elect_one();
    // Per tile t and half u: wait for P^T_u / dS^T_u; dV += P^T_u dO_u, dK += dS^T_u Q_u,
    // release the half's stage, dQ^T_u = K^T dS^T_u over the dP^T_u columns; then S^T_u of
    // the next tile over the columns that dV has just read (MMAs of one thread execute in
    // order) and, once the elementwise warps have read dQ^T_u, dP^T_u of the next tile. The
    // tensor core works on one half while the elementwise warps work on the other.
    bool ok = mbar_wait(B(bars->res_full), 0, wc);
    int qb = ok ? next_qb(-1, kb, bh, p, nqb) : nqb;
    auto s_half = [&](int g, int u) {  // S^T_u = K Q_u^T once stream half g has landed
      if (!(ok = mbar_wait(B(bars->st_full[stage_of(g)]), stage_parity(g), wc))) return;
      tc_fence_after();
      if (leader) issue_s_half<D, BF16>(tmem + 64 * u, sK, sQh(stage_of(g)));
    };
    auto dp_half = [&](int g, int u) {  // dP^T_u = V dO_u^T (stage g already landed)
      if (leader) {
        issue_s_half<D, BF16>(tmem + 128 + 64 * u, sV, sdOh(stage_of(g)));
        umma_commit(B(bars->s_full[u]));
      }
    };
    if (qb < nqb && ok) {
      s_half(0, 0);
      if (ok) dp_half(0, 0);
      if (ok) s_half(1, 1);
      if (ok) dp_half(1, 1);
    }
    int t = 0;
    while (qb < nqb && ok) {
      const int qn = next_qb(qb, kb, bh, p, nqb);
      for (int u = 0; u < 2 && ok; ++u) {
        const int g = 2 * t + u, h = stage_of(g);
        if (!(ok = mbar_wait(B(bars->p_full[u]), t & 1, wc))) break;
        tc_fence_after();
        if (leader) {
          const bool acc = t > 0 || u > 0;
          issue_pv_half<D, BF16>(tmem + 256, tmem + 64 * u, sdOh(h), acc);
          issue_dk_half<D, BF16>(tmem + 256 + D, sDS + u * C::DS, sQh(h), acc);
          umma_commit(B(bars->st_empty[h]));  // stage h free once these are done
          issue_dq_half<D, BF16>(tmem + 128 + 64 * u, sK, sDS + u * C::DS);
          umma_commit(B(bars->dq_full[u]));
        }
        if (qn < nqb) {
          s_half(g + 2, u);
          if (!ok || !(ok = mbar_wait(B(bars->dq_read[u]), t & 1, wc))) break;
          tc_fence_after();
          dp_half(g + 2, u);
        }
      }
      qb = qn;
      ++t;
    }
    if (leader) umma_commit(B(bars->acc_full));  // every MMA above done (or none issued)
    wait_quiet_b(B(bars->acc_full), 0, wc);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise + epilogue
    const int grp = warp / 4;  // 0..3: half u = grp / 2, columns [32 sub, 32 sub + 32) of it
    const int u = grp / 2, sub = grp % 2;
    const int row = (warp % 4) * 32 + lane;  // key row of the tile (= TMEM lane)
    const int j = kb * kBT + row;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const uint32_t c_s = 64 * u + 32 * sub;  // this thread's S^T columns; dP^T 128 further
    // this thread's part of dS^T_u: 16-byte chunks 4 sub .. 4 sub + 3 of key row `row`
    // (128-byte swizzle: chunk c of row r at position c ^ (r % 8))
    const uint32_t ds_row = sDS + u * C::DS + row * 128;
    // its TMEM lane in dQ^T_u is an element of d (with D = 64 only lanes 0-15 of each
    // quarter hold one), and its columns the same 32 queries
    const int dcol = D == 128 ? row : (lane < 16 ? (warp % 4) * 16 + lane : -1);
    const int sq4 = (p.Sq + 3) / 4;
    float* dq_col = b.dqacc + (static_cast<size_t>(bh) * sq4 * D + (dcol < 0 ? 0 : dcol)) * 4;
    bool ok = true;
    int t = 0;
    for (int qb = next_qb(-1, kb, bh, p, nqb); qb < nqb && ok; qb = next_qb(qb, kb, bh, p, nqb), ++t) {
      const int g = 2 * t + u, h = stage_of(g);
      // the stage's statistics: the stage cannot be refilled before this warpgroup has
      // written the P and dS that the MMAs reading it wait for
      ok = mbar_wait(B(bars->st_full[h]), stage_parity(g), wc);
      ok = __all_sync(0xffffffffu, ok);
      const float4* st4 = reinterpret_cast<const float4*>(stats + h * 2 * kHalf + 32 * sub);
      if (ok) {
        ok = mbar_wait(B(bars->s_full[u]), t & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const int m0 = qb * kBT + 64 * u + 32 * sub;
        const RowSpan vis = query_cols(j, m0, p.Sk, p);
        // the queries of this thread's 32 columns that see its key, as a bit mask; a warp
        // whose 32 keys all see all 32 queries takes the unmasked path
        uint32_t mk = 0u;
        if (vis.lo <= vis.hi && vis.hi >= 0 && vis.lo <= 31) {
          const int lo = max(vis.lo, 0), hi = min(vis.hi, 31);
          mk = (hi >= 31 ? 0xffffffffu : (2u << hi) - 1u) & ~((1u << lo) - 1u);
        }
        const bool all_vis = __all_sync(0xffffffffu, mk == 0xffffffffu);
        // two chunks of 16 queries: P^T of chunk c packed over columns [8c, 8c + 8) of this
        // thread's 32, which the first chunk has already read
        auto chunks = [&](auto masked) {
          constexpr bool kMasked = decltype(masked)::value;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t sv[16], dp[16];
            tmem_ld16(t_lane + c_s + 16 * c, sv);
            tmem_ld16(t_lane + 128 + c_s + 16 * c, dp);
            tmem_ld_wait<16>(sv);
            tmem_ld_tie<16>(dp);
#pragma unroll
            for (int e = 0; e < 16; e += 4) {  // 4 queries at a time; statistics from shared memory
              // negated statistics, two queries per packed FP32 instruction
              const float4 a = st4[(16 * c + e) / 4];
              const float4 d = st4[kHalf / 4 + (16 * c + e) / 4];
              const uint64_t nl2[2] = {f2(a.x, a.y), f2(a.z, a.w)}, ndd[2] = {f2(d.x, d.y), f2(d.z, d.w)};
              const uint64_t sl2 = f2(p.sl2, p.sl2);
              float pv[4], dv[4];
#pragma unroll
              for (int w = 0; w < 4; w += 2) {
                const uint64_t x = f2_fma(f2(__uint_as_float(sv[e + w]), __uint_as_float(sv[e + w + 1])),
                                          sl2, nl2[w / 2]);
                float x0, x1;
                f2_split(x, x0, x1);
                const int col = 16 * c + e + w;
                pv[w] = (!kMasked || ((mk >> col) & 1u)) ? ex2_approx(x0) : 0.f;
                pv[w + 1] = (!kMasked || ((mk >> (col + 1)) & 1u)) ? ex2_approx(x1) : 0.f;
                const uint64_t dd2 = f2_add(f2(__uint_as_float(dp[e + w]), __uint_as_float(dp[e + w + 1])),
                                            ndd[w / 2]);
                const uint64_t ds2 = f2_fma(f2(pv[w], pv[w + 1]), dd2, f2(0.f, 0.f));
                f2_split(ds2, dv[w], dv[w + 1]);
              }
              sv[e / 2] = BF16 ? cvt_pack_bf16(pv[0], pv[1]) : cvt_pack_f16(pv[0], pv[1]);
              sv[e / 2 + 1] = BF16 ? cvt_pack_bf16(pv[2], pv[3]) : cvt_pack_f16(pv[2], pv[3]);
              dp[e / 2] = BF16 ? cvt_pack_bf16(dv[0], dv[1]) : cvt_pack_f16(dv[0], dv[1]);
              dp[e / 2 + 1] = BF16 ? cvt_pack_bf16(dv[2], dv[3]) : cvt_pack_f16(dv[2], dv[3]);
            }
            tmem_st8(t_lane + c_s + 8 * c, sv);  // P^T over columns already read
#pragma unroll
            for (int i = 0; i < 2; ++i)  // dS^T into shared memory for the dK and dQ MMAs
              st_shared_v4(ds_row + ((static_cast<uint32_t>(4 * sub + 2 * c + i) ^ (row & 7)) << 4),
                           dp[4 * i], dp[4 * i + 1], dp[4 * i + 2], dp[4 * i + 3]);
          }
        };
        if (all_vis)
          chunks(std::false_type{});
        else
          chunks(std::true_type{});
        tmem_st_wait();
        fence_proxy_async_smem();  // the MMAs read dS^T through the async proxy
        tc_fence_before();
        mbar_arrive(B(bars->p_full[u]));
        // this half's dQ^T: read it, hand the columns back, add it into the accumulator
        ok = mbar_wait(B(bars->dq_full[u]), t & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t dq[32];
        tmem_ld32(t_lane + 128 + c_s, dq);
        tmem_ld_wait<32>(dq);
        tc_fence_before();
        mbar_arrive(B(bars->dq_read[u]));
        if (dcol >= 0) {  // per four queries: one warp instruction adds 512 contiguous bytes
          const int ng = min(8, (p.Sq - m0 + 3) / 4);  // groups holding a query below Sq
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (e < ng)
              red_add_v4_f32(dq_col + static_cast<size_t>(m0 / 4 + e) * D * 4, dq[4 * e],
                             dq[4 * e + 1], dq[4 * e + 2], dq[4 * e + 3]);
        }
      }
    }
    // epilogue of this thread's key: warpgroups 0, 1 write halves of dV, 2, 3 halves of
    // scale * dK (D/2 columns each)
    if (ok) {
      ok = mbar_wait(B(bars->acc_full), 0, wc);
      ok = __all_sync(0xffffffffu, ok);
    }
    if (ok) {
      tc_fence_after();
      const size_t orow = static_cast<size_t>(bh) * p.Sk + j;
      const bool is_k = grp >= 2;
      const int c_lo = (grp % 2) * (D / 64);
#pragma unroll 1
      for (int c = c_lo; c < c_lo + D / 64; ++c) {
        uint32_t v[32];
        tmem_ld32(t_lane + 256 + (is_k ? D : 0) + c * 32, v);
        tmem_ld_wait<32>(v);
        if (t == 0) {  // no query sees these keys: the gradients are 0, not TMEM contents
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (j < p.Sk)
          store_tile_row<D, BF16>(is_k ? b.dk : b.dv, orow, v, is_k ? b.scale : 1.f, c * 32);
      }
    }
  }
  bwd_teardown(tmem);
}

template <int D, bool BF16>
cudaError_t launch_bwd_t(const BwdLaunch& L, cudaStream_t stream) {
  if (L.b.head_group < 1) return cudaErrorInvalidValue;  // the launch order divides by it
  const int64_t rows = static_cast<int64_t>(L.p.BH) * L.p.Sq;
  if (rows > 0) {
    const int blocks = static_cast<int>((rows + 63) / 64 < 16384 ? (rows + 63) / 64 : 16384);
    const int64_t n4 = static_cast<int64_t>(L.p.BH) * ((L.p.Sq + 3) / 4) * D;
    bwd_prep_kernel<D, BF16><<<blocks, 256, 0, stream>>>(
        static_cast<const uint4*>(L.o), static_cast<const uint4*>(L.dout),
        const_cast<float*>(L.b.dsum), reinterpret_cast<float4*>(L.b.dqacc), rows, n4);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  constexpr int smem = BwdCfg<D>::SMEM;
  const int nkb = (L.p.Sk + kBT - 1) / kBT;
  if (nkb > 0) {  // with Sq = 0 it still writes the (zero) gradients of every key
    auto k1 = bwd_dkdv_kernel<D, BF16>;
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)))
      return e;
    k1<<<L.p.BH * nkb, kBwdThreads, smem, stream>>>(L.tmQ, L.tmK, L.tmV, L.tmdO, L.p, L.b);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (rows > 0) {  // with Sk = 0 the accumulator stays 0 and so does dq
    const int64_t nblk = static_cast<int64_t>(L.p.BH) * (((L.p.Sq + 3) / 4 + 7) / 8);
    const int blocks = static_cast<int>(nblk < 16384 ? nblk : 16384);
    bwd_dq_convert_kernel<D, BF16><<<blocks, 256, 0, stream>>>(
        reinterpret_cast<const float4*>(L.b.dqacc), static_cast<uint4*>(L.b.dq), L.b.scale,
        L.p.Sq, nblk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_backward(const BwdLaunch& L, int D, bool bf16, cudaStream_t stream) {
  if (D == 128) return bf16 ? launch_bwd_t<128, true>(L, stream) : launch_bwd_t<128, false>(L, stream);
  if (D == 64) return bf16 ? launch_bwd_t<64, true>(L, stream) : launch_bwd_t<64, false>(L, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fa
