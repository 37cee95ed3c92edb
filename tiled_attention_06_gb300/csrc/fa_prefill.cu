// FlashAttention forward (prefill) for sm_103a: tcgen05 MMAs with TMEM accumulators,
// TMA tile loads into a shared-memory ring, warp-specialised online softmax, tile
// skipping for causal and sliding-window(+global) masks, and a persistent
// longest-first tile schedule.
//
// The method is the tiled loop of the ops-transformer overview (gitcode.csdn.net,
// section 二.1 "FlashAttention算子"): an outer loop over query blocks, an inner loop
// over key/value blocks, the score tile S = Q K^T computed on chip and never stored,
// running statistics (max m, sum l) updated per block, and a single normalisation
// O / l at the end. The per-block update is the (m, l, O) recurrence of the zwxr.cn
// article, section 3.1, with the softmax denominator accumulated in FP32 (its
// section 5.1). Prefetching the next K/V block during the current block's compute
// (the same article, section 3.1, "异步预取") is the TMA ring below.
//
// Two kernels share the helpers in this file:
//
// prefill_bm256_kernel (default): a work item is 256 query rows of one (batch, head),
// held as two 128-row tiles A and B that share every K/V tile.
//   warps 0-3  softmax for tile A, warps 4-7 softmax for tile B: one thread per query
//              row (= TMEM lane); S from TMEM, mask on partial tiles, m and l, P
//              (16-bit) written back over S, lazy rescale of O, epilogue.
//   warp 8     TMA producer: Q_A, Q_B, then K0, V0, K1, V1, ... through the ring.
//   warp 9     MMA issuer (one thread). Tensor-pipe order:
//                S_A(0) S_B(0) | PV_A(0) S_A(1) | PV_B(0) S_B(1) | PV_A(1) S_A(2) | ...
//              so one tile's softmax runs while the tensor core works for the other,
//              and S_A(j) is always issued after PV_A(j-1): once the softmax sees
//              S_A(j) complete, O_A holds every earlier P.V product and can be
//              rescaled without waiting.
//   TMEM columns: S_A [0,BN), S_B [BN,2BN), O_A [2BN,2BN+D), O_B [2BN+D,2BN+2D).
//
// prefill_bm128_kernel: one 128-row tile per item, two S buffers so that S(j+1) is
// computed while the softmax works on S(j); warps 0-3 softmax, 4 TMA, 5 MMA.
//   TMEM columns: S0 [0,BN), S1 [BN,2BN), O [2BN,2BN+D).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cstdint>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kTile = 128;                // rows of one tcgen05 M=128 tile (= TMEM lanes)
constexpr float kTau = 8.0f;              // lazy-rescale threshold, log2 units
constexpr uint32_t kSmemLimit = 232448;   // 227 KB opt-in dynamic shared memory per CTA

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

// ------------------------------------------------------------------ shared helpers

// Key blocks visited by the query rows [m0, m1): [0, a_end) then [b_start, b_end),
// a_end <= b_start. Closed form of the mask: every block inside holds at least one
// visible pair for these rows, every block outside holds none.
struct Range {
  int a_end, b_start, b_end;
};

template <int BN>
__device__ __forceinline__ Range key_range(int m0, int m1, const PrefillParams& p) {
  Range r{0, 0, p.nnb};
  if (m0 >= m1) return Range{0, 0, 0};
  if (p.mask_mode == FA_MASK_NONE) return r;
  const int delta = p.Sk - p.Sq;
  const int r_lo = m0 + delta;      // key position of the first row
  const int r_hi = m1 - 1 + delta;  // key position of the last row
  if (r_hi < 0) return Range{0, 0, 0};
  r.b_end = min(p.nnb, r_hi / BN + 1);
  if (p.mask_mode == FA_MASK_CAUSAL_WINDOW) {
    const int band_lo = max(0, r_lo - p.window + 1);
    r.b_start = min(band_lo / BN, r.b_end);
    const int g_keys = min(min(p.n_global, r_hi + 1), p.Sk);
    r.a_end = g_keys > 0 ? (g_keys + BN - 1) / BN : 0;
    if (r.a_end >= r.b_start) {  // the two ranges touch: one range [0, b_end)
      r.a_end = 0;
      r.b_start = 0;
    }
  }
  return r;
}

__device__ __forceinline__ int range_count(const Range& r) { return r.a_end + r.b_end - r.b_start; }
__device__ __forceinline__ int range_nb(const Range& r, int t) {
  return t < r.a_end ? t : r.b_start + (t - r.a_end);
}
__device__ __forceinline__ bool range_has(const Range& r, int nb) {
  return nb < r.a_end || (nb >= r.b_start && nb < r.b_end);
}

// Work item t -> (batch*head, query block). Order: groups of `group_heads` heads; inside
// a group, query blocks from the last (most keys under a causal mask) to the first;
// inside that, the heads of the group.
__device__ __forceinline__ void item_coords(int t, const PrefillParams& p, int& bh, int& mb) {
  const int per_group = p.group_heads * p.nmb;
  const int g = t / per_group;
  const int gsize = min(p.group_heads, p.BH - g * p.group_heads);
  const int rem = t - g * per_group;
  mb = p.nmb - 1 - rem / gsize;
  bh = g * p.group_heads + rem % gsize;
}

// Snake assignment of items to persistent CTAs: round r covers items [r*G, r*G+G), walked
// forwards on even rounds and backwards on odd ones.
__device__ __forceinline__ int item_of_round(int r, int G, int cta) {
  return r * G + ((r & 1) ? (G - 1 - cta) : cta);
}

// True when every (row, key) pair of the 128-row tile at m0 and key block nb is in range
// and visible.
template <int BN>
__device__ __forceinline__ bool tile_full(int m0, int nb, const PrefillParams& p) {
  const int n0 = nb * BN, n1 = n0 + BN;
  if (m0 + kTile > p.Sq || n1 > p.Sk) return false;
  if (p.mask_mode == FA_MASK_NONE) return true;
  const int delta = p.Sk - p.Sq;
  const int r_lo = m0 + delta, r_hi = m0 + kTile - 1 + delta;
  if (n1 - 1 > r_lo) return false;
  if (p.mask_mode == FA_MASK_CAUSAL) return true;
  return n1 <= p.n_global || r_hi - max(n0, p.n_global) < p.window;
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The online-softmax step for one S tile, by one thread for its row:
// S (BN FP32 columns at s_col) is loaded from TMEM, masked unless the tile is full,
// the running max is updated, O (D columns at o_col) and l are rescaled when the max
// rose by more than kTau (warp-uniform decision; `before_rescale` makes O safe to touch
// and returns false on abort), and P = 2^(S*sl2 - m) is written over the first BN/2
// columns of S as packed 16-bit pairs. Returns false on abort.
template <int D, int BN, bool BF16, typename PreRescale>
__device__ __forceinline__ bool softmax_tile(uint32_t t_lane, uint32_t s_col, uint32_t o_col,
                                             bool full, int n0, int pos_q,
                                             const PrefillParams& p, float& m_ref, float& l,
                                             PreRescale before_rescale) {
  uint32_t s[BN];
#pragma unroll
  for (int c = 0; c < BN / 64; ++c) tmem_ld64(t_lane + s_col + c * 64, s + c * 64);
  tmem_ld_wait<BN>(s);
  if (!full) {
    int lim = min(pos_q, p.Sk - 1) - n0;
    if (p.mask_mode == FA_MASK_NONE) lim = p.Sk - 1 - n0;
    int lo = INT_MIN, gl = INT_MIN;
    if (p.mask_mode == FA_MASK_CAUSAL_WINDOW) {
      lo = pos_q - p.window + 1 - n0;
      gl = p.n_global - n0;
    }
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      const bool vis = (c <= lim) && (c >= lo || c < gl);
      if (!vis) s[c] = __float_as_uint(-INFINITY);
    }
  }
  // row max: four independent chains of three-input maxima, then combined
  float mx[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) mx[i] = __uint_as_float(s[i]);
#pragma unroll
  for (int c = 4; c < BN; c += 8)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      mx[i] = max3f(mx[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
  const float m_tile = max3f(mx[0], mx[1], fmaxf(mx[2], mx[3])) * p.sl2;
  const float m_new = fmaxf(m_ref, m_tile);
  const bool need = (m_ref != -INFINITY) && (m_new > m_ref + kTau);
  if (m_ref == -INFINITY) m_ref = m_new;
  if (__any_sync(0xffffffffu, need)) {
    if (!before_rescale()) return false;
    const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
    if (need) {
      l *= alpha;
      m_ref = m_new;
    }
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t ov[32];
      tmem_ld32(t_lane + o_col + c * 32, ov);
      tmem_ld_wait<32>(ov);
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
      tmem_st32(t_lane + o_col + c * 32, ov);
    }
  }
  // P = 2^(S*sl2 - m): the exponent argument two lanes at a time, one ex2 per element,
  // the row sum in four packed pairs.
  const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
  const uint64_t scale2 = f2(p.sl2, p.sl2), neg_m2 = f2(-m_use, -m_use);
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int c = 0; c < BN; c += 2) {
    const uint64_t x = f2_fma(f2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), scale2, neg_m2);
    float x0, x1;
    f2_split(x, x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    acc[(c / 2) & 3] = f2_add(acc[(c / 2) & 3], f2(p0, p1));
    s[c / 2] = BF16 ? cvt_pack_bf16(p0, p1) : cvt_pack_f16(p0, p1);
  }
  float a0, a1;
  f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
  l += a0 + a1;
#pragma unroll
  for (int c = 0; c < BN / 64; ++c) tmem_st32(t_lane + s_col + c * 32, s + c * 32);
  tmem_st_wait();
  return true;
}

// Epilogue for one thread's row: O (D columns at o_col) / l rounded to the dtype, and
// LSE = (m + log2 l) ln 2. Rows past Sq are not stored.
template <int D, bool BF16>
__device__ __forceinline__ void store_row(uint32_t t_lane, uint32_t o_col, bool valid,
                                          size_t orow, float m_ref, float l,
                                          const PrefillParams& p) {
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t ov[32];
    tmem_ld32(t_lane + o_col + c * 32, ov);
    tmem_ld_wait<32>(ov);
    if (valid) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l,
                      BF16);
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow * D + c * 32);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
    }
  }
  if (valid && p.lse)
    p.lse[orow] = l > 0.f ? (m_ref + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
}

template <int D>
__device__ __forceinline__ void store_zero_row(size_t orow, const PrefillParams& p) {
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow * D);
  for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
  if (p.lse) p.lse[orow] = -INFINITY;
}

// Wait that ignores the abort flag (used while winding down).
__device__ __forceinline__ void wait_quiet(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  volatile uint32_t zero = 0;
  WaitCtx w2 = wc;
  w2.abort = &zero;
  mbar_wait(bar, parity, w2);
}

// S = Q K^T for one 128-row tile: D/16 MMAs of K = 16, both operands K-major in
// 128-byte-swizzled shared memory (rows of 128 bytes, 8-row groups 1024 bytes apart,
// one region per 64 elements of d).
template <int D, int BN, bool BF16>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t id = idesc_f16(BF16, kTile, BN, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t a = smem_desc_sw128(q_smem + (kk / 4) * (kTile * 128) + (kk % 4) * 32, 16, 1024);
    const uint64_t b = smem_desc_sw128(k_smem + (kk / 4) * (BN * 128) + (kk % 4) * 32, 16, 1024);
    umma_ss(d_tmem, a, b, id, kk > 0);
  }
}

// O (+)= P V: A = P from TMEM (BN/2 packed columns), B = V (BN keys x D) MN-major in
// shared memory: 16 keys per MMA = two 8-row groups (1024 bytes apart), the second
// 64-element half of d one region (BN*128 bytes) further.
template <int D, int BN, bool BF16>
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
  constexpr uint32_t id = idesc_f16(BF16, kTile, D, true);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    const uint64_t b = smem_desc_sw128(v_smem + kk * 16 * 128, BN * 128, 1024);
    umma_ts(o_tmem, p_tmem + kk * 8, b, id, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// ------------------------------------------------------------------ BM = 256 kernel

// Three warpgroups: softmax A, softmax B, and the producers (TMA warp, MMA warp, two idle
// warps). Launched at 168 registers per thread (384 x 168 = 64,512); the producer group
// gives registers up so that the softmax groups can hold a whole S row:
// 128 x (200 + 200 + 104) = 64,512.
constexpr int kThreads256 = 384;
constexpr int kTmaWarp256 = 8;
constexpr int kMmaWarp256 = 9;
constexpr uint32_t kRegsSoftmax = 200;
constexpr uint32_t kRegsProducer = 104;

template <int D, int BN>
struct Cfg256 {
  static constexpr int KCH = D / 64;
  static constexpr int QT_BYTES = kTile * D * 2;     // one 128-row Q tile
  static constexpr int Q_BYTES = 2 * QT_BYTES;
  static constexpr int TILE_BYTES = BN * D * 2;      // one K or V tile
  static constexpr int BAR_BYTES = 1024;
  static constexpr int NSLOT_FIT = (int)((kSmemLimit - 1024 - BAR_BYTES - Q_BYTES) / TILE_BYTES);
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;
  static constexpr int SMEM = 1024 + Q_BYTES + NSLOT * TILE_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN + 2 * D);
  static_assert(NSLOT >= 2, "shared memory ring too small");
  static_assert(SMEM <= (int)kSmemLimit, "shared memory over budget");
  static_assert(2 * BN + 2 * D <= 512, "TMEM over budget");
};

struct Bars256 {
  uint64_t full[8], empty[8];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2], o_empty[2];
  uint64_t final_mma;
  uint32_t tmem_base;
  uint32_t abort;
};

template <int D, int BN, bool BF16>
__global__ void __launch_bounds__(kThreads256, 1)
    prefill_bm256_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = Cfg256<D, BN>;
  constexpr int BM = 2 * kTile;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base;  // Q_A then Q_B
  const uint32_t sRing = base + C::Q_BYTES;
  Bars256* bars = reinterpret_cast<Bars256*>(smem + C::Q_BYTES + C::NSLOT * C::TILE_BYTES);
  auto B = [&](uint64_t& b) { return smem_u32(&b); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(B(bars->full[i]), 1);
      mbar_init(B(bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B(bars->q_full[i]), 1);
      mbar_init(B(bars->q_empty[i]), 1);
      mbar_init(B(bars->s_full[i]), 1);
      mbar_init(B(bars->p_full[i]), 128);
      mbar_init(B(bars->pv_done[i]), 1);
      mbar_init(B(bars->o_empty[i]), 128);
    }
    mbar_init(B(bars->final_mma), 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kTmaWarp256 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx wc{&bars->abort, p.status, p.timeout_ns};
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  // The role branches never rejoin: each ends with the CTA-wide teardown barrier, so no
  // code runs under two different register budgets.
  if (warp >= 8) {
    regs_decrease<kRegsProducer>();
    if (warp == kTmaWarp256) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pos = 0, ii = 0;
      uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      uint32_t qfills[2] = {0, 0};
      bool ok = true;
      for (int r = 0; ok && r * G < p.total_items; ++r) {
        const int t = item_of_round(r, G, cta);
        if (t >= p.total_items) continue;
        int bh, mb;
        item_coords(t, p, bh, mb);
        const Range rg = key_range<BN>(mb * BM, min(mb * BM + BM, p.Sq), p);
        const int n = range_count(rg);
        if (n == 0) continue;
        for (int q = 0; q < 2 && ok; ++q) {
          if (ii > 0 && !(ok = mbar_wait(B(bars->q_empty[q]), (ii - 1) & 1, wc))) break;
          mbar_arrive_expect_tx(B(bars->q_full[q]), C::QT_BYTES);
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(sQ + q * C::QT_BYTES + c * (kTile * 128), &tmQ, B(bars->q_full[q]),
                        c * 64, mb * BM + q * kTile, bh);
          qfills[q] = ii + 1;
        }
        for (int s = 0; s < 2 * n && ok; ++s) {  // K0, V0, K1, V1, ...
          const int slot = pos % C::NSLOT;
          const uint32_t use = pos / C::NSLOT;
          if (!(ok = mbar_wait(B(bars->empty[slot]), (use & 1) ^ 1, wc))) break;
          const uint32_t dst = sRing + slot * C::TILE_BYTES;
          mbar_arrive_expect_tx(B(bars->full[slot]), C::TILE_BYTES);
          const int n0 = range_nb(rg, s / 2) * BN;
          const void* map = (s & 1) ? (const void*)&tmV : (const void*)&tmK;
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(dst + c * (BN * 128), map, B(bars->full[slot]), c * 64, n0, bh);
          fills[slot] = use + 1;
          ++pos;
        }
        ++ii;
      }
      if (!ok) {  // wind down: every load this thread issued lands before the CTA exits
        for (int s = 0; s < C::NSLOT; ++s)
          if (fills[s] > 0) wait_quiet(B(bars->full[s]), (fills[s] - 1) & 1, wc);
        for (int q = 0; q < 2; ++q)
          if (qfills[q] > 0) wait_quiet(B(bars->q_full[q]), (qfills[q] - 1) & 1, wc);
      }
    }
    __syncwarp();
    } else if (warp == kMmaWarp256) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t tS[2] = {tmem, tmem + BN};
      const uint32_t tO[2] = {tmem + 2 * BN, tmem + 2 * BN + D};
      uint32_t pos = 0, ii = 0, tc = 0;
      bool ok = true;
      for (int r = 0; ok && r * G < p.total_items; ++r) {
        const int t = item_of_round(r, G, cta);
        if (t >= p.total_items) continue;
        int bh, mb;
        item_coords(t, p, bh, mb);
        const Range rg = key_range<BN>(mb * BM, min(mb * BM + BM, p.Sq), p);
        const int n = range_count(rg);
        if (n == 0) continue;
        {  // S_A(0), S_B(0) with K0
          const int slot = pos % C::NSLOT;
          if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
          for (int q = 0; q < 2 && ok; ++q) {
            if (!(ok = mbar_wait(B(bars->q_full[q]), ii & 1, wc))) break;
            tc_fence_after();
            issue_qk<D, BN, BF16>(tS[q], sQ + q * C::QT_BYTES, sRing + slot * C::TILE_BYTES);
            umma_commit(B(bars->s_full[q]));
            if (n == 1) umma_commit(B(bars->q_empty[q]));
          }
          if (!ok) break;
          umma_commit(B(bars->empty[slot]));
          ++pos;
        }
        for (int j = 0; j < n && ok; ++j) {
          const int vslot = pos % C::NSLOT;
          const int kslot = (pos + 1) % C::NSLOT;
          if (!(ok = mbar_wait(B(bars->full[vslot]), (pos / C::NSLOT) & 1, wc))) break;
          tc_fence_after();
          for (int q = 0; q < 2 && ok; ++q) {
            if (!(ok = mbar_wait(B(bars->p_full[q]), tc & 1, wc))) break;
            tc_fence_after();
            if (j == 0 && ii > 0) {  // this tile's epilogue of the previous item has read O
              if (!(ok = mbar_wait(B(bars->o_empty[q]), (ii - 1) & 1, wc))) break;
              tc_fence_after();
            }
            issue_pv<D, BN, BF16>(tO[q], tS[q], sRing + vslot * C::TILE_BYTES, j > 0);
            if (j == n - 1) umma_commit(B(bars->pv_done[q]));
            if (q == 1) umma_commit(B(bars->empty[vslot]));
            if (j + 1 < n) {  // S(j+1) overwrites P(j) only after PV(j) in the pipe
              if (q == 0) {
                if (!(ok = mbar_wait(B(bars->full[kslot]), ((pos + 1) / C::NSLOT) & 1, wc))) break;
                tc_fence_after();
              }
              issue_qk<D, BN, BF16>(tS[q], sQ + q * C::QT_BYTES, sRing + kslot * C::TILE_BYTES);
              umma_commit(B(bars->s_full[q]));
              if (j + 2 == n) umma_commit(B(bars->q_empty[q]));
              if (q == 1) umma_commit(B(bars->empty[kslot]));
            }
          }
          pos += (j + 1 < n) ? 2 : 1;
          ++tc;
        }
        ++ii;
      }
      umma_commit(B(bars->final_mma));  // all MMAs done before TMEM is released
      wait_quiet(B(bars->final_mma), 0, wc);
    }
    __syncwarp();
    }
    tc_fence_before();
    __syncthreads();  // teardown: every role is done with TMEM and shared memory
    return;
  } else {
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax, tiles A / B
    const int q = warp / 4;        // 0: tile A, 1: tile B
    const int row = (warp % 4) * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const uint32_t s_col = q * BN, o_col = 2 * BN + q * D;
    const int delta = p.Sk - p.Sq;
    uint32_t ii = 0, tc = 0;
    bool ok = true;
    for (int r = 0; ok && r * G < p.total_items; ++r) {
      const int t = item_of_round(r, G, cta);
      if (t >= p.total_items) continue;
      int bh, mb;
      item_coords(t, p, bh, mb);
      const Range rg = key_range<BN>(mb * BM, min(mb * BM + BM, p.Sq), p);
      const int n = range_count(rg);
      const int m0 = mb * BM + q * kTile;  // first row of this tile
      const int qrow = m0 + row;
      const size_t orow = static_cast<size_t>(bh) * p.Sq + qrow;
      if (n == 0) {  // nothing visible for any row of the item
        if (qrow < p.Sq) store_zero_row<D>(orow, p);
        continue;
      }
      const Range mine = key_range<BN>(m0, min(m0 + kTile, p.Sq), p);
      const int pos_q = qrow + delta;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        const int nb = range_nb(rg, j);
        const bool full = tile_full<BN>(m0, nb, p);
        ok = mbar_wait(B(bars->s_full[q]), tc & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (p.trace && row == 0 && range_has(mine, nb))
          atomicAdd(p.trace + (static_cast<size_t>(bh) * ((p.Sq + kTile - 1) / kTile) +
                               m0 / kTile) * p.nnb + nb,
                    16 + (full ? 2 : 1));
        // S(j) was issued after PV(j-1), so O needs no wait before a rescale
        ok = softmax_tile<D, BN, BF16>(t_lane, s_col, o_col, full, nb * BN, pos_q, p, m_ref, l,
                                       [] { return true; });
        tc_fence_before();
        mbar_arrive(B(bars->p_full[q]));
        ++tc;
      }
      if (!ok) break;
      ok = mbar_wait(B(bars->pv_done[q]), ii & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      store_row<D, BF16>(t_lane, o_col, qrow < p.Sq, orow, m_ref, l, p);
      tc_fence_before();
      mbar_arrive(B(bars->o_empty[q]));
      ++ii;
    }
    tc_fence_before();
    __syncthreads();  // teardown: every role is done with TMEM and shared memory
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  }
}

// ------------------------------------------------------------------ BM = 128 kernel

constexpr int kThreads128 = 192;
constexpr int kTmaWarp128 = 4;
constexpr int kMmaWarp128 = 5;

template <int D, int BN>
struct Cfg128 {
  static constexpr int KCH = D / 64;
  static constexpr int Q_BYTES = kTile * D * 2;
  static constexpr int TILE_BYTES = BN * D * 2;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int NSLOT_FIT = (int)((kSmemLimit - 1024 - BAR_BYTES - Q_BYTES) / TILE_BYTES);
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;
  static constexpr int SMEM = 1024 + Q_BYTES + NSLOT * TILE_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN + D);
  static constexpr int O_COL = 2 * BN;
  static_assert(NSLOT >= 2, "shared memory ring too small");
  static_assert(SMEM <= (int)kSmemLimit, "shared memory over budget");
};

struct Bars128 {
  uint64_t full[8], empty[8];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_empty, final_mma;
  uint32_t tmem_base;
  uint32_t abort;
};

template <int D, int BN, bool BF16>
__global__ void __launch_bounds__(kThreads128, 1)
    prefill_bm128_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = Cfg128<D, BN>;
  constexpr int BM = kTile;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sRing = base + C::Q_BYTES;
  Bars128* bars = reinterpret_cast<Bars128*>(smem + C::Q_BYTES + C::NSLOT * C::TILE_BYTES);
  auto B = [&](uint64_t& b) { return smem_u32(&b); };

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(B(bars->full[i]), 1);
      mbar_init(B(bars->empty[i]), 1);
    }
    mbar_init(B(bars->q_full), 1);
    mbar_init(B(bars->q_empty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(B(bars->s_full[i]), 1);
      mbar_init(B(bars->p_full[i]), 128);
      mbar_init(B(bars->pv_done[i]), 1);
    }
    mbar_init(B(bars->o_empty), 128);
    mbar_init(B(bars->final_mma), 1);
    bars->abort = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == kTmaWarp128 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtx wc{&bars->abort, p.status, p.timeout_ns};
  const int G = gridDim.x;
  const int cta = blockIdx.x;

  if (warp == kTmaWarp128) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pos = 0, ii = 0, qfill = 0;
      uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      bool ok = true;
      for (int r = 0; ok && r * G < p.total_items; ++r) {
        const int t = item_of_round(r, G, cta);
        if (t >= p.total_items) continue;
        int bh, mb;
        item_coords(t, p, bh, mb);
        const Range rg = key_range<BN>(mb * BM, min(mb * BM + BM, p.Sq), p);
        const int n = range_count(rg);
        if (n == 0) continue;
        if (ii > 0 && !(ok = mbar_wait(B(bars->q_empty), (ii - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(B(bars->q_full), C::Q_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sQ + c * (kTile * 128), &tmQ, B(bars->q_full), c * 64, mb * BM, bh);
        qfill = ii + 1;
        // consumption order: K0, then for each j: K(j+1) (if any), V(j)
        for (int s = 0; s < 2 * n && ok; ++s) {
          int tile, is_v;
          if (s == 0) {
            tile = 0;
            is_v = 0;
          } else if (s == 2 * n - 1) {
            tile = n - 1;
            is_v = 1;
          } else {
            const int j = (s - 1) / 2;
            is_v = (s - 1) & 1;
            tile = is_v ? j : j + 1;
          }
          const int slot = pos % C::NSLOT;
          const uint32_t use = pos / C::NSLOT;
          if (!(ok = mbar_wait(B(bars->empty[slot]), (use & 1) ^ 1, wc))) break;
          const uint32_t dst = sRing + slot * C::TILE_BYTES;
          mbar_arrive_expect_tx(B(bars->full[slot]), C::TILE_BYTES);
          const int n0 = range_nb(rg, tile) * BN;
          const void* map = is_v ? (const void*)&tmV : (const void*)&tmK;
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(dst + c * (BN * 128), map, B(bars->full[slot]), c * 64, n0, bh);
          fills[slot] = use + 1;
          ++pos;
        }
        ++ii;
      }
      if (!ok) {
        for (int s = 0; s < C::NSLOT; ++s)
          if (fills[s] > 0) wait_quiet(B(bars->full[s]), (fills[s] - 1) & 1, wc);
        if (qfill > 0) wait_quiet(B(bars->q_full), (qfill - 1) & 1, wc);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp128) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t pos = 0, ii = 0, tc = 0;
      bool ok = true;
      for (int r = 0; ok && r * G < p.total_items; ++r) {
        const int t = item_of_round(r, G, cta);
        if (t >= p.total_items) continue;
        int bh, mb;
        item_coords(t, p, bh, mb);
        const Range rg = key_range<BN>(mb * BM, min(mb * BM + BM, p.Sq), p);
        const int n = range_count(rg);
        if (n == 0) continue;
        if (!(ok = mbar_wait(B(bars->q_full), ii & 1, wc))) break;
        tc_fence_after();
        {  // S_0
          const int slot = pos % C::NSLOT;
          if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
          tc_fence_after();
          issue_qk<D, BN, BF16>(tmem + (tc & 1) * BN, sQ, sRing + slot * C::TILE_BYTES);
          umma_commit(B(bars->s_full[tc & 1]));
          umma_commit(B(bars->empty[slot]));
          ++pos;
          if (n == 1) umma_commit(B(bars->q_empty));
        }
        for (int j = 0; j < n && ok; ++j) {
          if (j + 1 < n) {  // S_{j+1} into the other buffer while softmax works on S_j
            const int slot = pos % C::NSLOT;
            if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
            tc_fence_after();
            issue_qk<D, BN, BF16>(tmem + ((tc + 1) & 1) * BN, sQ, sRing + slot * C::TILE_BYTES);
            umma_commit(B(bars->s_full[(tc + 1) & 1]));
            umma_commit(B(bars->empty[slot]));
            ++pos;
            if (j + 2 == n) umma_commit(B(bars->q_empty));
          }
          if (!(ok = mbar_wait(B(bars->p_full[tc & 1]), (tc >> 1) & 1, wc))) break;
          tc_fence_after();
          if (j == 0 && ii > 0) {  // the previous item's epilogue has read O
            if (!(ok = mbar_wait(B(bars->o_empty), (ii - 1) & 1, wc))) break;
            tc_fence_after();
          }
          const int slot = pos % C::NSLOT;
          if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
          tc_fence_after();
          issue_pv<D, BN, BF16>(tmem + C::O_COL, tmem + (tc & 1) * BN,
                                sRing + slot * C::TILE_BYTES, j > 0);
          umma_commit(B(bars->pv_done[tc & 1]));
          umma_commit(B(bars->empty[slot]));
          ++pos;
          ++tc;
        }
        ++ii;
      }
      umma_commit(B(bars->final_mma));
      wait_quiet(B(bars->final_mma), 0, wc);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int row = warp * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int delta = p.Sk - p.Sq;
    uint32_t ii = 0, tc = 0;
    bool ok = true;
    for (int r = 0; ok && r * G < p.total_items; ++r) {
      const int t = item_of_round(r, G, cta);
      if (t >= p.total_items) continue;
      int bh, mb;
      item_coords(t, p, bh, mb);
      const Range rg = key_range<BN>(mb * BM, min(mb * BM + BM, p.Sq), p);
      const int n = range_count(rg);
      const int m0 = mb * BM;
      const int qrow = m0 + row;
      const size_t orow = static_cast<size_t>(bh) * p.Sq + qrow;
      if (n == 0) {
        if (qrow < p.Sq) store_zero_row<D>(orow, p);
        continue;
      }
      const int pos_q = qrow + delta;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j) {
        const int nb = range_nb(rg, j);
        const bool full = tile_full<BN>(m0, nb, p);
        ok = mbar_wait(B(bars->s_full[tc & 1]), (tc >> 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (p.trace && row == 0)
          atomicAdd(p.trace + (static_cast<size_t>(bh) * p.nmb + mb) * p.nnb + nb,
                    16 + (full ? 2 : 1));
        // O must hold every earlier P.V product before it is rescaled
        const uint32_t pc = tc - 1;
        auto wait_pv = [&]() {
          bool w = mbar_wait(B(bars->pv_done[pc & 1]), (pc >> 1) & 1, wc);
          w = __all_sync(0xffffffffu, w);
          if (w) tc_fence_after();
          return w;
        };
        ok = softmax_tile<D, BN, BF16>(t_lane, (tc & 1) * BN, C::O_COL, full, nb * BN, pos_q, p,
                                       m_ref, l, wait_pv);
        if (!ok) break;
        tc_fence_before();
        mbar_arrive(B(bars->p_full[tc & 1]));
        ++tc;
      }
      if (!ok) break;
      {
        const uint32_t pc = tc - 1;
        ok = mbar_wait(B(bars->pv_done[pc & 1]), (pc >> 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      tc_fence_after();
      store_row<D, BF16>(t_lane, C::O_COL, qrow < p.Sq, orow, m_ref, l, p);
      tc_fence_before();
      mbar_arrive(B(bars->o_empty));
      ++ii;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, int BN, bool BF16>
cudaError_t launch_t(const PrefillLaunch& L, int BM, cudaStream_t stream) {
  if (BM == 256) {
    auto kern = prefill_bm256_kernel<D, BN, BF16>;
    constexpr int smem = Cfg256<D, BN>::SMEM;
    // setmaxnreg.inc can only hand out registers the CTA was launched with; a build whose
    // launch register count is below the split would make the softmax warps wait forever,
    // so such a build is refused here instead of launched.
    cudaFuncAttributes fattr;
    cudaError_t e = cudaFuncGetAttributes(&fattr, kern);
    if (e != cudaSuccess) return e;
    if (fattr.numRegs * kThreads256 < 128 * static_cast<int>(2 * kRegsSoftmax + kRegsProducer))
      return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<L.grid, kThreads256, smem, stream>>>(L.tmQ, L.tmK, L.tmV, L.p);
  } else {
    auto kern = prefill_bm128_kernel<D, BN, BF16>;
    constexpr int smem = Cfg128<D, BN>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<L.grid, kThreads128, smem, stream>>>(L.tmQ, L.tmK, L.tmV, L.p);
  }
  return cudaGetLastError();
}

}  // namespace

int prefill_tile_rows() { return kTile; }

cudaError_t launch_prefill(const PrefillLaunch& L, int D, int BN, int BM, bool bf16,
                           cudaStream_t stream) {
  if (BM != 128 && BM != 256) return cudaErrorInvalidValue;
#define FA_CASE(d_, bn_, bf_) \
  if (D == d_ && BN == bn_ && bf16 == bf_) return launch_t<d_, bn_, bf_>(L, BM, stream);
  FA_CASE(64, 64, false)
  FA_CASE(64, 64, true)
  FA_CASE(64, 128, false)
  FA_CASE(64, 128, true)
  FA_CASE(128, 64, false)
  FA_CASE(128, 64, true)
  FA_CASE(128, 128, false)
  FA_CASE(128, 128, true)
#undef FA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fa
