// FlashAttention forward (prefill) for sm_103a: tcgen05 MMAs with TMEM accumulators,
// TMA tile loads into a shared-memory ring, warp-specialised online softmax, tile
// skipping for causal, sliding-window(+global), band and prefix-LM masks, and a persistent
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
// prefill_bm128_kernel (the band and block-sparse masks, or block_m = 128): a work item is
//   128 query rows of one (batch, head).
//   warps 0-7   softmax: two warpgroups, each owning half of every score row (TMEM lane =
//               row); partial row maxima are swapped through shared memory; P (16-bit)
//               overwrites S in TMEM; lazy rescale of O.
//   warps 8-11  epilogue: O / l and LSE of the previous item from the second O buffer.
//   warp 12     TMA producer: Q (double buffered), then K(0), and per tile K(t+1), V(t)
//               through a ring of shared-memory slots.
//   warp 13     MMA issuer (one elected lane): S(t+1) = Q K(t+1)^T, then O += P(t) V(t).
//   TMEM columns: S0 [0,BN), S1 [BN,2BN), O0 [2BN,2BN+D), O1 [2BN+D,2BN+2D).
//
// prefill_bm256_kernel (default for the other masks): a work item is 256 query rows held
// as two 128-row tiles A and B that share every K/V tile; one softmax warpgroup per tile (a
// whole row per thread, which also writes the epilogue), a TMA warp and an MMA warp.
// Tensor-pipe order
//   S_A(0) S_B(0) | PV_A(0) S_A(1) | PV_B(0) S_B(1) | ...
// so that one tile's softmax runs while the tensor core works for the other.
//   TMEM columns: S_A [0,BN), S_B [BN,2BN), O_A [2BN,2BN+D), O_B [2BN+D,2BN+2D).
//   Its SPLIT build (FP32 inputs, fa_prefill_split.cu) reads bf16 high and low planes of
//   Q, K, V and forms each product from both parts.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <type_traits>

#include "fa_internal.h"
#include "fa_plan.h"
#include "fa_ptx.cuh"
#include "fa_mma.cuh"

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

// Block-sparse: the layout byte of the 128-row query tile at m0 and the 128 keys holding
// key block nb, for (batch, head) bh.
template <int BN>
__device__ __forceinline__ bool layout_bit(int bh, int m0, int nb, const PrefillParams& p) {
  const size_t row = static_cast<size_t>(bh % p.H) * p.lnqb + m0 / kTile;
  return p.layout[row * p.lnkb + (nb * BN) / 128] != 0;
}

// True when every (row, key) pair of the 128-row tile at m0 and key block nb is in range
// and visible.
template <int BN, bool SPARSE, int TM = kTile>
__device__ __forceinline__ bool tile_full(int m0, int nb, int sk, int bh,
                                          const PrefillParams& p) {
  const int n0 = nb * BN, n1 = n0 + BN;
  if (m0 + TM > p.Sq || n1 > sk) return false;
  if constexpr (SPARSE) return layout_bit<BN>(bh, m0, nb, p);
  if (p.mask_mode == FA_MASK_NONE) return true;
  const int delta = sk - p.Sq;
  const int r_lo = m0 + delta, r_hi = m0 + TM - 1 + delta;
  if (p.mask_mode == FA_MASK_BAND)  // the largest |pos - j| of the tile is within w
    return static_cast<long long>(r_hi) - n0 <= p.window &&
           static_cast<long long>(n1 - 1) - r_lo <= p.window;
  if (p.mask_mode == FA_MASK_PREFIX_LM) return n1 <= p.n_global || n1 - 1 <= r_lo;
  if (n1 - 1 > r_lo) return false;
  if (p.mask_mode == FA_MASK_CAUSAL) return true;
  return n1 <= p.n_global || r_hi - max(n0, p.n_global) < p.window;
}

// The key blocks visited by query rows [m0, m1). The kernels are built twice: block-sparse
// (a scan of the layout rows, SparseRange) and every other mask (closed-form Range).
template <bool SPARSE>
__device__ __forceinline__ auto item_range(int m0, int m1, int BN, int sk, const PrefillParams& p,
                                           int bh) {
  if constexpr (SPARSE)
    return key_range_sparse(m0, m1, BN, sk, p, bh);
  else
    return key_range(m0, m1, BN, sk, p, bh);
}

__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16) {
  if (bf16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// The online-softmax step for one S tile, by one thread for NC columns of its row:
// S (NC FP32 columns at s_col, keys n0..n0+NC-1) is loaded from TMEM and masked unless
// the tile is full; `exchange` turns this thread's partial row maximum into the maximum
// of the whole row (identity when NC covers the row); the running max is updated; O (ON
// columns at o_col) and l are rescaled when the max rose by more than kTau (warp-uniform
// decision; `before_rescale` makes O safe to touch and returns false on abort); and
// P = 2^(S*sl2 - m) is written as packed 16-bit pairs to NC/2 columns at p_col.
// SPLIT (FP32 inputs): P is written as two bf16 parts, P_hi = bf16(P) at p_col and
// P_lo = bf16(P - P_hi) at p_col + NC/2, so that P_hi + P_lo holds P to 2^-16.
// l accumulates the sum over this thread's NC columns. With p.rescales set, the rows
// rescaled are counted for the 128-row tile (rs_bh, rs_m0) when rs_bh >= 0. P_SMEM (the
// 64-row kernel): P goes instead to row p_row of a 64-row, 128-byte-swizzled K-major tile
// at shared address p_col (regions of 64 keys 8 KB apart), when p_row >= 0, followed by a
// proxy fence so that the tensor core sees it. Returns false on abort.
template <int NC, int ON, bool BF16, bool SPLIT, bool P_SMEM = false, typename Exchange,
          typename PreRescale>
__device__ __forceinline__ bool softmax_cols(uint32_t t_lane, uint32_t s_col, uint32_t p_col,
                                             uint32_t o_col, bool full, int n0, int pos_q,
                                             int sk, const PrefillParams& p, float& m_ref,
                                             float& l, Exchange exchange,
                                             PreRescale before_rescale, int rs_bh, int rs_m0,
                                             int p_row = -1) {
  static_assert(NC == 32 || NC % 64 == 0, "column count");
  static_assert(!SPLIT || (BF16 && NC % 64 == 0), "split P: bf16, 64-column groups");
  uint32_t s[NC];
  uint32_t lo[SPLIT ? NC / 2 : 1];
  if constexpr (NC == 32) {
    tmem_ld32(t_lane + s_col, s);
  } else {
#pragma unroll
    for (int c = 0; c < NC / 64; ++c) tmem_ld64(t_lane + s_col + c * 64, s + c * 64);
  }
  tmem_ld_wait<NC>(s);
  if (!full) {
    int lim = min(pos_q, sk - 1) - n0;
    if (p.mask_mode == FA_MASK_NONE || p.mask_mode == FA_MASK_BLOCK_SPARSE) lim = sk - 1 - n0;
    int lo = INT_MIN, gl = INT_MIN;
    if (p.mask_mode == FA_MASK_CAUSAL_WINDOW) {
      lo = pos_q - p.window + 1 - n0;
      gl = p.n_global - n0;
    } else if (p.mask_mode == FA_MASK_BAND) {  // |pos - j| <= w, in 64 bits: w may be huge
      const long long hi = static_cast<long long>(pos_q) + p.window;
      lim = static_cast<int>((hi < sk - 1 ? hi : sk - 1) - n0);
      const long long l0 = static_cast<long long>(pos_q) - p.window - n0;
      lo = l0 < INT_MIN ? INT_MIN : static_cast<int>(l0);
    } else if (p.mask_mode == FA_MASK_PREFIX_LM) {
      lim = min(max(pos_q, p.n_global - 1), sk - 1) - n0;
    }
    // per 32 columns, a bit mask of the visible ones: c <= lim and (c >= lo or c < gl)
    lim = max(lim, -1);
    lo = max(lo, -1);
    gl = max(gl, 0);
#pragma unroll
    for (int k = 0; k < NC / 32; ++k) {
      const int b = lim - 32 * k, a = lo - 32 * k, g = gl - 32 * k;
      const uint32_t upto = b < 0 ? 0u : (b >= 31 ? 0xffffffffu : (2u << b) - 1u);
      const uint32_t from = a <= 0 ? 0xffffffffu : (a >= 32 ? 0u : ~((1u << a) - 1u));
      const uint32_t below = g <= 0 ? 0u : (g >= 32 ? 0xffffffffu : (1u << g) - 1u);
      const uint32_t mk = upto & (from | below);
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (!((mk >> c) & 1u)) s[32 * k + c] = __float_as_uint(-INFINITY);
    }
  }
  // partial row max: four independent chains of three-input maxima, then combined
  // (columns 0-7 seed the chains; each later group of 8 adds two columns per chain)
  float mx[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) mx[i] = fmaxf(__uint_as_float(s[2 * i]), __uint_as_float(s[2 * i + 1]));
#pragma unroll
  for (int c = 8; c < NC; c += 8)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      mx[i] = max3f(mx[i], __uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1]));
  const float m_tile = exchange(max3f(mx[0], mx[1], fmaxf(mx[2], mx[3]))) * p.sl2;
  const float m_new = fmaxf(m_ref, m_tile);
  const bool need = (m_ref != -INFINITY) && (m_new > m_ref + kTau);
  if (m_ref == -INFINITY) m_ref = m_new;
  if (__any_sync(0xffffffffu, need)) {
    if (p.rescales) {  // debug count: one atomic per warp (the ballot is warp-wide)
      const uint32_t who = __ballot_sync(0xffffffffu, need && rs_bh >= 0);
      if ((threadIdx.x & 31) == 0 && who != 0u && rs_bh >= 0)
        atomicAdd(p.rescales + static_cast<size_t>(rs_bh) * ((p.Sq + kTile - 1) / kTile) +
                      rs_m0 / kTile,
                  __popc(who));
    }
    if (!before_rescale()) return false;
    const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
    if (need) {
      l *= alpha;
      m_ref = m_new;
    }
#pragma unroll 1
    for (int c = 0; c < ON / 32; ++c) {
      uint32_t ov[32];
      tmem_ld32(t_lane + o_col + c * 32, ov);
      tmem_ld_wait<32>(ov);
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
      tmem_st32(t_lane + o_col + c * 32, ov);
    }
  }
  // P = 2^(S*sl2 - m): the exponent argument two lanes at a time, one exponential per
  // element (masked -inf entries give 0), the row sum in four packed pairs.
  const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
  const uint64_t scale2 = f2(p.sl2, p.sl2), neg_m2 = f2(-m_use, -m_use);
  uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
  for (int c = 0; c < NC; c += 2) {
    const uint64_t x =
        f2_fma(f2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), scale2, neg_m2);
    float x0, x1;
    f2_split(x, x0, x1);
    const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
    acc[(c / 2) & 3] = f2_add(acc[(c / 2) & 3], f2(p0, p1));
    const uint32_t hi = BF16 ? cvt_pack_bf16(p0, p1) : cvt_pack_f16(p0, p1);
    s[c / 2] = hi;
    if constexpr (SPLIT)  // residuals against the bf16 values (low half: p0)
      lo[c / 2] = cvt_pack_bf16(p0 - __uint_as_float(hi << 16),
                                p1 - __uint_as_float(hi & 0xffff0000u));
  }
  float a0, a1;
  f2_split(f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3])), a0, a1);
  l += a0 + a1;
  if constexpr (P_SMEM) {
    if (p_row >= 0) {
#pragma unroll
      for (int k = 0; k < NC / 8; ++k)  // 16-byte chunk k holds keys 8k .. 8k+7
        st_shared_v4(p_col + (k / 8) * (64 * 128) + p_row * 128 +
                         ((static_cast<uint32_t>(k % 8) ^ (p_row & 7)) << 4),
                     s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
    }
    fence_proxy_async_smem();
    tmem_st_wait();  // a rescale of O above must land before the next P.V reads it
    return true;
  }
  if constexpr (NC == 32) {
    tmem_st16(t_lane + p_col, s);
  } else {
#pragma unroll
    for (int c = 0; c < NC / 64; ++c) tmem_st32(t_lane + p_col + c * 32, s + c * 32);
  }
  if constexpr (SPLIT) {
#pragma unroll
    for (int c = 0; c < NC / 64; ++c) tmem_st32(t_lane + p_col + NC / 2 + c * 32, lo + c * 32);
  }
  tmem_st_wait();
  return true;
}

// A whole row per thread.
template <int D, int BN, bool BF16, bool SPLIT, typename PreRescale>
__device__ __forceinline__ bool softmax_tile(uint32_t t_lane, uint32_t s_col, uint32_t o_col,
                                             bool full, int n0, int pos_q, int sk,
                                             const PrefillParams& p, float& m_ref, float& l,
                                             PreRescale before_rescale, int rs_bh, int rs_m0) {
  return softmax_cols<BN, D, BF16, SPLIT>(t_lane, s_col, s_col, o_col, full, n0, pos_q, sk,
                                          p, m_ref, l, [](float m) { return m; },
                                          before_rescale, rs_bh, rs_m0);
}

// Epilogue for one thread's row: O (D columns at o_col) / l rounded to the dtype (FP32
// when OUT_F32), and LSE = (m + log2 l) ln 2. Rows past Sq are not stored.
template <int D, bool BF16, bool OUT_F32 = false>
__device__ __forceinline__ void store_row(uint32_t t_lane, uint32_t o_col, bool valid,
                                          size_t orow, float m_ref, float l,
                                          const PrefillParams& p) {
  const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t ov[32];
    tmem_ld32(t_lane + o_col + c * 32, ov);
    tmem_ld_wait<32>(ov);
    // 32-byte stores when O is 32-byte aligned (a row's chunk of 32 columns then starts on a
    // 32-byte boundary too), else 16-byte ones; the choice is the same for the whole launch
    const bool wide = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
    if (OUT_F32 && valid) {
#pragma unroll
      for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * inv_l);
      float* dst = static_cast<float*>(p.o) + orow * D + c * 32;
      if (wide) {
#pragma unroll
        for (int e = 0; e < 4; ++e) st_global_v8(dst + 8 * e, ov + 8 * e);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          reinterpret_cast<uint4*>(dst)[e] =
              make_uint4(ov[4 * e], ov[4 * e + 1], ov[4 * e + 2], ov[4 * e + 3]);
      }
    } else if (valid) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        pk[e] = pack2(__uint_as_float(ov[2 * e]) * inv_l, __uint_as_float(ov[2 * e + 1]) * inv_l,
                      BF16);
      uint16_t* dst = static_cast<uint16_t*>(p.o) + orow * D + c * 32;
      if (wide) {
        st_global_v8(dst, pk);
        st_global_v8(dst + 16, pk + 8);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          reinterpret_cast<uint4*>(dst)[e] =
              make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
    }
  }
  if (valid && p.lse)
    p.lse[orow] = l > 0.f ? (m_ref + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
}

template <int D, bool OUT_F32 = false>
__device__ __forceinline__ void store_zero_row(size_t orow, const PrefillParams& p) {
  constexpr int ESZ = OUT_F32 ? 4 : 2;  // bytes per element
  uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.o) + orow * D * ESZ);
  for (int c = 0; c < D * ESZ / 16; ++c) dst[c] = make_uint4(0, 0, 0, 0);
  if (p.lse) p.lse[orow] = -INFINITY;
}

// Keys of (batch, head) bh: Sk for contiguous K/V; the sequence's own length (clamped
// to the table's capacity) for a paged cache.
__device__ __forceinline__ int item_sk(const PrefillParams& p, int bh) {
  if (!p.block_table) return p.Sk;
  const int c = p.seq_k[bh / p.H];
  return c < 0 ? 0 : (c > p.Sk ? p.Sk : c);
}

// TMA coordinates (row y, plane z) of the BN-key K/V tile at key n0 of (batch, head) bh:
// (n0, bh) for contiguous K/V; for a paged cache the tile's rows lie in one page, at
// (offset in the page, physical page * H + head). A table entry out of range is reported
// (by `report` lanes) and page 0 is read instead.
__device__ __forceinline__ void kv_tile_coords(const PrefillParams& p, int bh, int n0, bool report,
                                               int& y, int& z) {
  y = n0;
  z = bh;
  if (!p.block_table) return;
  const int b = bh / p.H, lp = n0 / p.page_size;
  int phys = p.block_table[static_cast<size_t>(b) * p.max_pages + lp];
  if (phys < 0 || phys >= p.num_pages) {
    if (report) atomicOr(p.status, FA_DEV_BAD_PAGE);
    phys = 0;
  }
  y = n0 - lp * p.page_size;
  z = phys * p.H + (bh - b * p.H);
}

// Wait that ignores the abort flag (used while winding down).
__device__ __forceinline__ void wait_quiet(uint32_t bar, uint32_t parity, const WaitCtx& wc) {
  volatile uint32_t zero = 0;
  WaitCtx w2 = wc;
  w2.abort = &zero;
  mbar_wait(bar, parity, w2);
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

// SPLIT (FP32 inputs): every Q, K and V tile is held as two bf16 planes, the high parts
// then the low parts.
template <int D, int BN, bool SPLIT = false>
struct Cfg256 {
  static constexpr int KCH = D / 64;
  static constexpr int PLANES = SPLIT ? 2 : 1;
  static constexpr int QT_BYTES = kTile * D * 2;     // one plane of one 128-row Q tile
  static constexpr int Q_BYTES = 2 * PLANES * QT_BYTES;
  static constexpr int PLANE_BYTES = BN * D * 2;     // one plane of one K or V tile
  static constexpr int TILE_BYTES = PLANES * PLANE_BYTES;
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

// SPLIT: FP32 inputs given as bf16 high and low planes (the tensor maps' planes bh and
// BH + bh); each product is formed as hi*hi + hi*lo + lo*hi in the FP32 accumulator, P is
// split the same way in TMEM, and O is written in FP32.
template <int D, int BN, bool BF16, bool SPARSE, bool SPLIT>
__global__ void __launch_bounds__(kThreads256, 1)
    prefill_bm256_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p,
                         const __grid_constant__ PrefillSched sched) {
  using C = Cfg256<D, BN, SPLIT>;
  static_assert(!SPLIT || BF16, "split planes are bf16");
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
    {
      const bool leader = elect_one();
      uint32_t pos = 0, ii = 0;
      uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      uint32_t qfills[2] = {0, 0};
      bool ok = true;
      int t;
      for (int k = 0; ok && item_at(sched, p, cta, G, k, t); ++k) {
        if (t < 0) continue;
        int bh, mb;
        item_coords(t, p, bh, mb);
        const auto rg = item_range<SPARSE>(mb * BM, min(mb * BM + BM, p.Sq), BN, item_sk(p, bh), p, bh);
        const int n = range_count(rg);
        if (n == 0) continue;
        for (int q = 0; q < 2 && ok; ++q) {
          if (ii > 0 && !(ok = mbar_wait(B(bars->q_empty[q]), (ii - 1) & 1, wc))) break;
          if (leader) mbar_arrive_expect_tx(B(bars->q_full[q]), C::PLANES * C::QT_BYTES);
          if (leader)
            for (int h = 0; h < C::PLANES; ++h)
              for (int c = 0; c < C::KCH; ++c)
                tma_load_3d(sQ + (q * C::PLANES + h) * C::QT_BYTES + c * (kTile * 128), &tmQ,
                            B(bars->q_full[q]), c * 64, mb * BM + q * kTile, bh + h * p.BH);
          qfills[q] = ii + 1;
        }
        int nb = -1;
        for (int s = 0; s < 2 * n && ok; ++s) {  // K0, V0, K1, V1, ...
          if ((s & 1) == 0) nb = range_next(rg, nb);
          const int slot = pos % C::NSLOT;
          const uint32_t use = pos / C::NSLOT;
          if (!(ok = mbar_wait(B(bars->empty[slot]), (use & 1) ^ 1, wc))) break;
          const uint32_t dst = sRing + slot * C::TILE_BYTES;
          if (leader) mbar_arrive_expect_tx(B(bars->full[slot]), C::TILE_BYTES);
          int y, z;
          kv_tile_coords(p, bh, nb * BN, leader, y, z);
          const void* map = (s & 1) ? (const void*)&tmV : (const void*)&tmK;
          if (leader)
            for (int h = 0; h < C::PLANES; ++h)
              for (int c = 0; c < C::KCH; ++c)
                tma_load_3d(dst + h * C::PLANE_BYTES + c * (BN * 128), map, B(bars->full[slot]),
                            c * 64, y, z + h * p.BH);
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
    {
      const bool leader = elect_one();
      const uint32_t tS[2] = {tmem, tmem + BN};
      const uint32_t tO[2] = {tmem + 2 * BN, tmem + 2 * BN + D};
      // S_q = Q_q K^T and O_q (+)= P_q V with the operands in ring slot `slot` (issuing lane)
      auto qk = [&](int q, int slot) {
        const uint32_t qa = sQ + q * C::PLANES * C::QT_BYTES;
        const uint32_t kb = sRing + slot * C::TILE_BYTES;
        issue_qk<D, BN, BF16>(tS[q], qa, kb);
        if constexpr (SPLIT) {  // + Q_hi K_lo + Q_lo K_hi
          issue_qk<D, BN, BF16, true>(tS[q], qa, kb + C::PLANE_BYTES);
          issue_qk<D, BN, BF16, true>(tS[q], qa + C::QT_BYTES, kb);
        }
      };
      auto pv = [&](int q, int slot, bool acc) {
        const uint32_t vb = sRing + slot * C::TILE_BYTES;
        issue_pv<D, BN, BF16>(tO[q], tS[q], vb, acc);
        if constexpr (SPLIT) {  // + P_hi V_lo + P_lo V_hi
          issue_pv<D, BN, BF16>(tO[q], tS[q], vb + C::PLANE_BYTES, true);
          issue_pv<D, BN, BF16>(tO[q], tS[q] + BN / 2, vb, true);
        }
      };
      uint32_t pos = 0, ii = 0, tc = 0;
      bool ok = true;
      int t;
      for (int k = 0; ok && item_at(sched, p, cta, G, k, t); ++k) {
        if (t < 0) continue;
        int bh, mb;
        item_coords(t, p, bh, mb);
        const auto rg = item_range<SPARSE>(mb * BM, min(mb * BM + BM, p.Sq), BN, item_sk(p, bh), p, bh);
        const int n = range_count(rg);
        if (n == 0) continue;
        {  // S_A(0), S_B(0) with K0
          const int slot = pos % C::NSLOT;
          if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
          for (int q = 0; q < 2 && ok; ++q) {
            if (!(ok = mbar_wait(B(bars->q_full[q]), ii & 1, wc))) break;
            tc_fence_after();
            if (leader) qk(q, slot);
            if (leader) umma_commit(B(bars->s_full[q]));
            if (leader && n == 1) umma_commit(B(bars->q_empty[q]));
          }
          if (!ok) break;
          if (leader) umma_commit(B(bars->empty[slot]));
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
            if (leader) pv(q, vslot, j > 0);
            if (leader && j == n - 1) umma_commit(B(bars->pv_done[q]));
            if (leader && q == 1) umma_commit(B(bars->empty[vslot]));
            if (j + 1 < n) {  // S(j+1) overwrites P(j) only after PV(j) in the pipe
              if (q == 0) {
                if (!(ok = mbar_wait(B(bars->full[kslot]), ((pos + 1) / C::NSLOT) & 1, wc))) break;
                tc_fence_after();
              }
              if (leader) qk(q, kslot);
              if (leader) umma_commit(B(bars->s_full[q]));
              if (leader && j + 2 == n) umma_commit(B(bars->q_empty[q]));
              if (leader && q == 1) umma_commit(B(bars->empty[kslot]));
            }
          }
          pos += (j + 1 < n) ? 2 : 1;
          ++tc;
        }
        ++ii;
      }
      if (leader) umma_commit(B(bars->final_mma));  // all MMAs done before TMEM is released
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
    uint32_t ii = 0, tc = 0;
    bool ok = true;
    int t;
    for (int k = 0; ok && item_at(sched, p, cta, G, k, t); ++k) {
      if (t < 0) continue;
      int bh, mb;
      item_coords(t, p, bh, mb);
      const int sk = item_sk(p, bh);
      const auto rg = item_range<SPARSE>(mb * BM, min(mb * BM + BM, p.Sq), BN, sk, p, bh);
      const int n = range_count(rg);
      const int m0 = mb * BM + q * kTile;  // first row of this tile
      const int qrow = m0 + row;
      const size_t orow = static_cast<size_t>(bh) * p.Sq + qrow;
      if (n == 0) {  // nothing visible for any row of the item
        if (qrow < p.Sq) store_zero_row<D, SPLIT>(orow, p);
        continue;
      }
      const auto mine = item_range<SPARSE>(m0, min(m0 + kTile, p.Sq), BN, sk, p, bh);
      const int pos_q = qrow + sk - p.Sq;  // key position of this query
      float m_ref = -INFINITY, l = 0.f;
      int nb = -1;
      for (int j = 0; j < n; ++j) {
        nb = range_next(rg, nb);
        const bool full = tile_full<BN, SPARSE>(m0, nb, sk, bh, p);
        // a block-sparse item visits the blocks of either tile: one that is off for this
        // tile is masked whole (as if it held no key)
        const bool off = SPARSE && !range_has(mine, nb);
        const int sk_t = off ? nb * BN : sk;
        ok = mbar_wait(B(bars->s_full[q]), tc & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (p.trace && row == 0 && range_has(mine, nb))
          atomicAdd(p.trace + (static_cast<size_t>(bh) * ((p.Sq + kTile - 1) / kTile) +
                               m0 / kTile) * p.nnb + nb,
                    16 + (full ? 2 : 1));
        // S(j) was issued after PV(j-1), so O needs no wait before a rescale
        ok = softmax_tile<D, BN, BF16, SPLIT>(t_lane, s_col, o_col, full, nb * BN, pos_q, sk_t, p,
                                              m_ref, l, [] { return true; }, bh, m0);
        tc_fence_before();
        mbar_arrive(B(bars->p_full[q]));
        ++tc;
      }
      if (!ok) break;
      ok = mbar_wait(B(bars->pv_done[q]), ii & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      store_row<D, BF16, SPLIT>(t_lane, o_col, qrow < p.Sq, orow, m_ref, l, p);
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
//
// One 128-row query tile per work item, and one continuous stream of tiles across the
// items a CTA runs. Four warpgroups:
//   warps 0-3   softmax, first half of every score row (keys 0..BN/2-1 of the tile)
//   warps 4-7   softmax, second half; warps w and w+4 own the same 32 rows (TMEM lanes)
//               and swap their partial row maxima through shared memory each tile, so
//               that every scheduler has two independent softmax streams
//   warps 8-11  epilogue: O / l from TMEM to global memory, LSE; it works on the
//               previous item while the softmax warps start the next one
//   warp 12     TMA producer, warp 13 MMA issuer (one elected lane each), warps 14-15 idle
// TMEM: S0 [0,BN), S1 [BN,2BN) hold the score tiles of consecutive tiles; O0, O1
// (D columns each, from 2BN) hold the outputs of consecutive items. Q is double
// buffered in shared memory, so the first score tile of the next item is computed while
// the softmax still works on the last tile of the current one. Tensor-pipe order:
//   S(0) S(1) PV(0) S(2) PV(1) ... S(g+1) PV(g) ..., item boundaries included,
// so S(g) is always issued after PV(g-2) (it reuses that tile's S buffer).

constexpr int kThreads128 = 512;
constexpr int kTmaWarp128 = 12;
constexpr int kMmaWarp128 = 13;
// launched at 128 registers per thread: 128 x (152 + 152 + 104 + 104) = 512 x 128 = 65,536
constexpr uint32_t kRegs128Softmax = 152;
constexpr uint32_t kRegs128Epilogue = 104;
constexpr uint32_t kRegs128Producer = 104;

template <int D, int BN>
struct Cfg128 {
  static constexpr int KCH = D / 64;
  static constexpr int Q_BYTES = kTile * D * 2;  // one Q buffer
  static constexpr int TILE_BYTES = BN * D * 2;
  static constexpr int STATS_BYTES = 2 * 2 * kTile * 8;  // (m, l) per row and half, two items
  static constexpr int XMAX_BYTES = 2 * 2 * kTile * 4;   // partial row maxima, two tiles
  static constexpr int BAR_BYTES = 1024;
  static constexpr int NSLOT_FIT = (int)((kSmemLimit - 1024 - BAR_BYTES - STATS_BYTES -
                                          XMAX_BYTES - 2 * Q_BYTES) / TILE_BYTES);
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;
  static constexpr bool kRelease = NSLOT == 4;  // slots released by s_full / pv_done
  static constexpr int SMEM =
      1024 + 2 * Q_BYTES + NSLOT * TILE_BYTES + STATS_BYTES + XMAX_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN + 2 * D);
  static_assert(NSLOT >= 3, "shared memory ring too small");
  static_assert(SMEM <= (int)kSmemLimit, "shared memory over budget");
  static_assert(2 * BN + 2 * D <= 512, "TMEM over budget");
};

struct Bars128 {
  uint64_t full[8], empty[8];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_full[2], o_empty[2], stats_full[2];
  uint64_t xbar[2][4];  // row-max exchange between the two softmax halves, per tile parity
  uint64_t final_mma;
  uint32_t tmem_base;
  uint32_t abort;
};

template <bool SPARSE>
struct ItemRef {
  int bh, mb, n, sk;
  std::conditional_t<SPARSE, SparseRange, Range> rg;
};


// Next item of this CTA (empty ones included when `with_empty`): false when none is left.
template <int BM, bool SPARSE>
__device__ __forceinline__ bool next_item(const PrefillSched& s, const PrefillParams& p, int cta,
                                          int G, int BN, int& k, ItemRef<SPARSE>& it,
                                          bool with_empty) {
  int t;
  while (item_at(s, p, cta, G, k, t)) {
    ++k;
    if (t < 0) continue;
    item_coords(t, p, it.bh, it.mb);
    it.sk = item_sk(p, it.bh);
    it.rg = item_range<SPARSE>(it.mb * BM, min(it.mb * BM + BM, p.Sq), BN, it.sk, p, it.bh);
    it.n = range_count(it.rg);
    if (it.n > 0 || with_empty) return true;
  }
  return false;
}

template <int D, int BN, bool BF16, bool SPARSE>
__global__ void __launch_bounds__(kThreads128, 1)
    prefill_bm128_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p,
                         const __grid_constant__ PrefillSched sched) {
  using C = Cfg128<D, BN>;
  constexpr int BM = kTile;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base;  // two Q buffers
  const uint32_t sRing = base + 2 * C::Q_BYTES;
  float2* stats = reinterpret_cast<float2*>(smem + 2 * C::Q_BYTES + C::NSLOT * C::TILE_BYTES);
  float* xmax = reinterpret_cast<float*>(smem + 2 * C::Q_BYTES + C::NSLOT * C::TILE_BYTES +
                                         C::STATS_BYTES);
  Bars128* bars = reinterpret_cast<Bars128*>(smem + 2 * C::Q_BYTES + C::NSLOT * C::TILE_BYTES +
                                             C::STATS_BYTES + C::XMAX_BYTES);
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
      mbar_init(B(bars->p_full[i]), 256);
      mbar_init(B(bars->pv_done[i]), 1);
      mbar_init(B(bars->o_full[i]), 1);
      mbar_init(B(bars->o_empty[i]), 128);
      mbar_init(B(bars->stats_full[i]), 256);
      for (int w = 0; w < 4; ++w) mbar_init(B(bars->xbar[i][w]), 64);
    }
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

  // The role branches never rejoin: each ends with the CTA-wide teardown barrier.
  if (warp >= 12) {
    regs_decrease<kRegs128Producer>();
    if (warp == kTmaWarp128) {
      // ---------------------------------------------------------- TMA producer
      const bool leader = elect_one();
      // Loads in the MMA's consumption order: Q and K(0) of the first item, then per
      // tile: K of the following tile (the next item's Q first when it starts one), V.
      uint32_t pos = 0, ii = 0;
      uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      uint32_t qfills[2] = {0, 0};
      // With a four-slot ring (two tiles) a slot is free again once the MMA that read
      // its previous tile is complete: S(t) (s_full[t&1]) for K(t), P.V(t) (pv_done[t&1])
      // for V(t), so the MMA issuer needs no per-slot commits. No barrier can be two
      // phases ahead of such a wait, because the next MMA on it needs the tile about to
      // be loaded. The one exception is the first reuse (V(1) into the slot of K(0)),
      // which waits for S(1) instead (a commit covers every earlier MMA, and S(3) needs
      // K(3)). A deeper ring reuses slots more than two tiles later, where a parity wait
      // on those barriers would be ambiguous: it keeps one `empty` barrier per slot.
      uint32_t rel_bar[C::NSLOT] = {}, rel_par[C::NSLOT] = {};
      uint32_t nk = 0, nv = 0;  // K and V tiles loaded so far
      bool ok = true;
      int kc = 0;
      ItemRef<SPARSE> cur, nxt;
      auto load_q = [&](const ItemRef<SPARSE>& it, uint32_t idx) {
        const int qb = idx & 1;
        if (idx >= 2 && !(ok = mbar_wait(B(bars->q_empty[qb]), ((idx >> 1) - 1) & 1, wc)))
          return;
        if (leader) {
          mbar_arrive_expect_tx(B(bars->q_full[qb]), C::Q_BYTES);
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(sQ + qb * C::Q_BYTES + c * (kTile * 128), &tmQ, B(bars->q_full[qb]),
                        c * 64, it.mb * BM, it.bh);
        }
        qfills[qb] = (idx >> 1) + 1;
      };
      auto emit = [&](const ItemRef<SPARSE>& it, int nb, bool is_v) {
        const int slot = pos % C::NSLOT;
        if constexpr (!C::kRelease) {
          if (!(ok = mbar_wait(B(bars->empty[slot]), ((pos / C::NSLOT) & 1) ^ 1, wc))) return;
        } else if (pos >= C::NSLOT && !(ok = mbar_wait(rel_bar[slot], rel_par[slot], wc))) {
          return;
        }
        if (is_v) {
          rel_bar[slot] = B(bars->pv_done[nv & 1]);
          rel_par[slot] = (nv >> 1) & 1;
          ++nv;
        } else {
          const uint32_t t = nk == 0 ? 1 : nk;  // K(0): released by S(1), see above
          rel_bar[slot] = B(bars->s_full[t & 1]);
          rel_par[slot] = (t >> 1) & 1;
          ++nk;
        }
        const uint32_t dst = sRing + slot * C::TILE_BYTES;
        if (leader) mbar_arrive_expect_tx(B(bars->full[slot]), C::TILE_BYTES);
        int y, z;
        kv_tile_coords(p, it.bh, nb * BN, leader, y, z);
        const void* map = is_v ? (const void*)&tmV : (const void*)&tmK;
        if (leader)
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(dst + c * (BN * 128), map, B(bars->full[slot]), c * 64, y, z);
        fills[slot] = pos / C::NSLOT + 1;  // uses of this slot so far
        ++pos;
      };
      bool has = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, cur, false);
      int nb_cur = -1;  // key block of the current tile
      if (has) {
        load_q(cur, 0);
        nb_cur = range_next(cur.rg, -1);
        if (ok) emit(cur, nb_cur, false);
      }
      while (has && ok) {
        bool has_nxt = false;
        for (int j = 0; j < cur.n && ok; ++j) {
          int nb_next = -1;  // key block of the following tile
          if (j + 1 < cur.n) {
            nb_next = range_next(cur.rg, nb_cur);
            emit(cur, nb_next, false);
          } else {
            has_nxt = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, nxt, false);
            if (has_nxt) {
              load_q(nxt, ii + 1);
              nb_next = range_next(nxt.rg, -1);
              if (ok) emit(nxt, nb_next, false);
            }
          }
          if (ok) emit(cur, nb_cur, true);
          nb_cur = nb_next;
        }
        ++ii;
        cur = nxt;
        has = has_nxt;
      }
      if (!ok) {  // wind down: every load this thread issued lands before the CTA exits
        for (int s = 0; s < C::NSLOT; ++s)
          if (fills[s] > 0) wait_quiet(B(bars->full[s]), (fills[s] - 1) & 1, wc);
        for (int q = 0; q < 2; ++q)
          if (qfills[q] > 0) wait_quiet(B(bars->q_full[q]), (qfills[q] - 1) & 1, wc);
      }
    } else if (warp == kMmaWarp128) {
      // ---------------------------------------------------------- MMA issuer
      // The whole warp runs the loop and the waits; one elected lane issues the MMAs and
      // the commits that track them (a commit covers the MMAs of the thread issuing it).
      const bool leader = elect_one();
      auto commit = [&](uint64_t& bar) {
        if (leader) umma_commit(B(bar));
      };
      uint32_t pos = 0, ii = 0, g = 0;
      bool ok = true;
      int kc = 0;
      ItemRef<SPARSE> cur, nxt;
      auto issue_s = [&](uint32_t sbuf, uint32_t qb) {
        const int slot = pos % C::NSLOT;
        if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) return;
        tc_fence_after();
        if (leader) {
          issue_qk<D, BN, BF16>(tmem + sbuf * BN, sQ + qb * C::Q_BYTES,
                                sRing + slot * C::TILE_BYTES);
          umma_commit(B(bars->s_full[sbuf]));
          if constexpr (!C::kRelease) umma_commit(B(bars->empty[slot]));
        }
        ++pos;
      };
      bool has = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, cur, false);
      if (has) {
        if ((ok = mbar_wait(B(bars->q_full[0]), 0, wc))) {
          tc_fence_after();
          issue_s(0, 0);
          if (ok && cur.n == 1) commit(bars->q_empty[0]);
        }
      }
      while (has && ok) {
        const uint32_t buf = ii & 1;
        bool has_nxt = false;
        for (int j = 0; j < cur.n && ok; ++j, ++g) {
          // score tile of the following tile, into the other S buffer
          if (j + 1 < cur.n) {
            issue_s((g + 1) & 1, buf);
            if (ok && j + 2 == cur.n) commit(bars->q_empty[buf]);
          } else {
            has_nxt = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, nxt, false);
            if (has_nxt) {
              const uint32_t nb = (ii + 1) & 1;
              if (!(ok = mbar_wait(B(bars->q_full[nb]), ((ii + 1) >> 1) & 1, wc))) break;
              tc_fence_after();
              issue_s((g + 1) & 1, nb);
              if (ok && nxt.n == 1) commit(bars->q_empty[nb]);
            }
          }
          if (!ok) break;
          // O(item) += P(g) V(g)
          if (!(ok = mbar_wait(B(bars->p_full[g & 1]), (g >> 1) & 1, wc))) break;
          tc_fence_after();
          if (j == 0 && ii >= 2) {  // the epilogue of two items back has read this O
            if (!(ok = mbar_wait(B(bars->o_empty[buf]), ((ii >> 1) - 1) & 1, wc))) break;
            tc_fence_after();
          }
          const int slot = pos % C::NSLOT;
          if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
          tc_fence_after();
          if (leader) {
            issue_pv<D, BN, BF16>(tmem + 2 * BN + buf * D, tmem + (g & 1) * BN,
                                  sRing + slot * C::TILE_BYTES, j > 0);
            umma_commit(B(bars->pv_done[g & 1]));
            if constexpr (!C::kRelease) umma_commit(B(bars->empty[slot]));
            if (j + 1 == cur.n) umma_commit(B(bars->o_full[buf]));
          }
          ++pos;
        }
        ++ii;
        cur = nxt;
        has = has_nxt;
      }
      if (leader) umma_commit(B(bars->final_mma));  // all MMAs done before TMEM is released
      wait_quiet(B(bars->final_mma), 0, wc);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();  // teardown
    return;
  } else if (warp >= 8) {
    regs_decrease<kRegs128Epilogue>();
    // ------------------------------------------------------------ epilogue warps 8-11
    const int row = (warp % 4) * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    uint32_t ii = 0;
    bool ok = true;
    int kc = 0;
    ItemRef<SPARSE> it;
    while (ok && next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, it, true)) {
      const int qrow = it.mb * BM + row;
      const size_t orow = static_cast<size_t>(it.bh) * p.Sq + qrow;
      if (it.n == 0) {  // no row of this item sees a key
        if (qrow < p.Sq) store_zero_row<D>(orow, p);
        continue;
      }
      const uint32_t buf = ii & 1, use = ii >> 1;
      ok = mbar_wait(B(bars->stats_full[buf]), use & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      ok = mbar_wait(B(bars->o_full[buf]), use & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const float2 h0 = stats[(buf * 2 + 0) * kTile + row];
      const float2 h1 = stats[(buf * 2 + 1) * kTile + row];
      store_row<D, BF16>(t_lane, 2 * BN + buf * D, qrow < p.Sq, orow, h0.x, h0.y + h1.y, p);
      tc_fence_before();
      mbar_arrive(B(bars->o_empty[buf]));
      ++ii;
    }
    tc_fence_before();
    __syncthreads();  // teardown
    return;
  } else {
    regs_increase<kRegs128Softmax>();
    // ------------------------------------------------------------ softmax warps 0-7
    const int half = warp / 4;  // 0: keys [0, BN/2) of each tile, 1: keys [BN/2, BN)
    const int row = (warp % 4) * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    uint32_t ii = 0, g = 0;
    bool ok = true;
    int kc = 0;
    ItemRef<SPARSE> it;
    while (ok && next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, it, false)) {
      const uint32_t buf = ii & 1;
      const int m0 = it.mb * BM;
      const int pos_q = m0 + row + it.sk - p.Sq;  // key position of this query
      float m_ref = -INFINITY, l = 0.f;
      int nb = -1;
      for (int j = 0; j < it.n; ++j, ++g) {
        nb = range_next(it.rg, nb);
        const bool full = tile_full<BN, SPARSE>(m0, nb, it.sk, it.bh, p);
        ok = mbar_wait(B(bars->s_full[g & 1]), (g >> 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (p.trace && half == 0 && row == 0)
          atomicAdd(p.trace + (static_cast<size_t>(it.bh) * p.nmb + it.mb) * p.nnb + nb,
                    16 + (full ? 2 : 1));
        // The two halves of a row swap partial maxima (double buffered by tile parity,
        // one barrier per warp pair: a bounded wait, so an abort cannot strand the
        // partner). The barrier also guarantees that both halves hold their S values in
        // registers before either writes P over the S columns.
        bool x_ok = true;
        auto exchange = [&](float mp) {
          float* xm = xmax + (g & 1) * 2 * kTile;
          xm[half * kTile + row] = mp;
          const uint32_t xb = B(bars->xbar[g & 1][warp % 4]);
          mbar_arrive(xb);
          x_ok = mbar_wait(xb, (g >> 1) & 1, wc);
          x_ok = __all_sync(0xffffffffu, x_ok);
          return x_ok ? fmaxf(mp, xm[(1 - half) * kTile + row]) : mp;
        };
        // O must hold every earlier P.V product of this item before it is rescaled
        const uint32_t pc = g - 1;
        auto wait_pv = [&]() {
          bool w = mbar_wait(B(bars->pv_done[pc & 1]), (pc >> 1) & 1, wc);
          w = __all_sync(0xffffffffu, w);
          if (w) tc_fence_after();
          return w;
        };
        const uint32_t s_col = (g & 1) * BN;
        ok = softmax_cols<BN / 2, D / 2, BF16, false>(t_lane, s_col + half * (BN / 2),
                                               s_col + half * (BN / 4),
                                               2 * BN + buf * D + half * (D / 2), full,
                                               nb * BN + half * (BN / 2), pos_q, it.sk, p, m_ref,
                                               l, exchange, wait_pv, half == 0 ? it.bh : -1, m0);
        if (!ok || !x_ok) {
          ok = false;
          break;
        }
        tc_fence_before();
        mbar_arrive(B(bars->p_full[g & 1]));
      }
      if (!ok) break;
      // hand this row's statistics to the epilogue (its buffer is free once the
      // epilogue of two items back is done)
      if (ii >= 2) {
        ok = mbar_wait(B(bars->o_empty[buf]), ((ii >> 1) - 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      stats[(buf * 2 + half) * kTile + row] = make_float2(m_ref, l);
      mbar_arrive(B(bars->stats_full[buf]));
      ++ii;
    }
    tc_fence_before();
    __syncthreads();  // teardown
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
  }
}

// ------------------------------------------------------------------ BM = 64 kernel
//
// One 64-row query tile per work item, on tcgen05 MMAs with M = 64: the BLOCK_M = 64 point
// of the tile-size tuning the ops-transformer overview describes (section 三.1, 64x64,
// 128x128 and 256x256 blocks). Roles (192 threads):
//   warps 0-3   softmax and epilogue. The accumulator of an M = 64 MMA occupies TMEM
//               lanes 0-15 of each warp's 32-lane quarter (row 16w + l in lane 32w + l),
//               so lanes 0-15 of each warp own a row; lanes 16-31 take part in the
//               warp-wide TMEM loads and stores but own nothing.
//   warp 4      TMA producer: Q (double buffered), then K of the next tile and V of the
//               current one, as in the 128-row kernel.
//   warp 5      MMA issuer (elected lane): S(g+1) = Q K^T, then O += P(g) V(g).
// P is written to shared memory (two 64 x BN buffers) rather than TMEM and the P.V MMA
// reads both operands from shared memory.
// TMEM: S0 [0,BN), S1 [BN,2BN), O0 [2BN,2BN+D), O1 [2BN+D,2BN+2D) (items alternate).
constexpr int kTile64 = 64;
constexpr int kThreads64 = 192;
constexpr int kTmaWarp64 = 4;
constexpr int kMmaWarp64 = 5;

template <int D, int BN>
struct Cfg64 {
  static constexpr int KCH = D / 64;
  static constexpr int Q_BYTES = kTile64 * D * 2;   // one Q buffer
  static constexpr int P_BYTES = kTile64 * BN * 2;  // one P buffer
  static constexpr int TILE_BYTES = BN * D * 2;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int NSLOT_FIT =
      (int)((kSmemLimit - 1024 - BAR_BYTES - 2 * Q_BYTES - 2 * P_BYTES) / TILE_BYTES);
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;
  static constexpr int SMEM = 1024 + 2 * Q_BYTES + 2 * P_BYTES + NSLOT * TILE_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN + 2 * D);
  static_assert(NSLOT >= 3, "shared memory ring too small");
  static_assert(SMEM <= (int)kSmemLimit, "shared memory over budget");
  static_assert(2 * BN + 2 * D <= 512, "TMEM over budget");
};

struct Bars64 {
  uint64_t full[8], empty[8];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2], o_empty[2];
  uint64_t final_mma;
  uint32_t tmem_base;
  uint32_t abort;
};

template <int D, int BN, bool BF16, bool SPARSE>
__global__ void __launch_bounds__(kThreads64, 1)
    prefill_bm64_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const PrefillParams p,
                        const __grid_constant__ PrefillSched sched) {
  using C = Cfg64<D, BN>;
  constexpr int BM = kTile64;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base;                          // two Q buffers
  const uint32_t sP = base + 2 * C::Q_BYTES;         // two P buffers
  const uint32_t sRing = sP + 2 * C::P_BYTES;
  Bars64* bars = reinterpret_cast<Bars64*>(smem + 2 * C::Q_BYTES + 2 * C::P_BYTES +
                                           C::NSLOT * C::TILE_BYTES);
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
  if (warp == kTmaWarp64 && lane == 0) {
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

  if (warp == kTmaWarp64) {
    // ------------------------------------------------------------ TMA producer
    const bool leader = elect_one();
    uint32_t pos = 0, ii = 0;
    uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    uint32_t qfills[2] = {0, 0};
    bool ok = true;
    int kc = 0;
    ItemRef<SPARSE> cur, nxt;
    auto load_q = [&](const ItemRef<SPARSE>& it, uint32_t idx) {
      const int qb = idx & 1;
      if (idx >= 2 && !(ok = mbar_wait(B(bars->q_empty[qb]), ((idx >> 1) - 1) & 1, wc))) return;
      if (leader) {
        mbar_arrive_expect_tx(B(bars->q_full[qb]), C::Q_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sQ + qb * C::Q_BYTES + c * (BM * 128), &tmQ, B(bars->q_full[qb]), c * 64,
                      it.mb * BM, it.bh);
      }
      qfills[qb] = (idx >> 1) + 1;
    };
    auto emit = [&](const ItemRef<SPARSE>& it, int nb, bool is_v) {
      const int slot = pos % C::NSLOT;
      if (!(ok = mbar_wait(B(bars->empty[slot]), ((pos / C::NSLOT) & 1) ^ 1, wc))) return;
      const uint32_t dst = sRing + slot * C::TILE_BYTES;
      if (leader) mbar_arrive_expect_tx(B(bars->full[slot]), C::TILE_BYTES);
      int y, z;
      kv_tile_coords(p, it.bh, nb * BN, leader, y, z);
      const void* map = is_v ? (const void*)&tmV : (const void*)&tmK;
      if (leader)
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(dst + c * (BN * 128), map, B(bars->full[slot]), c * 64, y, z);
      fills[slot] = pos / C::NSLOT + 1;
      ++pos;
    };
    // loads in the MMA's consumption order: Q and K(0) of the first item, then per tile K
    // of the following tile (the next item's Q first when it starts one), V
    bool has = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, cur, false);
    int nb_cur = -1;
    if (has) {
      load_q(cur, 0);
      nb_cur = range_next(cur.rg, -1);
      if (ok) emit(cur, nb_cur, false);
    }
    while (has && ok) {
      bool has_nxt = false;
      for (int j = 0; j < cur.n && ok; ++j) {
        int nb_next = -1;
        if (j + 1 < cur.n) {
          nb_next = range_next(cur.rg, nb_cur);
          emit(cur, nb_next, false);
        } else {
          has_nxt = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, nxt, false);
          if (has_nxt) {
            load_q(nxt, ii + 1);
            nb_next = range_next(nxt.rg, -1);
            if (ok) emit(nxt, nb_next, false);
          }
        }
        if (ok) emit(cur, nb_cur, true);
        nb_cur = nb_next;
      }
      ++ii;
      cur = nxt;
      has = has_nxt;
    }
    if (!ok) {  // wind down: every load this thread issued lands before the CTA exits
      for (int s = 0; s < C::NSLOT; ++s)
        if (fills[s] > 0) wait_quiet(B(bars->full[s]), (fills[s] - 1) & 1, wc);
      for (int q = 0; q < 2; ++q)
        if (qfills[q] > 0) wait_quiet(B(bars->q_full[q]), (qfills[q] - 1) & 1, wc);
    }
    __syncwarp();
  } else if (warp == kMmaWarp64) {
    // ------------------------------------------------------------ MMA issuer
    // Pipe order S(0) S(1) PV(0) S(2) PV(1) ...: S(g) is issued after PV(g-2), so the
    // softmax's wait for S(g) also covers the P buffer and S columns that PV(g-2) read.
    const bool leader = elect_one();
    uint32_t pos = 0, ii = 0, g = 0;
    bool ok = true;
    int kc = 0;
    ItemRef<SPARSE> cur, nxt;
    auto issue_s = [&](uint32_t sbuf, uint32_t qb) {
      const int slot = pos % C::NSLOT;
      if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) return;
      tc_fence_after();
      if (leader) {
        issue_qk_m64<D, BN, BF16>(tmem + sbuf * BN, sQ + qb * C::Q_BYTES,
                                  sRing + slot * C::TILE_BYTES);
        umma_commit(B(bars->s_full[sbuf]));
        umma_commit(B(bars->empty[slot]));
      }
      ++pos;
    };
    bool has = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, cur, false);
    if (has && (ok = mbar_wait(B(bars->q_full[0]), 0, wc))) {
      tc_fence_after();
      issue_s(0, 0);
      if (ok && cur.n == 1 && leader) umma_commit(B(bars->q_empty[0]));
    }
    while (has && ok) {
      const uint32_t buf = ii & 1;
      bool has_nxt = false;
      for (int j = 0; j < cur.n && ok; ++j, ++g) {
        if (j + 1 < cur.n) {  // scores of the following tile, into the other S buffer
          issue_s((g + 1) & 1, buf);
          if (ok && j + 2 == cur.n && leader) umma_commit(B(bars->q_empty[buf]));
        } else {
          has_nxt = next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, nxt, false);
          if (has_nxt) {
            const uint32_t nb = (ii + 1) & 1;
            if (!(ok = mbar_wait(B(bars->q_full[nb]), ((ii + 1) >> 1) & 1, wc))) break;
            tc_fence_after();
            issue_s((g + 1) & 1, nb);
            if (ok && nxt.n == 1 && leader) umma_commit(B(bars->q_empty[nb]));
          }
        }
        if (!ok) break;
        // O(item) += P(g) V(g)
        if (!(ok = mbar_wait(B(bars->p_full[g & 1]), (g >> 1) & 1, wc))) break;
        tc_fence_after();
        if (j == 0 && ii >= 2) {  // the epilogue of two items back has read this O
          if (!(ok = mbar_wait(B(bars->o_empty[buf]), ((ii >> 1) - 1) & 1, wc))) break;
          tc_fence_after();
        }
        const int slot = pos % C::NSLOT;
        if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
        tc_fence_after();
        if (leader) {
          issue_pv_m64<D, BN, BF16>(tmem + 2 * BN + buf * D, sP + (g & 1) * C::P_BYTES,
                                    sRing + slot * C::TILE_BYTES, j > 0);
          umma_commit(B(bars->pv_done[g & 1]));
          umma_commit(B(bars->empty[slot]));
        }
        ++pos;
      }
      ++ii;
      cur = nxt;
      has = has_nxt;
    }
    if (leader) umma_commit(B(bars->final_mma));  // all MMAs done before TMEM is released
    wait_quiet(B(bars->final_mma), 0, wc);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const bool mine = lane < 16;  // this lane owns a row of the tile
    const int row = (warp % 4) * 16 + (lane & 15);
    const uint32_t t_lane = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    uint32_t ii = 0, g = 0;
    bool ok = true;
    int kc = 0;
    ItemRef<SPARSE> it;
    while (ok && next_item<BM, SPARSE>(sched, p, cta, G, BN, kc, it, true)) {
      const int m0 = it.mb * BM;
      const int qrow = m0 + row;
      const size_t orow = static_cast<size_t>(it.bh) * p.Sq + qrow;
      if (it.n == 0) {  // no row of this item sees a key
        if (mine && qrow < p.Sq) store_zero_row<D>(orow, p);
        continue;
      }
      const uint32_t buf = ii & 1;
      const int pos_q = qrow + it.sk - p.Sq;  // key position of this query
      float m_ref = -INFINITY, l = 0.f;
      int nb = -1;
      for (int j = 0; j < it.n; ++j, ++g) {
        nb = range_next(it.rg, nb);
        const bool full = tile_full<BN, SPARSE, BM>(m0, nb, it.sk, it.bh, p);
        ok = mbar_wait(B(bars->s_full[g & 1]), (g >> 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        if (p.trace && warp == 0 && lane == 0)
          atomicAdd(p.trace + (static_cast<size_t>(it.bh) * p.nmb + it.mb) * p.nnb + nb,
                    16 + (full ? 2 : 1));
        // O must hold every earlier P.V product of this item before it is rescaled
        const uint32_t pc = g - 1;
        auto wait_pv = [&]() {
          bool w = mbar_wait(B(bars->pv_done[pc & 1]), (pc >> 1) & 1, wc);
          w = __all_sync(0xffffffffu, w);
          if (w) tc_fence_after();
          return w;
        };
        // lanes that own no row see every key masked (a query at position -1 with no
        // keys), so they never ask for a rescale and write no P
        ok = softmax_cols<BN, D, BF16, false, true>(
            t_lane, (g & 1) * BN, sP + (g & 1) * C::P_BYTES, 2 * BN + buf * D, full && mine,
            nb * BN, mine ? pos_q : -1, mine ? it.sk : 0, p, m_ref, l,
            [](float m) { return m; }, wait_pv, mine ? it.bh : -1, m0, mine ? row : -1);
        if (!ok) break;
        tc_fence_before();
        mbar_arrive(B(bars->p_full[g & 1]));
      }
      if (!ok) break;
      // epilogue: the item's last P.V, then O / l and LSE
      const uint32_t pl = g - 1;
      ok = mbar_wait(B(bars->pv_done[pl & 1]), (pl >> 1) & 1, wc);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      store_row<D, BF16>(t_lane, 2 * BN + buf * D, mine && qrow < p.Sq, orow, m_ref, l, p);
      tc_fence_before();
      mbar_arrive(B(bars->o_empty[buf]));
      ++ii;
    }
    tc_fence_before();
    __syncthreads();  // teardown
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    }
    return;
  }
  tc_fence_before();
  __syncthreads();  // teardown
}

// Once per kernel and device (the attributes belong to the device's copy of the kernel):
// check that the launch register count covers the kernel's setmaxnreg split (setmaxnreg.inc
// can only hand out registers the CTA was launched with, so a build below the split would
// make the softmax warps wait forever: it is refused instead of launched), and raise the
// dynamic shared-memory limit.
template <auto KERN>
cudaError_t prepare_kernel(int threads, int split_regs_x128, int smem) {
  static std::atomic<uint64_t> ready{0};  // this kernel: one bit per device index below 64
  const auto kern = KERN;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit && (ready.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  cudaFuncAttributes fattr;
  if ((e = cudaFuncGetAttributes(&fattr, kern)) != cudaSuccess) return e;
  if (fattr.numRegs * threads < split_regs_x128 * 128) return cudaErrorInvalidConfiguration;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) !=
      cudaSuccess)
    return e;
  ready.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

template <int D, int BN, bool BF16, bool SPARSE, bool SPLIT = false>
cudaError_t launch_k(const PrefillLaunch& L, int BM, cudaStream_t stream) {
  if constexpr (!SPLIT) {
    if (BM == 64) {
      auto kern = prefill_bm64_kernel<D, BN, BF16, SPARSE>;
      constexpr int smem = Cfg64<D, BN>::SMEM;
      cudaError_t e = prepare_kernel<prefill_bm64_kernel<D, BN, BF16, SPARSE>>(kThreads64, 0, smem);
      if (e != cudaSuccess) return e;
      kern<<<L.grid, kThreads64, smem, stream>>>(L.tmQ, L.tmK, L.tmV, L.p, *L.sched);
      return cudaGetLastError();
    }
  }
  if (SPLIT || BM == 256) {
    auto kern = prefill_bm256_kernel<D, BN, BF16, SPARSE, SPLIT>;
    constexpr int smem = Cfg256<D, BN, SPLIT>::SMEM;
    cudaError_t e = prepare_kernel<prefill_bm256_kernel<D, BN, BF16, SPARSE, SPLIT>>(
        kThreads256, 2 * kRegsSoftmax + kRegsProducer, smem);
    if (e != cudaSuccess) return e;
    kern<<<L.grid, kThreads256, smem, stream>>>(L.tmQ, L.tmK, L.tmV, L.p, *L.sched);
  } else if constexpr (!SPLIT) {
    auto kern = prefill_bm128_kernel<D, BN, BF16, SPARSE>;
    constexpr int smem = Cfg128<D, BN>::SMEM;
    cudaError_t e = prepare_kernel<prefill_bm128_kernel<D, BN, BF16, SPARSE>>(
        kThreads128, kRegs128Softmax + kRegs128Epilogue + kRegs128Producer, smem);
    if (e != cudaSuccess) return e;
    kern<<<L.grid, kThreads128, smem, stream>>>(L.tmQ, L.tmK, L.tmV, L.p, *L.sched);
  }
  return cudaGetLastError();
}

#ifndef FA_PREFILL_SPLIT_TU
template <int D, int BN, bool BF16>
cudaError_t launch_t(const PrefillLaunch& L, int BM, cudaStream_t stream) {
  return L.p.mask_mode == FA_MASK_BLOCK_SPARSE ? launch_k<D, BN, BF16, true>(L, BM, stream)
                                               : launch_k<D, BN, BF16, false>(L, BM, stream);
}
#else
// FP32 inputs, step 1: x -> (hi, lo) = (bf16(x), bf16(x - hi)), eight elements per
// thread and iteration, over the three tensors Q, K, V in one launch. x - hi is exact in
// FP32 (hi is x rounded to 8 significant bits), so hi + lo equals x to 2^-16 relative:
// the split of the "bf16x3" products of Henry, Tang and Heinecke, "Leveraging the bfloat16
// Artificial Intelligence Datatype For Higher-Precision Computations" (ARITH 2019).
__global__ void __launch_bounds__(256) split_bf16_kernel(const SplitArgs a) {
  const size_t n0 = a.n8[0], n01 = n0 + a.n8[1], total = n01 + a.n8[2];
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const int t = i < n0 ? 0 : (i < n01 ? 1 : 2);
    const size_t j = i - (t == 0 ? 0 : (t == 1 ? n0 : n01));
    const float* src = t == 0 ? a.src[0] : (t == 1 ? a.src[1] : a.src[2]);
    uint16_t* hi = t == 0 ? a.hi[0] : (t == 1 ? a.hi[1] : a.hi[2]);
    uint16_t* lo = t == 0 ? a.lo[0] : (t == 1 ? a.lo[1] : a.lo[2]);
    const float4* x4 = reinterpret_cast<const float4*>(src) + 2 * j;
    const float4 u = __ldcs(x4), w = __ldcs(x4 + 1);
    const float x[8] = {u.x, u.y, u.z, u.w, w.x, w.y, w.z, w.w};
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h[e] = cvt_pack_bf16(x[2 * e], x[2 * e + 1]);  // low half: the even element
      l[e] = cvt_pack_bf16(x[2 * e] - __uint_as_float(h[e] << 16),
                           x[2 * e + 1] - __uint_as_float(h[e] & 0xffff0000u));
    }
    reinterpret_cast<uint4*>(hi)[j] = make_uint4(h[0], h[1], h[2], h[3]);
    reinterpret_cast<uint4*>(lo)[j] = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

template <int D, bool SPARSE>
cudaError_t launch_split_t(const PrefillLaunch& L, cudaStream_t stream) {
  return launch_k<D, kSplitBlockN, true, SPARSE, true>(L, 256, stream);
}
#endif

}  // namespace

#ifndef FA_PREFILL_SPLIT_TU
int prefill_tile_rows() { return kTile; }

cudaError_t launch_prefill(const PrefillLaunch& L, int D, int BN, int BM, bool bf16,
                           cudaStream_t stream) {
  if (BM != 64 && BM != 128 && BM != 256) return cudaErrorInvalidValue;
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
#else
cudaError_t launch_split_bf16(const SplitArgs& a, int sms, cudaStream_t stream) {
  const size_t total = a.n8[0] + a.n8[1] + a.n8[2];
  if (total == 0) return cudaSuccess;
  size_t blocks = (total + 255) / 256;
  const size_t cap = static_cast<size_t>(sms > 0 ? sms : 1) * 8;  // 8 x 256 threads per SM
  if (blocks > cap) blocks = cap;
  split_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_split(const PrefillLaunch& L, int D, cudaStream_t stream) {
  const bool sparse = L.p.mask_mode == FA_MASK_BLOCK_SPARSE;
  if (D == 64) return sparse ? launch_split_t<64, true>(L, stream) : launch_split_t<64, false>(L, stream);
  if (D == 128)
    return sparse ? launch_split_t<128, true>(L, stream) : launch_split_t<128, false>(L, stream);
  return cudaErrorInvalidValue;
}
#endif

}  // namespace fa
