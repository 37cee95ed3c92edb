// Work-item planning shared by the host planner (fa_api.cu) and the prefill kernels:
// which key blocks a block of query rows visits, how work items are numbered, and the
// per-CTA item lists that balance a persistent launch.
#pragma once

#include <cstdint>

#include "fa_internal.h"

#if defined(__CUDACC__)
#define FA_HD __host__ __device__ __forceinline__
#else
#define FA_HD inline
#endif

namespace fa {

// Key blocks visited by the query rows [m0, m1): [0, a_end) then [b_start, b_end),
// a_end <= b_start. Closed form of the mask: every block inside holds at least one
// visible pair for these rows, every block outside holds none.
struct Range {
  int a_end, b_start, b_end;
};

// A block-sparse mask (device code only) visits the blocks of [0, b_end) whose layout
// byte is set in the row of either query block (la, lb; key block nb -> layout column
// nb >> shift). Kept apart from Range so that the other masks carry none of it.
struct SparseRange {
  int a_end, b_start, b_end;
  const uint8_t* la;
  const uint8_t* lb;
  int shift;
};

FA_HD int imin(int a, int b) { return a < b ? a : b; }
FA_HD int imax(int a, int b) { return a > b ? a : b; }

// `sk` is the number of keys of this (batch, head): p.Sk for contiguous K/V, the
// sequence's own length for a paged cache.
FA_HD Range key_range(int m0, int m1, int BN, int sk, const PrefillParams& p, int bh) {
  (void)bh;
  const int nnb = (sk + BN - 1) / BN;
  Range r{0, 0, nnb};
  if (m0 >= m1 || nnb == 0) return Range{0, 0, 0};
  if (p.mask_mode == FA_MASK_NONE) return r;
  if (p.mask_mode == FA_MASK_BLOCK_SPARSE) return r;  // every block (see key_range_sparse)
  const int delta = sk - p.Sq;
  const int r_lo = m0 + delta;      // key position of the first row
  const int r_hi = m1 - 1 + delta;  // key position of the last row
  if (p.mask_mode == FA_MASK_BAND) {  // keys [r_lo - w, r_hi + w], clipped to [0, sk)
    const long long k_lo = static_cast<long long>(r_lo) - p.window;
    const long long k_hi = static_cast<long long>(r_hi) + p.window;
    if (k_hi < 0 || k_lo >= sk) return Range{0, 0, 0};
    const int lo = k_lo > 0 ? static_cast<int>(k_lo) : 0;
    const int hi = k_hi < sk - 1 ? static_cast<int>(k_hi) : sk - 1;
    return Range{0, lo / BN, hi / BN + 1};
  }
  if (p.mask_mode == FA_MASK_PREFIX_LM) {  // keys [0, max(n_global, r_hi + 1)), clipped
    const int keys = imin(sk, imax(p.n_global, r_hi + 1));
    return keys > 0 ? Range{0, 0, (keys + BN - 1) / BN} : Range{0, 0, 0};
  }
  if (r_hi < 0) return Range{0, 0, 0};
  r.b_end = imin(nnb, r_hi / BN + 1);
  if (p.mask_mode == FA_MASK_CAUSAL_WINDOW) {
    const int band_lo = imax(0, r_lo - p.window + 1);
    r.b_start = imin(band_lo / BN, r.b_end);
    const int g_keys = imin(imin(p.n_global, r_hi + 1), sk);
    r.a_end = g_keys > 0 ? (g_keys + BN - 1) / BN : 0;
    if (r.a_end >= r.b_start) {  // the two ranges touch: one range [0, b_end)
      r.a_end = 0;
      r.b_start = 0;
    }
  }
  return r;
}

FA_HD int range_count(const Range& r) { return r.a_end + r.b_end - r.b_start; }
// The key block visited after block nb (the first one for nb = -1); callers ask for no
// more than range_count blocks.
FA_HD int range_next(const Range& r, int nb) {
  const int t = nb + 1;
  return (t >= r.a_end && t < r.b_start) ? r.b_start : t;
}
FA_HD bool range_has(const Range& r, int nb) {
  return nb < r.a_end || (nb >= r.b_start && nb < r.b_end);
}

#if defined(__CUDACC__)
// Block-sparse ranges: the layout rows of the query blocks of [m0, m1) (at most two).
__device__ __forceinline__ SparseRange key_range_sparse(int m0, int m1, int BN, int sk,
                                                        const PrefillParams& p, int bh) {
  const int nnb = (sk + BN - 1) / BN;
  if (m0 >= m1 || nnb == 0) return SparseRange{0, 0, 0, nullptr, nullptr, 0};
  const uint8_t* head = p.layout + static_cast<size_t>(bh % p.H) * p.lnqb * p.lnkb;
  const uint8_t* la = head + static_cast<size_t>(m0 / 128) * p.lnkb;
  return SparseRange{0, 0, nnb, la, m1 - m0 > 128 ? la + p.lnkb : nullptr, BN == 64 ? 1 : 0};
}
__device__ __forceinline__ bool range_vis(const SparseRange& r, int nb) {
  return (r.la[nb >> r.shift] | (r.lb ? r.lb[nb >> r.shift] : 0)) != 0;
}
__device__ __forceinline__ int range_count(const SparseRange& r) {
  int n = 0;
  for (int nb = 0; nb < r.b_end; ++nb) n += range_vis(r, nb);
  return n;
}
__device__ __forceinline__ int range_next(const SparseRange& r, int nb) {
  int t = nb + 1;
  while (t < r.b_end && !range_vis(r, t)) ++t;
  return t;
}
__device__ __forceinline__ bool range_has(const SparseRange& r, int nb) {
  return r.la && nb >= 0 && nb < r.b_end && range_vis(r, nb);
}
#endif

// Work item t -> (batch*head, query block). Order: groups of `group_heads` heads; inside
// a group, query blocks from the last (most keys under a causal mask) to the first;
// inside that, the heads of the group.
FA_HD void item_coords(int t, const PrefillParams& p, int& bh, int& mb) {
  const int per_group = p.group_heads * p.nmb;
  const int g = t / per_group;
  const int gsize = imin(p.group_heads, p.BH - g * p.group_heads);
  const int rem = t - g * per_group;
  mb = p.nmb - 1 - rem / gsize;
  bh = g * p.group_heads + rem % gsize;
}

// Snake assignment of items to persistent CTAs: round r covers items [r*G, r*G+G), walked
// forwards on even rounds and backwards on odd ones.
FA_HD int item_of_round(int r, int G, int cta) { return r * G + ((r & 1) ? (G - 1 - cta) : cta); }

// Per-CTA item lists, passed to the kernel in its parameter space. CTA c runs
// items[offs[c]] .. items[offs[c+1]-1] in that order. When `enabled` is 0 (more CTAs or
// items than fit) the kernel falls back to the snake order above.
constexpr int kSchedMaxCtas = 192;
constexpr int kSchedMaxItems = 14336;
struct PrefillSched {
  int32_t enabled;
  uint16_t offs[kSchedMaxCtas + 1];
  uint16_t items[kSchedMaxItems];
};

// The k-th item of CTA `cta`: false when it has none left; t = -1 for an empty snake slot.
FA_HD bool item_at(const PrefillSched& s, const PrefillParams& p, int cta, int G, int k, int& t) {
  if (s.enabled) {
    const int i = s.offs[cta] + k;
    if (i >= s.offs[cta + 1]) return false;
    t = s.items[i];
    return true;
  }
  if (k * G >= p.total_items) return false;
  t = item_of_round(k, G, cta);
  if (t >= p.total_items) t = -1;
  return true;
}

}  // namespace fa
