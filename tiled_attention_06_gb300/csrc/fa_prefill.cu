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
// Roles inside one CTA (6 warps):
//   warps 0-3  softmax: one thread per query row (= TMEM lane). Loads S from TMEM,
//              masks partial tiles, keeps m and l, writes P (16-bit) back into the
//              S columns of TMEM, lazily rescales O, and runs the epilogue.
//   warp 4     TMA producer: Q once per work item, then K and V tiles through the
//              ring in exactly the order the MMA warp consumes them.
//   warp 5     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM S buffers,
//              then O += P_j V_j with P read from TMEM.
// TMEM columns: S0 [0,BN), S1 [BN,2BN), O [2BN, 2BN+D).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <climits>
#include <cstdint>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kBM = 128;
constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kTau = 8.0f;  // lazy-rescale threshold, log2 units
constexpr uint32_t kSmemLimit = 232448;  // 227 KB opt-in dynamic shared memory per CTA

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p *= 2;
  return p;
}

template <int D, int BN>
struct Cfg {
  static constexpr int KCH = D / 64;                 // 128-byte chunks along d
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int TILE_BYTES = BN * D * 2;      // one K or one V tile
  static constexpr int Q_CHUNK = kBM * 128;          // bytes per d-chunk of Q
  static constexpr int T_CHUNK = BN * 128;           // bytes per d-chunk of a K/V tile
  static constexpr int BAR_BYTES = 1024;
  static constexpr int NSLOT_FIT = (int)((kSmemLimit - 1024 - BAR_BYTES - Q_BYTES) / TILE_BYTES);
  static constexpr int NSLOT = NSLOT_FIT > 8 ? 8 : NSLOT_FIT;
  static constexpr int SMEM = 1024 /*align slack*/ + Q_BYTES + NSLOT * TILE_BYTES + BAR_BYTES;
  static constexpr int TMEM_COLS = pow2_at_least(2 * BN + D);
  static constexpr int O_COL = 2 * BN;
  static_assert(NSLOT >= 2, "shared memory ring too small");
  static_assert(SMEM <= (int)kSmemLimit, "shared memory over budget");
};

struct Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_empty, final_mma;
  uint32_t tmem_base;
  uint32_t abort;
};

// One work item: a block of kBM query rows of one (batch, head), and the key blocks
// it visits: [0, a_end) then [b_start, b_end). a_end <= b_start.
struct Item {
  int bh, mb, a_end, b_start, b_end, n;
};


// Key-block ranges of query block mb (closed form of the mask; every block in the
// ranges holds at least one visible pair, every block outside holds none).
template <int BN>
__device__ __forceinline__ Item make_item(int t, const PrefillParams& p) {
  Item it;
  // order: groups of `group_heads` (batch, head) pairs; inside a group, query blocks
  // from the last (most keys under a causal mask) to the first; inside that, heads.
  const int per_group = p.group_heads * p.nmb;
  const int g = t / per_group;
  const int gsize = min(p.group_heads, p.BH - g * p.group_heads);
  const int rem = t - g * per_group;
  it.mb = p.nmb - 1 - rem / gsize;
  it.bh = g * p.group_heads + rem % gsize;
  const int delta = p.Sk - p.Sq;
  const int m0 = it.mb * kBM;
  const int m1 = min(m0 + kBM, p.Sq);
  const int r_lo = m0 + delta;       // key position of the first row
  const int r_hi = m1 - 1 + delta;   // key position of the last valid row
  const int nnb = p.nnb;
  it.a_end = 0;
  it.b_start = 0;
  it.b_end = nnb;
  if (p.mask_mode != FA_MASK_NONE) {
    if (r_hi < 0) {
      it.b_end = 0;
    } else {
      it.b_end = min(nnb, r_hi / BN + 1);
      if (p.mask_mode == FA_MASK_CAUSAL_WINDOW) {
        const int band_lo = max(0, r_lo - p.window + 1);
        it.b_start = min(band_lo / BN, it.b_end);
        const int g_keys = min(min(p.n_global, r_hi + 1), p.Sk);
        it.a_end = g_keys > 0 ? (g_keys + BN - 1) / BN : 0;
        if (it.a_end >= it.b_start) {  // the ranges touch: one range [0, b_end)
          it.a_end = 0;
          it.b_start = 0;
        }
      }
    }
  }
  it.n = it.a_end + (it.b_end - it.b_start);
  return it;
}

__device__ __forceinline__ int tile_nb(const Item& it, int t) {
  return t < it.a_end ? t : it.b_start + (t - it.a_end);
}

// True when every (row, key) pair of the tile is in range and visible.
template <int BN>
__device__ __forceinline__ bool tile_full(const Item& it, int nb, const PrefillParams& p) {
  const int m0 = it.mb * kBM, n0 = nb * BN, n1 = n0 + BN;
  if (m0 + kBM > p.Sq || n1 > p.Sk) return false;
  if (p.mask_mode == FA_MASK_NONE) return true;
  const int delta = p.Sk - p.Sq;
  const int r_lo = m0 + delta, r_hi = m0 + kBM - 1 + delta;
  if (n1 - 1 > r_lo) return false;
  if (p.mask_mode == FA_MASK_CAUSAL) return true;
  return n1 <= p.n_global || r_hi - max(n0, p.n_global) < p.window;
}

template <int D, int BN, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = Cfg<D, BN>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sRing = base + C::Q_BYTES;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::Q_BYTES + C::NSLOT * C::TILE_BYTES);
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
  if (warp == kTmaWarp && lane == 0) {
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

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t pos = 0, ii = 0;
      uint32_t fills[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      bool ok = true;
      for (int r = 0; ok; ++r) {
        if (r * G >= p.total_items) break;
        const int t = r * G + ((r & 1) ? (G - 1 - cta) : cta);
        if (t >= p.total_items) continue;
        const Item it = make_item<BN>(t, p);
        if (it.n == 0) continue;
        if (ii > 0 && !(ok = mbar_wait(B(bars->q_empty), (ii - 1) & 1, wc))) break;
        mbar_arrive_expect_tx(B(bars->q_full), C::Q_BYTES);
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sQ + c * C::Q_CHUNK, &tmQ, B(bars->q_full), c * 64, it.mb * kBM, it.bh);
        // consumption order: K0, then for each j: K(j+1) (if any), V(j)
        for (int s = 0; s < 2 * it.n && ok; ++s) {
          int tile, is_v;
          if (s == 0) {
            tile = 0;
            is_v = 0;
          } else if (s == 2 * it.n - 1) {
            tile = it.n - 1;
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
          const int n0 = tile_nb(it, tile) * BN;
          const void* map = is_v ? (const void*)&tmV : (const void*)&tmK;
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(dst + c * C::T_CHUNK, map, B(bars->full[slot]), c * 64, n0, it.bh);
          fills[slot] = use + 1;
          ++pos;
        }
        ++ii;
      }
      if (!ok) {
        // wind down: let every load this thread issued land before the CTA exits
        for (int s = 0; s < C::NSLOT; ++s)
          if (fills[s] > 0) {
            WaitCtx w2 = wc;
            volatile uint32_t zero = 0;
            w2.abort = &zero;
            mbar_wait(B(bars->full[s]), (fills[s] - 1) & 1, w2);
          }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_f16(BF16, kBM, BN, false);
      constexpr uint32_t idO = idesc_f16(BF16, kBM, D, true);
      uint32_t pos = 0, ii = 0, tc = 0;
      bool ok = true;
      auto issue_s = [&](uint32_t sbuf, uint32_t slot) {
        const uint32_t kb = sRing + slot * C::TILE_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t a = smem_desc_sw128(sQ + (kk / 4) * C::Q_CHUNK + (kk % 4) * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(kb + (kk / 4) * C::T_CHUNK + (kk % 4) * 32, 16, 1024);
          umma_ss(tmem + sbuf * BN, a, b, idS, kk > 0);
        }
      };
      for (int r = 0; ok; ++r) {
        if (r * G >= p.total_items) break;
        const int t = r * G + ((r & 1) ? (G - 1 - cta) : cta);
        if (t >= p.total_items) continue;
        const Item it = make_item<BN>(t, p);
        if (it.n == 0) continue;
        if (!(ok = mbar_wait(B(bars->q_full), ii & 1, wc))) break;
        tc_fence_after();
        {  // S_0
          const int slot = pos % C::NSLOT;
          if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
          tc_fence_after();
          issue_s(tc & 1, slot);
          umma_commit(B(bars->s_full[tc & 1]));
          umma_commit(B(bars->empty[slot]));
          ++pos;
          if (it.n == 1) umma_commit(B(bars->q_empty));
        }
        for (int j = 0; j < it.n && ok; ++j) {
          if (j + 1 < it.n) {  // S_{j+1} into the other buffer while softmax works on S_j
            const int slot = pos % C::NSLOT;
            if (!(ok = mbar_wait(B(bars->full[slot]), (pos / C::NSLOT) & 1, wc))) break;
            tc_fence_after();
            issue_s((tc + 1) & 1, slot);
            umma_commit(B(bars->s_full[(tc + 1) & 1]));
            umma_commit(B(bars->empty[slot]));
            ++pos;
            if (j + 2 == it.n) umma_commit(B(bars->q_empty));
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
          const uint32_t vb = sRing + slot * C::TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint64_t b = smem_desc_sw128(vb + kk * 16 * 128, C::T_CHUNK, 1024);
            umma_ts(tmem + C::O_COL, tmem + (tc & 1) * BN + kk * 8, b, idO, (j > 0 || kk > 0));
          }
          umma_commit(B(bars->pv_done[tc & 1]));
          umma_commit(B(bars->empty[slot]));
          ++pos;
          ++tc;
        }
        ++ii;
      }
      // every MMA issued by this thread completes before TMEM is released
      umma_commit(B(bars->final_mma));
      WaitCtx w2 = wc;
      volatile uint32_t zero = 0;
      w2.abort = &zero;
      mbar_wait(B(bars->final_mma), 0, w2);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int row = warp * 32 + lane;  // TMEM lane and query row inside the tile
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int delta = p.Sk - p.Sq;
    uint32_t ii = 0, tc = 0;
    bool ok = true;
    for (int r = 0; ok; ++r) {
      if (r * G >= p.total_items) break;
      const int t = r * G + ((r & 1) ? (G - 1 - cta) : cta);
      if (t >= p.total_items) continue;
      const Item it = make_item<BN>(t, p);
      const int qrow = it.mb * kBM + row;
      const size_t orow = static_cast<size_t>(it.bh) * p.Sq + qrow;
      if (it.n == 0) {  // nothing visible: O = 0, LSE = -inf
        if (qrow < p.Sq) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow * D);
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          if (p.lse) p.lse[orow] = -INFINITY;
        }
        continue;
      }
      const int pos_q = qrow + delta;  // key position of this query
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < it.n; ++j) {
        const int nb = tile_nb(it, j);
        const int n0 = nb * BN;
        const bool full = tile_full<BN>(it, nb, p);
        ok = mbar_wait(B(bars->s_full[tc & 1]), (tc >> 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        uint32_t s[BN];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tmem_ld32(t_lane + (tc & 1) * BN + c * 32, s + c * 32);
        tmem_ld_wait<BN>(s);
        if (p.trace && threadIdx.x == 0)
          atomicAdd(p.trace + (static_cast<size_t>(it.bh) * p.nmb + it.mb) * p.nnb + nb,
                    16 + (full ? 2 : 1));
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
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < BN; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
        const float m_tile = mx * p.sl2;
        const float m_new = fmaxf(m_ref, m_tile);
        const bool need = (m_ref != -INFINITY) && (m_new > m_ref + kTau);
        if (m_ref == -INFINITY) m_ref = m_new;
        if (__any_sync(0xffffffffu, need)) {
          // O must hold every earlier P V product before it is rescaled
          const uint32_t pc = tc - 1;
          ok = mbar_wait(B(bars->pv_done[pc & 1]), (pc >> 1) & 1, wc);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          tc_fence_after();
          const float alpha = need ? ex2_approx(m_ref - m_new) : 1.f;
          if (need) {
            l *= alpha;
            m_ref = m_new;
          }
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld32(t_lane + C::O_COL + c * 32, ov);
            tmem_ld_wait<32>(ov);
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(t_lane + C::O_COL + c * 32, ov);
          }
        }
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < BN; c += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(s[c]), p.sl2, -m_use));
          const float p1 = ex2_approx(fmaf(__uint_as_float(s[c + 1]), p.sl2, -m_use));
          lsum += p0 + p1;
          uint32_t packed;
          if constexpr (BF16) {
            __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
            packed = *reinterpret_cast<uint32_t*>(&h);
          } else {
            __half2 h = __floats2half2_rn(p0, p1);
            packed = *reinterpret_cast<uint32_t*>(&h);
          }
          s[c / 2] = packed;
        }
        l += lsum;
#pragma unroll
        for (int c = 0; c < BN / 64; ++c) tmem_st32(t_lane + (tc & 1) * BN + c * 32, s + c * 32);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(B(bars->p_full[tc & 1]));
        ++tc;
      }
      if (!ok) break;
      // ---------------------------------------------------------- epilogue
      {
        const uint32_t pc = tc - 1;
        ok = mbar_wait(B(bars->pv_done[pc & 1]), (pc >> 1) & 1, wc);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld32(t_lane + C::O_COL + c * 32, ov);
          tmem_ld_wait<32>(ov);
          if (qrow < p.Sq) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float a = __uint_as_float(ov[2 * e]) * inv_l;
              const float b = __uint_as_float(ov[2 * e + 1]) * inv_l;
              if constexpr (BF16) {
                __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                pk[e] = *reinterpret_cast<uint32_t*>(&h);
              } else {
                __half2 h = __floats2half2_rn(a, b);
                pk[e] = *reinterpret_cast<uint32_t*>(&h);
              }
            }
            uint4* dst =
                reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + orow * D + c * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
          }
        }
        if (qrow < p.Sq && p.lse)
          p.lse[orow] = l > 0.f ? (m_ref + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
        tc_fence_before();
        mbar_arrive(B(bars->o_empty));
      }
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
cudaError_t launch_prefill_t(const PrefillLaunch& L, cudaStream_t stream) {
  using C = Cfg<D, BN>;
  auto kern = prefill_kernel<D, BN, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  kern<<<L.grid, kThreads, C::SMEM, stream>>>(L.tmQ, L.tmK, L.tmV, L.p);
  return cudaGetLastError();
}

}  // namespace

int prefill_block_m() { return kBM; }

cudaError_t launch_prefill(const PrefillLaunch& L, int D, int BN, bool bf16, cudaStream_t stream) {
#define FA_CASE(d_, bn_, bf_) \
  if (D == d_ && BN == bn_ && bf16 == bf_) return launch_prefill_t<d_, bn_, bf_>(L, stream);
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
