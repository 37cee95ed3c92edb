// Paged-KV decode for sm_103a: one query token per sequence against a KV cache held in
// fixed-size pages ("ascend-transformer-boost 实战" (ai6s.net), scenario 2: pages of 256
// tokens, taken on demand; loads of the next K/V batch overlap compute).
//
// The work is HBM-bound (each cached token is read once, 4*d bytes per head for K and V,
// for 4*d multiply-adds), so it runs on the CUDA cores with wide coalesced loads:
//   kernel 1 (split): one CTA per (b*H + h, split). A split is a run of `pages_per_split` pages
//     of one sequence and one head. A group of d/16 lanes owns one token row: each lane
//     loads 32 bytes of K and of V in one access (d/8 lanes and 16 bytes when a pool is
//     only 16-byte aligned), the q.k dot is reduced with xor-shuffles inside the group,
//     and the group keeps an online softmax state (m, l, acc) in registers, several
//     tokens in flight per lane. The groups are merged in shared memory and the split
//     writes its FP32 partial (acc, m, l) to the workspace.
//   kernel 2 (merge): per (b, h), M = max m_s, L = sum l_s 2^(m_s - M),
//     O = sum 2^(m_s - M) acc_s / L, LSE = (M + log2 L) ln 2, formed in one pass over the
//     splits with the same running-max recurrence as the tiled forward (ops-transformer
//     overview, section 二.1).
// Scores are kept in log2 units (q is pre-multiplied by scale*log2(e)).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const void* ptr) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}

// 32 bytes in one access (sm_100 family); the address must be 32-byte aligned.
__device__ __forceinline__ void ld_stream32(const void* ptr, uint4& a, uint4& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                 "=r"(b.w)
               : "l"(ptr));
}

// A context length outside [0, page_size * max_pages] would index past the sequence's
// block-table row: it is clamped (and reported once) instead.
__device__ __forceinline__ int clamp_ctx(const DecodeParams& p, int b, bool report) {
  const int c = p.ctx_lens[b];
  const int cmax = p.page_size * p.max_pages;
  if (c >= 0 && c <= cmax) return c;
  if (report) atomicOr(p.status, FA_DEV_BAD_PAGE);
  return c < 0 ? 0 : cmax;
}

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      float2 t = __bfloat1622float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

template <int D, bool BF16, int EPL>
__global__ void __launch_bounds__(kDecThreads) decode_split_kernel(const DecodeParams p) {
  constexpr int NV = EPL / 8;            // 16-byte vectors per lane per token row (EPL elements)
  constexpr int LPT = D / EPL;           // lanes per token row
  constexpr int TPW = 32 / LPT;          // token groups per warp
  constexpr int NG = kDecWarps * TPW;    // token groups per CTA
  __shared__ float sm_m[NG], sm_l[NG];
  __shared__ float sm_acc[NG][D];

  const int split = blockIdx.x % p.nsplit_max;  // consecutive CTAs walk one sequence
  const int bh = blockIdx.x / p.nsplit_max;
  const int b = bh / p.H, h = bh - (bh / p.H) * p.H;
  const int ctx = clamp_ctx(p, b, threadIdx.x == 0 && split == 0);
  const int span = p.pages_per_split * p.page_size;
  const int t0 = min(split * span, ctx);
  const int t1 = min(t0 + span, ctx);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    if (p.trace_splits) {
      int32_t* ts = p.trace_splits + (static_cast<size_t>(bh) * p.nsplit_max + split) * 2;
      ts[0] = t0;
      ts[1] = t1;
    }
    if (p.trace_pages && t0 < t1) {
      for (int lp = t0 / p.page_size; lp * p.page_size < t1; ++lp)
        p.trace_pages[static_cast<size_t>(bh) * p.max_pages + lp] =
            p.block_table[static_cast<size_t>(b) * p.max_pages + lp];
    }
  }
  if (t0 >= t1) return;  // past the end of this sequence: no partial

  const int grp = warp * TPW + lane / LPT;  // token group of this lane
  const int cl = lane % LPT;                // which EPL elements of d
  float qf[EPL];
#pragma unroll
  for (int v = 0; v < NV; ++v) {
    const uint4 qu = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) +
                                                     static_cast<size_t>(bh) * D + cl * EPL + 8 * v);
    unpack8<BF16>(qu, qf + 8 * v);
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) qf[e] *= p.sl2;
  const int32_t* table = p.block_table + static_cast<size_t>(b) * p.max_pages;
  const uint16_t* kp = static_cast<const uint16_t*>(p.k_pages);
  const uint16_t* vp = static_cast<const uint16_t*>(p.v_pages);
  const size_t head_off = static_cast<size_t>(h) * p.page_size * D + cl * EPL;
  const size_t page_stride = static_cast<size_t>(p.H) * p.page_size * D;

  float m = -INFINITY, l = 0.f, acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  bool bad = false;

  // the loop bound is warp-uniform so that every lane takes part in every shuffle
  const int sub = lane / LPT;
  for (int wb = t0 + warp * TPW; wb < t1; wb += NG * kUnroll) {
    uint4 ku[kUnroll][NV], vu[kUnroll][NV];
    bool live[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int t = wb + sub + u * NG;
      live[u] = t < t1;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        ku[u][v] = make_uint4(0, 0, 0, 0);
        vu[u][v] = make_uint4(0, 0, 0, 0);
      }
      if (live[u]) {
        const int lp = t / p.page_size;
        const int phys = __ldg(table + lp);
        if (phys < 0 || phys >= p.num_pages) {
          live[u] = false;
          bad = true;
        } else {
          const size_t off = phys * page_stride + head_off +
                             static_cast<size_t>(t - lp * p.page_size) * D;
          if constexpr (NV == 2) {
            ld_stream32(kp + off, ku[u][0], ku[u][1]);
            ld_stream32(vp + off, vu[u][0], vu[u][1]);
          } else {
            ku[u][0] = ld_stream(kp + off);
            vu[u][0] = ld_stream(vp + off);
          }
        }
      }
    }
    float s[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float dot = 0.f;
#pragma unroll
      for (int v = 0; v < NV; ++v) {
        float kf[8];
        unpack8<BF16>(ku[u][v], kf);
#pragma unroll
        for (int e = 0; e < 8; ++e) dot = fmaf(qf[8 * v + e], kf[e], dot);
      }
#pragma unroll
      for (int off = LPT / 2; off > 0; off /= 2) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      s[u] = live[u] ? dot : -INFINITY;
    }
    float mt = s[0];
#pragma unroll
    for (int u = 1; u < kUnroll; ++u) mt = fmaxf(mt, s[u]);
    const float m_new = fmaxf(m, mt);
    if (m_new != -INFINITY) {
      const float alpha = ex2_approx(m - m_new);  // m = -inf gives 0
      l *= alpha;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= alpha;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const float pu = ex2_approx(s[u] - m_new);
        l += pu;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          float vf[8];
          unpack8<BF16>(vu[u][v], vf);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[8 * v + e] = fmaf(pu, vf[e], acc[8 * v + e]);
        }
      }
      m = m_new;
    }
  }
  if (bad) atomicOr(p.status, FA_DEV_BAD_PAGE);

  // merge the token groups of this CTA
  if (cl == 0) {
    sm_m[grp] = m;
    sm_l[grp] = l;
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) sm_acc[grp][cl * EPL + e] = acc[e];
  __syncthreads();
  float* out = p.part + (static_cast<size_t>(bh) * p.nsplit_max + split) * (D + 2);
  for (int e = threadIdx.x; e < D; e += kDecThreads) {
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < NG; ++g) M = fmaxf(M, sm_m[g]);
    float a = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int g = 0; g < NG; ++g) {
        const float w = ex2_approx(sm_m[g] - M);
        a = fmaf(w, sm_acc[g][e], a);
        L = fmaf(w, sm_l[g], L);
      }
    }
    out[e] = a;
    if (e == 0) {
      out[D] = M;
      out[D + 1] = L;
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeParams p) {
  constexpr int kBatch = 8;  // splits whose loads are in flight together
  const int bh = blockIdx.x;
  const int b = bh / p.H;
  const int e = threadIdx.x;
  const int ctx = clamp_ctx(p, b, false);
  const int span = p.pages_per_split * p.page_size;
  const int nsplit = (ctx + span - 1) / span;
  const float* part = p.part + static_cast<size_t>(bh) * p.nsplit_max * (D + 2);
  // One pass with a running maximum (the same recurrence as inside a split), the partials
  // of kBatch splits loaded before any is used, so that the pass waits for one load
  // latency per batch rather than two per split.
  float M = -INFINITY, a = 0.f, L = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += kBatch) {
    float ms[kBatch], ls[kBatch], as[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      ls[u] = 0.f;
      ms[u] = -INFINITY;
      as[u] = 0.f;
      if (s0 + u < nsplit) {
        const float* ps = part + static_cast<size_t>(s0 + u) * (D + 2);
        ms[u] = ps[D];
        ls[u] = ps[D + 1];
        as[u] = ps[e];
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (ls[u] > 0.f) {  // a split with no visible token adds nothing
        const float m_new = fmaxf(M, ms[u]);
        const float c = ex2_approx(M - m_new);  // M = -inf gives 0
        const float w = ex2_approx(ms[u] - m_new);
        a = fmaf(w, as[u], a * c);
        L = fmaf(w, ls[u], L * c);
        M = m_new;
      }
    }
  }
  const float o = L > 0.f ? a / L : 0.f;
  uint16_t bits;
  if constexpr (BF16) {
    __nv_bfloat16 v = __float2bfloat16_rn(o);
    bits = *reinterpret_cast<uint16_t*>(&v);
  } else {
    __half v = __float2half_rn(o);
    bits = *reinterpret_cast<uint16_t*>(&v);
  }
  static_cast<uint16_t*>(p.o)[static_cast<size_t>(bh) * D + e] = bits;
  if (e == 0 && p.lse)
    p.lse[bh] = L > 0.f ? (M + lg2_approx(L)) * 0.69314718055994531f : -INFINITY;
}

template <int D, bool BF16>
cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  // 32 bytes per lane per token row when both pools are 32-byte aligned, else 16
  if ((reinterpret_cast<uintptr_t>(p.k_pages) | reinterpret_cast<uintptr_t>(p.v_pages)) % 32 == 0)
    decode_split_kernel<D, BF16, 16><<<p.nsplit_max * p.B * p.H, kDecThreads, 0, stream>>>(p);
  else
    decode_split_kernel<D, BF16, 8><<<p.nsplit_max * p.B * p.H, kDecThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_merge_kernel<D, BF16><<<p.B * p.H, D, 0, stream>>>(p);
  return cudaGetLastError();
}

// A barrier that nothing ever completes: the bounded wait must run out and report.
__global__ void selftest_timeout_kernel(uint32_t* status, uint64_t timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
    const WaitCtx w{&abort_flag, status, timeout_ns};
    mbar_wait(smem_u32(&bar), 0, w);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int D, bool bf16, cudaStream_t stream) {
  if (D == 64) return bf16 ? launch_decode_t<64, true>(p, stream) : launch_decode_t<64, false>(p, stream);
  if (D == 128)
    return bf16 ? launch_decode_t<128, true>(p, stream) : launch_decode_t<128, false>(p, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_selftest_timeout(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
  selftest_timeout_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa

// ---------------------------------------------------------------------------------------
// Paged decode without a caller-provided workspace (fa_decode_paged_noalloc).
//
// Some callers cannot hand the library a device buffer: a serving loop whose device
// memory budget is fixed when it starts, or a host program that owns every device
// allocation and gives its plug-ins no allocator. For them the split partials live in
// this file-scope array instead: 16 MiB of FP32, reserved on every GPU that loads the
// library and held until the process exits. Nothing here calls cudaMalloc or cudaFree.
//
// The array's name is only a host-side stand-in for the device object, so host code
// never passes it to a kernel directly: the first call on each device (with that device
// current) looks up the real device address with cudaGetSymbolAddress and keeps it.
// All calls on a device share the array and it keeps whatever the last call left;
// no part of it has to start at zero, because every partial the merge kernel reads is
// written by the split kernel earlier in the same call. Two calls whose kernels overlap
// on the GPU (for example on different streams) race on the array.
// ---------------------------------------------------------------------------------------
#include <mutex>

namespace fa {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

std::mutex g_noalloc_mu;
float* g_noalloc_ptr[64] = {};

}  // namespace

size_t noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

cudaError_t launch_decode_noalloc(const DecodeParams& p_in, int D, bool bf16,
                                  cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  float* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
      if (e != cudaSuccess) return e;
      g_noalloc_ptr[dev] = static_cast<float*>(addr);
    }
    scratch = g_noalloc_ptr[dev];
  }
  DecodeParams p = p_in;
  p.part = scratch;
  return launch_decode(p, D, bf16, stream);
}

}  // namespace fa
