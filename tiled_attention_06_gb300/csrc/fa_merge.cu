// Merge of two attention results over disjoint key sets for the same queries.
//
// Splitting one attention into several calls with separate masks and combining them is
// exact ("ascend-transformer-boost 实战" (ai6s.net), scenario 4: the multimodal attention
// is cut into vision-internal, text-internal and text-to-vision calls with identical
// results). With each part normalised and carrying its log-sum-exp, the combination is
// the same running-max recurrence as the tiled forward (ops-transformer overview,
// section 二.1):
//   M = max(lse_a, lse_b),  w_x = exp(lse_x - M),
//   O = (w_a O_a + w_b O_b) / (w_a + w_b),  LSE = M + ln(w_a + w_b).
// A part with LSE = -inf (no visible key) contributes nothing; if both are empty the row
// is O = 0, LSE = -inf.
//
// Element-wise and HBM-bound: one group of d/8 threads per row, 16-byte loads and stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

template <bool BF16>
__device__ __forceinline__ void to_float8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t;
    if constexpr (BF16)
      t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
    else
      t = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <bool BF16>
__device__ __forceinline__ uint4 from_float8(const float* f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    } else {
      __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) merge_kernel(const uint4* __restrict__ oa,
                                                    const float* __restrict__ la,
                                                    const uint4* __restrict__ ob,
                                                    const float* __restrict__ lb, uint4* o,
                                                    float* lse, int64_t rows) {
  constexpr int TPR = D / 8;  // threads per row
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < rows * TPR; i += nthreads) {
    const int64_t r = i / TPR;
    const float a = la[r], b = lb[r];
    const float M = fmaxf(a, b);
    float wa = 0.f, wb = 0.f;
    if (M != -INFINITY) {
      wa = __expf(a - M);
      wb = __expf(b - M);
    }
    const float den = wa + wb;
    float fa_[8], fb_[8], out[8];
    to_float8<BF16>(oa[i], fa_);
    to_float8<BF16>(ob[i], fb_);
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = (wa * fa_[e] + wb * fb_[e]) * inv;
    o[i] = from_float8<BF16>(out);
    if (lse && i % TPR == 0) lse[r] = den > 0.f ? M + __logf(den) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_merge(const void* oa, const float* la, const void* ob, const float* lb,
                         void* o, float* lse, int64_t rows, int D, bool bf16, int sms,
                         cudaStream_t stream) {
  const int64_t work = rows * (D / 8);
  int64_t blocks = (work + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 g(static_cast<unsigned>(blocks));
  auto* a = static_cast<const uint4*>(oa);
  auto* b = static_cast<const uint4*>(ob);
  auto* out = static_cast<uint4*>(o);
  if (D == 64 && !bf16) merge_kernel<64, false><<<g, 256, 0, stream>>>(a, la, b, lb, out, lse, rows);
  else if (D == 64) merge_kernel<64, true><<<g, 256, 0, stream>>>(a, la, b, lb, out, lse, rows);
  else if (D == 128 && !bf16) merge_kernel<128, false><<<g, 256, 0, stream>>>(a, la, b, lb, out, lse, rows);
  else if (D == 128) merge_kernel<128, true><<<g, 256, 0, stream>>>(a, la, b, lb, out, lse, rows);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace fa
