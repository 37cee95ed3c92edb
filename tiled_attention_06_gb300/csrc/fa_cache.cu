// Appending new tokens to a paged KV cache ("ascend-transformer-boost 实战" (ai6s.net),
// scenario 2: the cache is cut into fixed-size pages and a sequence takes a new page when
// it grows). Token t of sequence b's new chunk goes to position ctx_b + t, i.e. to page
// block_table[b, (ctx_b + t) / page] at offset (ctx_b + t) % page; the caller has put the
// pages the chunk needs into the table. After the chunk, the rest of its last page is
// zero-filled: a paged prefill reads whole key tiles, and the slots past a sequence's end
// are then finite (their probabilities are exactly zero, and 0 times a finite value
// contributes nothing to O).
//
// A plain HBM copy: one CTA per (sequence, head, slice of kAppendRows positions), 16-byte
// loads and stores, so that a chunk of a few hundred tokens still spreads over several waves
// of CTAs.
#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kAppendRows = 64;  // cache positions per CTA

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        uint4* k_pages, uint4* v_pages,
                                                        const KvAppendParams p, int nslice) {
  const int bh = blockIdx.x / nslice, slice = blockIdx.x - (blockIdx.x / nslice) * nslice;
  const int b = bh / p.H, h = bh - b * p.H;
  const int cpt = p.d / 8;  // 16-byte chunks per token row
  const int cap = p.page_size * p.max_pages;
  int ctx = p.ctx_lens[b];
  int n = p.new_lens ? p.new_lens[b] : p.T;
  if (n > p.T) n = p.T;
  if (ctx < 0 || n < 0 || ctx + n > cap) {
    if (threadIdx.x == 0 && h == 0 && slice == 0) atomicOr(p.status, FA_DEV_BAD_PAGE);
    return;
  }
  if (n == 0) return;
  const int end = ctx + n;
  const int tail_end = ((end + p.page_size - 1) / p.page_size) * p.page_size;
  // this CTA's positions [r0, r1) of [ctx, tail_end): the new rows, then the zeroed tail
  const int r0 = ctx + slice * kAppendRows, r1 = min(r0 + kAppendRows, tail_end);
  if (r0 >= r1) return;
  const int32_t* table = p.block_table + static_cast<size_t>(b) * p.max_pages;
  const size_t src_row0 = static_cast<size_t>(bh) * p.T;
  const int total = (r1 - r0) * cpt;
#pragma unroll 4
  for (int i = threadIdx.x; i < total; i += blockDim.x) {
    const int pos = r0 + i / cpt, c = i - (i / cpt) * cpt;
    const int lp = pos / p.page_size;
    const int phys = table[lp];
    if (phys < 0 || phys >= p.num_pages) {
      atomicOr(p.status, FA_DEV_BAD_PAGE);
      continue;
    }
    const size_t dst = ((static_cast<size_t>(phys) * p.H + h) * p.page_size +
                        (pos - lp * p.page_size)) * cpt + c;
    if (pos < end) {
      const size_t src = (src_row0 + (pos - ctx)) * cpt + c;
      k_pages[dst] = k_new[src];
      v_pages[dst] = v_new[src];
    } else {
      k_pages[dst] = make_uint4(0, 0, 0, 0);
      v_pages[dst] = make_uint4(0, 0, 0, 0);
    }
  }
}

}  // namespace

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                             const KvAppendParams& p, cudaStream_t stream) {
  // a chunk covers at most T + page_size - 1 positions with its zeroed tail
  const int nslice = static_cast<int>(
      (static_cast<int64_t>(p.T) + p.page_size - 1 + kAppendRows - 1) / kAppendRows);
  const int64_t grid = static_cast<int64_t>(p.B) * p.H * nslice;
  if (grid > 0x7fffffff) return cudaErrorInvalidConfiguration;
  kv_append_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_pages), static_cast<uint4*>(v_pages), p, nslice);
  return cudaGetLastError();
}

}  // namespace fa
