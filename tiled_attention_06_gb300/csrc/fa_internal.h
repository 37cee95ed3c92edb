// Internal interface between the C-ABI layer (fa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "fa.h"

namespace fa {

// bits of the device status word
// FA_DEV_SMEM_BASE: a kernel found its dynamic shared memory too far from a 1024-byte
// boundary for its layout and did nothing.
enum : uint32_t { FA_DEV_TIMEOUT = 1u, FA_DEV_BAD_PAGE = 2u, FA_DEV_SMEM_BASE = 4u };

struct PrefillParams {
  void* o;            // [B,H,Sq,D] 16-bit (FP32 for FP32 inputs)
  float* lse;         // [B,H,Sq] or nullptr
  int BH, Sq, Sk;
  int nmb, nnb;       // query blocks (BM rows per work item), key blocks (BN keys)
  int mask_mode, window, n_global;
  float sl2;          // scale * log2(e)
  int group_heads;    // (batch, head) pairs per scheduling group
  int total_items;    // BH * nmb
  uint32_t* status;   // device status word
  uint64_t timeout_ns;
  int32_t* trace;     // optional [BH, ceil(Sq/128), nnb] visit log (16 + class per visit)
  int32_t* rescales;  // optional [BH, ceil(Sq/128)]: (row, key tile) pairs whose O was rescaled
  // Paged K/V (chunked prefill into a paged cache). block_table == nullptr: K and V are
  // contiguous [B,H,Sk,d]. Otherwise K/V tile rows come from pools [num_pages,H,page,d]
  // through block_table [B, max_pages], sequence b has seq_k[b] keys and Sk is only the
  // upper bound max_pages*page_size (used for nnb and for planning).
  const int32_t* block_table;
  const int32_t* seq_k;
  int H, page_size, max_pages, num_pages;
  // Block-sparse layout uint8 [H, lnqb, lnkb] (128 x 128 blocks), or nullptr.
  const uint8_t* layout;
  int lnqb, lnkb;
};

struct PrefillSched;  // fa_plan.h

struct PrefillLaunch {
  CUtensorMap tmQ, tmK, tmV;
  PrefillParams p;
  const PrefillSched* sched;  // host copy of the per-CTA item lists (passed by value)
  int grid;
};

int prefill_tile_rows();
cudaError_t launch_prefill(const PrefillLaunch& L, int D, int BN, int BM, bool bf16,
                           cudaStream_t stream);

// FP32 inputs. Step 1 splits Q, K and V (n8[t] groups of 8 elements each) into bf16 high
// and low planes; step 2 is the 256-row prefill kernel over those planes (tensor maps of
// [2*BH, S, d] bf16: plane bh the high parts, BH + bh the low parts) with key blocks of
// kSplitBlockN, writing FP32 O.
constexpr int kSplitBlockN = 64;
struct SplitArgs {
  const float* src[3];
  uint16_t* hi[3];
  uint16_t* lo[3];
  size_t n8[3];
};
cudaError_t launch_split_bf16(const SplitArgs& a, int sms, cudaStream_t stream);
cudaError_t launch_prefill_split(const PrefillLaunch& L, int D, cudaStream_t stream);

// Backward: what the kernels read besides the forward's parameters.
struct BwdParams {
  const float* lse;   // [B,H,Sq] natural-log LSE of the forward
  const float* dsum;  // [B,H,Sq] D_i = dO_i . O_i (written by the first kernel)
  float* dqacc;       // [B*H][ceil(Sq/4)][d][4] FP32 dQ accumulator (zeroed by the first kernel)
  void* dq;           // [B,H,Sq,d] 16-bit
  void* dk;           // [B,H,Sk,d]
  void* dv;
  float scale;
  int head_group;  // heads per group of the dK/dV kernel's launch order (1 <= head_group)
};

struct BwdLaunch {
  CUtensorMap tmQ, tmK, tmV, tmdO;
  PrefillParams p;  // sizes, mask, sl2, status, timeout (contiguous K/V)
  BwdParams b;
  const void* o;     // forward output [B,H,Sq,d]
  const void* dout;  // upstream gradient [B,H,Sq,d]
};

cudaError_t launch_backward(const BwdLaunch& L, int D, bool bf16, cudaStream_t stream);

struct DecodeParams {
  const void* q;            // [B,H,D]
  const void* k_pages;      // [num_pages,H,page_size,D]
  const void* v_pages;
  const int32_t* block_table;  // [B,max_pages]
  const int32_t* ctx_lens;     // [B]
  void* o;                  // [B,H,D]
  float* lse;               // [B,H] or nullptr
  float* part;              // workspace [B*H, nsplit_max, D+2] FP32 partials
  int B, H, page_size, max_pages, num_pages;
  int pages_per_split, nsplit_max;
  float sl2;                // scale * log2(e)
  uint32_t* status;
  int32_t* trace_pages;     // optional [B*H, max_pages]: physical page read per logical page
  int32_t* trace_splits;    // optional [B*H, nsplit_max, 2]: token range per split
};

cudaError_t launch_decode(const DecodeParams& p, int D, bool bf16, cudaStream_t stream);
// Decode with the split partials in the library's own file-scope scratch array.
size_t noalloc_scratch_bytes();
cudaError_t launch_decode_noalloc(const DecodeParams& p, int D, bool bf16, cudaStream_t stream);
cudaError_t launch_merge(const void* oa, const float* la, const void* ob, const float* lb,
                         void* o, float* lse, int64_t rows, int D, bool bf16, int sms,
                         cudaStream_t stream);
struct KvAppendParams {
  const int32_t* block_table;  // [B, max_pages]
  const int32_t* ctx_lens;     // [B] tokens already cached
  const int32_t* new_lens;     // [B] tokens to append (<= T), or nullptr for T each
  int B, H, T, d, page_size, max_pages, num_pages;
  uint32_t* status;
};

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                             const KvAppendParams& p, cudaStream_t stream);
cudaError_t launch_selftest_timeout(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace fa
