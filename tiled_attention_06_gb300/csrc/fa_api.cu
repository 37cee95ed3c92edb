// The C ABI (include/fa.h): argument validation, launch planning, TMA tensor-map
// encoding and the device status word. Every check here runs on the host before
// anything is launched; a rejected call launches nothing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <string>
#include <vector>

#include "fa.h"
#include "fa_bwd_tiles.h"
#include "fa_internal.h"
#include "fa_plan.h"

namespace {

__device__ uint32_t g_status_word;

thread_local std::string t_last_error = "no error";

fa_status fail(fa_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  uint32_t* status = nullptr;
};
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Per-device facts, looked up once per device with that device current.
fa_status device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device index %d", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    d.status = static_cast<uint32_t*>(p);
    d.ready = true;
  }
  *out = d;
  return FA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A [BH, S, D] tensor of 16-bit elements as a 3-D TMA map with 128-byte swizzle;
// one box is 64 elements of d by `rows` rows of one (batch, head).
fa_status make_map(CUtensorMap* m, const void* ptr, bool bf16, int D, int S, int BH, int rows) {
  auto enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S > 0 ? S : 1),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(S > 0 ? S : 1) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FA_OK;
}

// Per-CTA item lists for a persistent prefill launch. Items are taken in their numbering
// order (head groups, then query blocks from most keys to fewest) and each goes to the CTA
// that would be free first, with cost = visited key blocks + a fixed per-item overhead:
// the list schedule a dynamic work queue would produce, fixed in advance so that the
// kernel needs no global counter. Cached per shape; the kernel receives a copy at launch.
constexpr double kItemOverheadTiles = 2.0;
std::mutex g_plan_mu;
std::map<std::array<int, 11>, std::unique_ptr<fa::PrefillSched>> g_plans;

const fa::PrefillSched* plan_for(const fa::PrefillParams& p, int BM, int BN, int grid) {
  const std::array<int, 11> key{p.BH, p.Sq, p.Sk, BM, BN, p.mask_mode, p.window, p.n_global,
                                p.group_heads, grid, p.nmb};
  std::lock_guard<std::mutex> lock(g_plan_mu);
  auto it = g_plans.find(key);
  if (it != g_plans.end()) return it->second.get();
  if (g_plans.size() >= 256) g_plans.clear();  // launches copy their plan; old ones can go
  auto plan = std::make_unique<fa::PrefillSched>();
  std::memset(plan.get(), 0, sizeof(fa::PrefillSched));
  if (grid <= fa::kSchedMaxCtas && p.total_items <= fa::kSchedMaxItems) {
    using Slot = std::pair<double, int>;  // (busy until, cta)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
    for (int c = 0; c < grid; ++c) free_at.push({0.0, c});
    std::vector<std::vector<uint16_t>> lists(grid);
    for (int t = 0; t < p.total_items; ++t) {
      int bh, mb;
      fa::item_coords(t, p, bh, mb);
      const fa::Range r = fa::key_range(mb * BM, std::min(mb * BM + BM, p.Sq), BN, p.Sk, p, 0);
      const int n = fa::range_count(r);
      Slot s = free_at.top();
      free_at.pop();
      lists[s.second].push_back(static_cast<uint16_t>(t));
      s.first += n + kItemOverheadTiles;
      free_at.push(s);
    }
    int k = 0;
    for (int c = 0; c < grid; ++c) {
      plan->offs[c] = static_cast<uint16_t>(k);
      for (uint16_t t : lists[c]) plan->items[k++] = t;
    }
    plan->offs[grid] = static_cast<uint16_t>(k);
    plan->enabled = 1;
  }
  const fa::PrefillSched* out = plan.get();
  g_plans.emplace(key, std::move(plan));
  return out;
}

// The same list schedule with every item weighed by the key tiles it really visits, known
// on the host only when the caller gives what decides them there too: a paged prefill's
// sequence lengths (the plan otherwise weighs every item by the pool capacity) or a
// block-sparse layout (otherwise planned as dense). Items are taken longest first: over
// all items (`per_group` false: a paged prefill's heads have few items each, and the two
// of a head stay next to each other), or within each head group of the numbering
// (`per_group` true: the many items of a block-sparse head then still run together and
// share its K/V in L2; sorting them across groups measured 25 % slower). Only the
// assignment of items to CTAs changes, so the results are those of the unplanned call.
// Built per call (it depends on the data), into `plan`.
void plan_with_costs(const fa::PrefillParams& p, int grid, const std::vector<int>& cost,
                     bool per_group, fa::PrefillSched* plan) {
  std::memset(plan, 0, sizeof(fa::PrefillSched));
  if (grid > fa::kSchedMaxCtas || p.total_items > fa::kSchedMaxItems) return;
  std::vector<int> order(p.total_items);
  for (int t = 0; t < p.total_items; ++t) order[t] = t;
  const int span = per_group ? p.group_heads * p.nmb : p.total_items;  // items of a group
  for (int a = 0; a < p.total_items; a += span)
    std::stable_sort(order.begin() + a, order.begin() + std::min(a + span, p.total_items),
                     [&](int x, int y) { return cost[x] > cost[y]; });
  using Slot = std::pair<double, int>;  // (busy until, cta)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  for (int c = 0; c < grid; ++c) free_at.push({0.0, c});
  std::vector<std::vector<uint16_t>> lists(grid);
  for (int t : order) {
    Slot sl = free_at.top();
    free_at.pop();
    lists[sl.second].push_back(static_cast<uint16_t>(t));
    sl.first += cost[t] + kItemOverheadTiles;
    free_at.push(sl);
  }
  int k = 0;
  for (int c = 0; c < grid; ++c) {
    plan->offs[c] = static_cast<uint16_t>(k);
    for (uint16_t t : lists[c]) plan->items[k++] = t;
  }
  plan->offs[grid] = static_cast<uint16_t>(k);
  plan->enabled = 1;
}

// Key tiles of every item of a paged prefill, from the sequences' lengths (clamped to the
// pool capacity `cap`, as on the device).
std::vector<int> costs_from_lengths(const fa::PrefillParams& p, int BM, int BN,
                                    const int32_t* sk_host, int cap) {
  std::vector<int> cost(p.total_items);
  for (int t = 0; t < p.total_items; ++t) {
    int bh, mb;
    fa::item_coords(t, p, bh, mb);
    const int len = sk_host[bh / p.H];
    const int sk = len < 0 ? 0 : (len > cap ? cap : len);
    cost[t] = fa::range_count(fa::key_range(mb * BM, std::min(mb * BM + BM, p.Sq), BN, sk, p, 0));
  }
  return cost;
}

// Key tiles of every item of a block-sparse prefill, from the layout [H][lnqb][lnkb] (one
// byte per 128 x 128 block): the blocks on in any layout row the item's rows fall in, times
// the key tiles per layout block.
std::vector<int> costs_from_layout(const fa::PrefillParams& p, int BM, int BN,
                                   const uint8_t* layout) {
  std::vector<int> cost(p.total_items);
  const int per = FA_LAYOUT_BLOCK / BN;
  for (int t = 0; t < p.total_items; ++t) {
    int bh, mb;
    fa::item_coords(t, p, bh, mb);
    const int r0 = (mb * BM) / FA_LAYOUT_BLOCK;
    const int r1 = std::min((mb * BM + BM - 1) / FA_LAYOUT_BLOCK, p.lnqb - 1);
    const uint8_t* rows = layout + static_cast<size_t>(bh % p.H) * p.lnqb * p.lnkb;
    int n = 0;
    for (int kb = 0; kb < p.lnkb; ++kb) {
      bool on = false;
      for (int r = r0; r <= r1 && !on; ++r) on = rows[static_cast<size_t>(r) * p.lnkb + kb] != 0;
      n += on ? per : 0;
    }
    cost[t] = n;
  }
  return cost;
}

// Plans built from host data, cached by the shape and an FNV-1a-style hash of that data (the
// lengths, or the layout bytes), so that repeated calls with the same lengths or layout pay
// for the hash only.
std::map<std::pair<std::array<int, 12>, uint64_t>, std::unique_ptr<fa::PrefillSched>> g_data_plans;

// FNV-1a over 8-byte words (then the tail bytes): a layout of tens of KB is hashed on every
// call, so a word at a time.
uint64_t fnv1a(const void* data, size_t n) {
  const uint8_t* b = static_cast<const uint8_t*>(data);
  uint64_t h = 1469598103934665603ull;
  size_t i = 0;
  for (; i + 8 <= n; i += 8) {
    uint64_t w;
    std::memcpy(&w, b + i, 8);
    h = (h ^ w) * 1099511628211ull;
  }
  for (; i < n; ++i) h = (h ^ b[i]) * 1099511628211ull;
  return h;
}

const fa::PrefillSched* plan_for_data(const fa::PrefillParams& p, int BM, int BN, int grid,
                                      const int32_t* sk_host, const uint8_t* layout, int cap) {
  const uint64_t h = layout ? fnv1a(layout, static_cast<size_t>(p.H) * p.lnqb * p.lnkb)
                            : fnv1a(sk_host, static_cast<size_t>(p.BH / p.H) * sizeof(int32_t));
  const std::pair<std::array<int, 12>, uint64_t> key{
      {p.BH, p.Sq, p.Sk, BM, BN, p.mask_mode, p.window, p.n_global, p.group_heads, grid, p.nmb,
       layout ? 1 : 0},
      h};
  std::lock_guard<std::mutex> lock(g_plan_mu);
  auto it = g_data_plans.find(key);
  if (it != g_data_plans.end()) return it->second.get();
  if (g_data_plans.size() >= 64) g_data_plans.clear();  // launches copy their plan
  auto plan = std::make_unique<fa::PrefillSched>();
  plan_with_costs(p, grid,
                  layout ? costs_from_layout(p, BM, BN, layout)
                         : costs_from_lengths(p, BM, BN, sk_host, cap),
                  layout != nullptr, plan.get());
  const fa::PrefillSched* out = plan.get();
  g_data_plans.emplace(key, std::move(plan));
  return out;
}

size_t fwd_workspace_bytes(int B, int H, int Sq, int Sk, int d, int dtype) {
  if (dtype != FA_F32 || B < 1 || H < 1 || Sq < 0 || Sk < 0 || d < 1) return 0;
  // a bf16 high and low plane of every Q, K and V element
  return static_cast<size_t>(4) * d * B * H * (static_cast<size_t>(Sq) + 2 * static_cast<size_t>(Sk));
}

// allow_f32: FP32 inputs are taken by fa_fwd_ex (contiguous K/V, with a workspace) only.
fa_status check_fwd(const fa_fwd_params& p, bool allow_f32 = false) {
  // q and o may be null only when Sq == 0, k and v only when Sk == 0
  if ((p.Sq > 0 && (!p.q || !p.o)) || (p.Sk > 0 && (!p.k || !p.v)))
    return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (!aligned16(p.q) || !aligned16(p.k) || !aligned16(p.v) || !aligned16(p.o))
    return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if (p.lse && !aligned4(p.lse)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (p.B < 1 || p.H < 1 || p.Sq < 0 || p.Sk < 0)
    return fail(FA_ERR_INVALID_ARG, "need B >= 1, H >= 1, Sq >= 0, Sk >= 0 (got %d %d %d %d)", p.B,
                p.H, p.Sq, p.Sk);
  if (p.d != 64 && p.d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", p.d);
  if (p.dtype != FA_F16 && p.dtype != FA_BF16 && !(allow_f32 && p.dtype == FA_F32))
    return fail(FA_ERR_UNSUPPORTED, "dtype %d%s", p.dtype,
                p.dtype == FA_F32 ? " (FP32 inputs: fa_fwd_ex over contiguous K/V)" : "");
  if (!std::isfinite(p.scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  if (p.mask_mode < FA_MASK_NONE || p.mask_mode > FA_MASK_BLOCK_SPARSE)
    return fail(FA_ERR_INVALID_ARG, "mask_mode %d", p.mask_mode);
  if (p.mask_mode == FA_MASK_BLOCK_SPARSE && !p.block_layout && p.Sq > 0)
    return fail(FA_ERR_INVALID_ARG, "BLOCK_SPARSE needs params.block_layout");
  if (p.mask_mode == FA_MASK_CAUSAL_WINDOW && (p.window < 1 || p.n_global < 0))
    return fail(FA_ERR_INVALID_ARG, "CAUSAL_WINDOW needs window >= 1 and n_global >= 0");
  if (p.mask_mode == FA_MASK_BAND && p.window < 0)
    return fail(FA_ERR_INVALID_ARG, "BAND needs window >= 0");
  if (p.mask_mode == FA_MASK_PREFIX_LM && p.n_global < 0)
    return fail(FA_ERR_INVALID_ARG, "PREFIX_LM needs n_global >= 0");
  const long long BH = static_cast<long long>(p.B) * p.H;
  const long long S = p.Sq > p.Sk ? p.Sq : p.Sk;
  if (BH > (1LL << 30) || S > (1LL << 30) || BH * ((S + 63) / 64) > (1LL << 31) - 1)
    return fail(FA_ERR_INVALID_ARG, "problem too large for 32-bit tile indices");
  if (p.block_n != 0 && p.block_n != 64 && p.block_n != 128)
    return fail(FA_ERR_UNSUPPORTED, "block_n %d (supported: 64, 128)", p.block_n);
  if (p.block_m != 0 && p.block_m != 64 && p.block_m != 128 && p.block_m != 256)
    return fail(FA_ERR_UNSUPPORTED, "block_m %d (supported: 64, 128, 256)", p.block_m);
  if (p.num_ctas < 0 || p.group_heads < 0) return fail(FA_ERR_INVALID_ARG, "negative plan parameter");
  if (p.dtype == FA_F32) {
    if (BH > (1LL << 29))  // the tensor maps see 2 * B * H planes
      return fail(FA_ERR_INVALID_ARG, "FA_F32: B * H above 2^29");
    if (p.block_n != 0 && p.block_n != fa::kSplitBlockN)
      return fail(FA_ERR_UNSUPPORTED, "block_n %d with FA_F32 (supported: 64)", p.block_n);
    if (p.block_m != 0 && p.block_m != 256)
      return fail(FA_ERR_UNSUPPORTED, "block_m %d with FA_F32 (supported: 256)", p.block_m);
    const size_t need = fwd_workspace_bytes(p.B, p.H, p.Sq, p.Sk, p.d, p.dtype);
    if (p.Sq > 0 && (!p.workspace || !aligned16(p.workspace)))
      return fail(FA_ERR_INVALID_ARG, "FA_F32 needs a 16-byte aligned workspace");
    if (p.Sq > 0 && p.workspace_bytes < need)
      return fail(FA_ERR_INVALID_ARG, "workspace has %zu bytes, FA_F32 needs %zu",
                  p.workspace_bytes, need);
  }
  return FA_OK;
}

}  // namespace

extern "C" {

int fa_version(void) { return 100; }

const char* fa_last_error_string(void) { return t_last_error.c_str(); }

int fa_fwd_block_m(void) { return fa::prefill_tile_rows(); }

size_t fa_fwd_workspace_size(int B, int H, int Sq, int Sk, int d, int dtype) {
  return fwd_workspace_bytes(B, H, Sq, Sk, d, dtype);
}

int fa_fwd_default_block_m(int mask_mode) {
  if (mask_mode < FA_MASK_NONE || mask_mode > FA_MASK_BLOCK_SPARSE) return 0;
  // the band's narrow key ranges, and block-sparse rows whose union over two query
  // blocks is much larger than either, favour one tile per item
  return mask_mode == FA_MASK_BAND || mask_mode == FA_MASK_BLOCK_SPARSE ? 128 : 256;
}

}  // extern "C"

namespace {

// K/V read through a page table (chunked prefill into a paged cache).
struct PagedKV {
  const void* k_pages;
  const void* v_pages;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  int page_size, max_pages, num_pages;
};

// Plan and launch one prefill. `a` has passed check_fwd; with `pg` set, a.Sk is the
// table's capacity and K/V come from the pools.
fa_status run_fwd(const fa_fwd_params& a, const PagedKV* pg, fa_stream_t stream,
                  const int32_t* sk_host = nullptr) {
  fa_status st;
  if (a.Sq == 0) return FA_OK;  // nothing to compute
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;

  const bool f32 = a.dtype == FA_F32;  // split into bf16 planes; 256-row items, 64-key blocks
  const int BM = f32 ? 256 : (a.block_m ? a.block_m : fa_fwd_default_block_m(a.mask_mode));
  const int BN = f32 ? fa::kSplitBlockN : (a.block_n ? a.block_n : 128);
  const int BH = a.B * a.H;
  fa::PrefillLaunch L;
  std::memset(&L, 0, sizeof L);
  fa::PrefillParams& p = L.p;
  p.o = a.o;
  p.lse = a.lse;
  p.BH = BH;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.nmb = (a.Sq + BM - 1) / BM;
  p.nnb = (a.Sk + BN - 1) / BN;
  p.mask_mode = a.mask_mode;
  const bool uses_window = a.mask_mode == FA_MASK_CAUSAL_WINDOW || a.mask_mode == FA_MASK_BAND;
  const bool uses_global = a.mask_mode == FA_MASK_CAUSAL_WINDOW || a.mask_mode == FA_MASK_PREFIX_LM;
  p.window = uses_window ? a.window : 0;
  p.n_global = uses_global ? a.n_global : 0;
  p.sl2 = a.scale * 1.4426950408889634f;
  // Heads scheduled together so that their K/V stays resident in L2 (~48 MiB budget).
  long long kv_keys = a.Sk;
  if (a.mask_mode == FA_MASK_CAUSAL_WINDOW) {
    const long long band = static_cast<long long>(a.window) + a.n_global + BM + BN;
    if (band < kv_keys) kv_keys = band;
  } else if (a.mask_mode == FA_MASK_BAND) {
    const long long band = 2LL * a.window + BM + BN;
    if (band < kv_keys) kv_keys = band;
  }
  const long long kv_bytes = kv_keys * a.d * (f32 ? 8 : 4) + 1;
  long long hg = a.group_heads ? a.group_heads : (48LL << 20) / kv_bytes;
  if (hg < 1) hg = 1;
  if (hg > BH) hg = BH;
  p.group_heads = static_cast<int>(hg);
  p.total_items = BH * p.nmb;
  p.status = dev.status;
  p.timeout_ns = static_cast<uint64_t>(a.timeout_us ? a.timeout_us : 1000000u) * 1000u;
  p.trace = a.trace;
  p.rescales = a.rescale_count;
  p.H = a.H;
  if (a.mask_mode == FA_MASK_BLOCK_SPARSE) {  // planned as dense: the layout is on the device
    p.layout = a.block_layout;
    p.lnqb = (a.Sq + FA_LAYOUT_BLOCK - 1) / FA_LAYOUT_BLOCK;
    p.lnkb = (a.Sk + FA_LAYOUT_BLOCK - 1) / FA_LAYOUT_BLOCK;
  }
  L.grid = a.num_ctas ? a.num_ctas : dev.sms;
  if (L.grid > p.total_items) L.grid = p.total_items;
  const bool layout_hint = a.mask_mode == FA_MASK_BLOCK_SPARSE && a.block_layout_host;
  if ((pg && sk_host) || layout_hint) {
    L.sched = layout_hint ? plan_for_data(p, BM, BN, L.grid, nullptr, a.block_layout_host, 0)
                          : plan_for_data(p, BM, BN, L.grid, sk_host, nullptr, a.Sk);
  } else {
    L.sched = plan_for(p, BM, BN, L.grid);
  }

  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (f32) {
    // workspace planes Q_hi Q_lo K_hi K_lo V_hi V_lo, each [B*H, S, d] bf16: the maps see
    // a tensor's two planes as one [2*B*H, S, d] tensor
    uint16_t* qh = static_cast<uint16_t*>(a.workspace);
    const size_t nq = static_cast<size_t>(BH) * a.Sq * a.d, nk = static_cast<size_t>(BH) * a.Sk * a.d;
    uint16_t* kh = qh + 2 * nq;
    uint16_t* vh = kh + 2 * nk;
    const fa::SplitArgs sa{{static_cast<const float*>(a.q), static_cast<const float*>(a.k),
                            static_cast<const float*>(a.v)},
                           {qh, kh, vh},
                           {qh + nq, kh + nk, vh + nk},
                           {nq / 8, nk / 8, nk / 8}};
    cudaError_t e = fa::launch_split_bf16(sa, dev.sms, cs);
    if (e != cudaSuccess) return cuda_fail(e, "split launch");
    if ((st = make_map(&L.tmQ, qh, true, a.d, a.Sq, 2 * BH, fa::prefill_tile_rows())) != FA_OK)
      return st;
    if ((st = make_map(&L.tmK, a.Sk ? kh : qh, true, a.d, a.Sk, 2 * BH, BN)) != FA_OK) return st;
    if ((st = make_map(&L.tmV, a.Sk ? vh : qh, true, a.d, a.Sk, 2 * BH, BN)) != FA_OK) return st;
    e = fa::launch_prefill_split(L, a.d, cs);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return FA_OK;
  }
  const bool bf16 = a.dtype == FA_BF16;
  // one Q box is one tensor-core tile: 64 rows for 64-row items, else 128
  const int q_rows = BM == 64 ? 64 : fa::prefill_tile_rows();
  if ((st = make_map(&L.tmQ, a.q, bf16, a.d, a.Sq, BH, q_rows)) != FA_OK) return st;
  if (pg) {
    // pools [num_pages, H, page, d] seen as (d, page, num_pages*H); a tile is BN rows of
    // one (page, head)
    p.block_table = pg->block_table;
    p.seq_k = pg->ctx_lens;
    p.H = a.H;
    p.page_size = pg->page_size;
    p.max_pages = pg->max_pages;
    p.num_pages = pg->num_pages;
    const int zdim = pg->num_pages * a.H;
    if ((st = make_map(&L.tmK, pg->k_pages, bf16, a.d, pg->page_size, zdim, BN)) != FA_OK)
      return st;
    if ((st = make_map(&L.tmV, pg->v_pages, bf16, a.d, pg->page_size, zdim, BN)) != FA_OK)
      return st;
  } else {
    // with Sk == 0 no key tile is ever loaded; the maps only need a valid address
    if ((st = make_map(&L.tmK, a.Sk ? a.k : a.q, bf16, a.d, a.Sk, BH, BN)) != FA_OK) return st;
    if ((st = make_map(&L.tmV, a.Sk ? a.v : a.q, bf16, a.d, a.Sk, BH, BN)) != FA_OK) return st;
  }
  cudaError_t e = fa::launch_prefill(L, a.d, BN, BM, bf16, cs);
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  return FA_OK;
}

}  // namespace

extern "C" {

fa_status fa_fwd_ex(const fa_fwd_params* params, fa_stream_t stream) {
  if (!params) return fail(FA_ERR_INVALID_ARG, "params is null");
  fa_status st = check_fwd(*params, true);
  if (st != FA_OK) return st;
  return run_fwd(*params, nullptr, stream);
}

static fa_status fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                           const int32_t* block_table, const int32_t* ctx_lens,
                           const int32_t* ctx_lens_host, void* o, float* lse, int B, int H,
                           int Sq, int d, int page_size, int max_pages_per_seq, int num_pages,
                           float scale, int mask_mode, int window, int n_global, int dtype,
                           fa_stream_t stream) {
  if (!k_pages || !v_pages || !block_table || !ctx_lens)
    return fail(FA_ERR_INVALID_ARG, "k_pages, v_pages, block_table and ctx_lens must be non-null");
  if (!aligned16(k_pages) || !aligned16(v_pages))
    return fail(FA_ERR_INVALID_ARG, "pools must be 16-byte aligned");
  if (!aligned4(block_table) || !aligned4(ctx_lens))
    return fail(FA_ERR_INVALID_ARG, "block_table and ctx_lens must be 4-byte aligned");
  if (max_pages_per_seq < 1 || num_pages < 1)
    return fail(FA_ERR_INVALID_ARG, "need max_pages_per_seq, num_pages >= 1");
  if (page_size < 64 || page_size > 4096 || page_size % 64 != 0)
    return fail(FA_ERR_UNSUPPORTED, "page_size %d (a multiple of 64 in [64, 4096])", page_size);
  const long long cap = static_cast<long long>(page_size) * max_pages_per_seq;
  const long long zdim = static_cast<long long>(num_pages) * (H > 0 ? H : 1);
  if (cap > (1LL << 30) || zdim > (1LL << 31) - 1)
    return fail(FA_ERR_INVALID_ARG, "problem too large");
  fa_fwd_params a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Sq = Sq;
  a.Sk = static_cast<int>(cap);
  a.d = d;
  a.scale = scale;
  a.mask_mode = mask_mode;
  a.window = window;
  a.n_global = n_global;
  a.dtype = dtype;
  a.block_m = fa_fwd_default_block_m(mask_mode);
  a.block_n = page_size % 128 == 0 ? 128 : 64;  // a K/V tile never crosses a page
  fa_status st = check_fwd(a);
  if (st != FA_OK) return st;
  const PagedKV pg{k_pages, v_pages, block_table, ctx_lens, page_size, max_pages_per_seq,
                   num_pages};
  return run_fwd(a, &pg, stream, ctx_lens_host);
}

fa_status fa_fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                       const int32_t* block_table, const int32_t* ctx_lens, void* o, float* lse,
                       int B, int H, int Sq, int d, int page_size, int max_pages_per_seq,
                       int num_pages, float scale, int mask_mode, int window, int n_global,
                       int dtype, fa_stream_t stream) {
  return fwd_paged(q, k_pages, v_pages, block_table, ctx_lens, nullptr, o, lse, B, H, Sq, d,
                   page_size, max_pages_per_seq, num_pages, scale, mask_mode, window, n_global,
                   dtype, stream);
}

fa_status fa_fwd_paged_host_lens(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* ctx_lens,
                                 const int32_t* ctx_lens_host, void* o, float* lse, int B, int H,
                                 int Sq, int d, int page_size, int max_pages_per_seq,
                                 int num_pages, float scale, int mask_mode, int window,
                                 int n_global, int dtype, fa_stream_t stream) {
  return fwd_paged(q, k_pages, v_pages, block_table, ctx_lens, ctx_lens_host, o, lse, B, H, Sq,
                   d, page_size, max_pages_per_seq, num_pages, scale, mask_mode, window,
                   n_global, dtype, stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Sq, int Sk, int d, float scale, int mask_mode, int window, int n_global,
                 int dtype, fa_stream_t stream) {
  fa_fwd_params p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k = k;
  p.v = v;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.d = d;
  p.scale = scale;
  p.mask_mode = mask_mode;
  p.window = window;
  p.n_global = n_global;
  p.dtype = dtype;
  if (dtype == FA_F32 && Sq > 0)
    return fail(FA_ERR_INVALID_ARG,
                "FA_F32 inputs need a workspace: call fa_fwd_ex with params.workspace of "
                "fa_fwd_workspace_size() bytes");
  return fa_fwd_ex(&p, stream);
}

int fa_decode_default_pages_per_split(int B, int H, int max_pages_per_seq) {
  // Enough splits that the ragged mix of context lengths still fills the GPU
  // several times over, without making the merge step large.
  const long long bh = static_cast<long long>(B > 0 ? B : 1) * (H > 0 ? H : 1);
  int pps = 1;
  while (pps < max_pages_per_seq && bh * ((max_pages_per_seq + pps - 1) / pps) > 16384) pps *= 2;
  return pps;
}

size_t fa_decode_workspace_size(int B, int H, int d, int max_pages_per_seq, int page_size) {
  (void)page_size;
  if (B < 1 || H < 1 || d < 1 || max_pages_per_seq < 1) return 0;
  return static_cast<size_t>(B) * H * max_pages_per_seq * (d + 2) * sizeof(float);
}

fa_status fa_decode_paged_ex(const fa_decode_params* params, fa_stream_t stream) {
  if (!params) return fail(FA_ERR_INVALID_ARG, "params is null");
  const fa_decode_params& a = *params;
  if (!a.q || !a.k_pages || !a.v_pages || !a.block_table || !a.ctx_lens || !a.o || !a.workspace)
    return fail(FA_ERR_INVALID_ARG, "q, k_pages, v_pages, block_table, ctx_lens, o, workspace must be non-null");
  if (!aligned16(a.q) || !aligned16(a.k_pages) || !aligned16(a.v_pages) || !aligned16(a.o) ||
      !aligned16(a.workspace))
    return fail(FA_ERR_INVALID_ARG, "q, pools, o and workspace must be 16-byte aligned");
  if (!aligned4(a.block_table) || !aligned4(a.ctx_lens) || (a.lse && !aligned4(a.lse)))
    return fail(FA_ERR_INVALID_ARG, "block_table, ctx_lens and lse must be 4-byte aligned");
  if (a.B < 1 || a.H < 1 || a.max_pages_per_seq < 1 || a.num_pages < 1)
    return fail(FA_ERR_INVALID_ARG, "need B, H, max_pages_per_seq, num_pages >= 1");
  if (a.d != 64 && a.d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", a.d);
  if (a.dtype != FA_F16 && a.dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "dtype %d", a.dtype);
  if (a.page_size < 16 || a.page_size > 4096 || a.page_size % 16 != 0)
    return fail(FA_ERR_UNSUPPORTED, "page_size %d (a multiple of 16 in [16, 4096])", a.page_size);
  if (!std::isfinite(a.scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  const long long max_ctx = static_cast<long long>(a.page_size) * a.max_pages_per_seq;
  const long long pool = static_cast<long long>(a.num_pages) * a.H * a.page_size * a.d;
  if (max_ctx > (1LL << 30) || static_cast<long long>(a.B) * a.H > (1LL << 30) || pool > (1LL << 46))
    return fail(FA_ERR_INVALID_ARG, "problem too large");
  const size_t need = fa_decode_workspace_size(a.B, a.H, a.d, a.max_pages_per_seq, a.page_size);
  if (a.workspace_bytes < need)
    return fail(FA_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", a.workspace_bytes, need);
  int pps = a.pages_per_split ? a.pages_per_split
                              : fa_decode_default_pages_per_split(a.B, a.H, a.max_pages_per_seq);
  if (pps < 1 || pps > a.max_pages_per_seq) return fail(FA_ERR_INVALID_ARG, "pages_per_split %d", pps);
  const long long nsplit = (a.max_pages_per_seq + pps - 1) / pps;
  if (nsplit * a.B * a.H > (1LL << 31) - 1) return fail(FA_ERR_INVALID_ARG, "too many splits");
  DeviceInfo dev;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;

  fa::DecodeParams p;
  std::memset(&p, 0, sizeof p);
  p.q = a.q;
  p.k_pages = a.k_pages;
  p.v_pages = a.v_pages;
  p.block_table = a.block_table;
  p.ctx_lens = a.ctx_lens;
  p.o = a.o;
  p.lse = a.lse;
  p.part = static_cast<float*>(a.workspace);
  p.B = a.B;
  p.H = a.H;
  p.page_size = a.page_size;
  p.max_pages = a.max_pages_per_seq;
  p.num_pages = a.num_pages;
  p.pages_per_split = pps;
  p.nsplit_max = static_cast<int>(nsplit);
  p.sl2 = a.scale * 1.4426950408889634f;
  p.status = dev.status;
  p.trace_pages = a.trace_pages;
  p.trace_splits = a.trace_splits;
  cudaError_t e = fa::launch_decode(p, a.d, a.dtype == FA_BF16, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return FA_OK;
}

fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* block_table, const int32_t* ctx_lens, void* o, float* lse,
                          int B, int H, int d, int page_size, int max_pages_per_seq, int num_pages,
                          float scale, int dtype, void* workspace, size_t workspace_bytes,
                          fa_stream_t stream) {
  fa_decode_params p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.d = d;
  p.page_size = page_size;
  p.max_pages_per_seq = max_pages_per_seq;
  p.num_pages = num_pages;
  p.scale = scale;
  p.dtype = dtype;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  return fa_decode_paged_ex(&p, stream);
}

fa_status fa_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                  const int32_t* block_table, const int32_t* ctx_lens, void* o,
                                  float* lse, int B, int H, int d, int page_size,
                                  int max_pages_per_seq, int num_pages, float scale, int dtype,
                                  fa_stream_t stream) {
  if (!q || !k_pages || !v_pages || !block_table || !ctx_lens || !o)
    return fail(FA_ERR_INVALID_ARG, "q, k_pages, v_pages, block_table, ctx_lens and o must be non-null");
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o))
    return fail(FA_ERR_INVALID_ARG, "q, pools and o must be 16-byte aligned");
  if (!aligned4(block_table) || !aligned4(ctx_lens) || (lse && !aligned4(lse)))
    return fail(FA_ERR_INVALID_ARG, "block_table, ctx_lens and lse must be 4-byte aligned");
  if (B < 1 || H < 1 || max_pages_per_seq < 1 || num_pages < 1)
    return fail(FA_ERR_INVALID_ARG, "need B, H, max_pages_per_seq, num_pages >= 1");
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", d);
  if (dtype != FA_F16 && dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (page_size < 16 || page_size > 4096 || page_size % 16 != 0)
    return fail(FA_ERR_UNSUPPORTED, "page_size %d (a multiple of 16 in [16, 4096])", page_size);
  if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  const long long max_ctx = static_cast<long long>(page_size) * max_pages_per_seq;
  const long long pool = static_cast<long long>(num_pages) * H * page_size * d;
  if (max_ctx > (1LL << 30) || static_cast<long long>(B) * H > (1LL << 30) || pool > (1LL << 46))
    return fail(FA_ERR_INVALID_ARG, "problem too large");
  // The split size is fa_decode_paged's default. That default keeps B*H*splits at or
  // below 16384 whenever one split per sequence allows it (16384*(d+2)*4 bytes, 8.5 MB
  // at d = 128, fit the scratch), and is one split per sequence otherwise, so the
  // partials fit exactly when B*H*(d+2)*4 bytes do.
  const size_t cap = fa::noalloc_scratch_bytes();
  const int pps = fa_decode_default_pages_per_split(B, H, max_pages_per_seq);
  const size_t partial_bytes = static_cast<size_t>(B) * H *
                               ((max_pages_per_seq + pps - 1) / pps) * (d + 2) * sizeof(float);
  if (partial_bytes > cap)
    return fail(FA_ERR_INVALID_ARG,
                "%zu bytes of split partials exceed the %zu-byte scratch of "
                "fa_decode_paged_noalloc (B*H*(d+2)*4 must fit); use fa_decode_paged with a "
                "workspace",
                partial_bytes, cap);
  DeviceInfo dev;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  fa::DecodeParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.block_table = block_table;
  p.ctx_lens = ctx_lens;
  p.o = o;
  p.lse = lse;
  p.B = B;
  p.H = H;
  p.page_size = page_size;
  p.max_pages = max_pages_per_seq;
  p.num_pages = num_pages;
  p.pages_per_split = pps;
  p.nsplit_max = (max_pages_per_seq + pps - 1) / pps;
  p.sl2 = scale * 1.4426950408889634f;
  p.status = dev.status;
  cudaError_t e =
      fa::launch_decode_noalloc(p, d, dtype == FA_BF16, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode (no-alloc) launch");
  return FA_OK;
}

// Workspace of fa_bwd at head dimension d: the FP32 dQ accumulator [B*H][ceil(Sq/4)][d][4]
// first, then D [B,H,Sq]; fa_bwd_workspace_size covers the largest supported d.
static size_t bwd_workspace_bytes(int B, int H, int Sq, int d) {
  const size_t s = Sq > 0 ? static_cast<size_t>(Sq) : 1;
  return static_cast<size_t>(B) * H * ((s + 3) / 4 * 4 * static_cast<size_t>(d) + s) *
         sizeof(float);
}

size_t fa_bwd_workspace_size(int B, int H, int Sq) {
  if (B < 1 || H < 1 || Sq < 0) return 0;
  return bwd_workspace_bytes(B, H, Sq, 128);
}

static fa_status bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dout, const float* lse, void* dq, void* dk, void* dv,
                     void* workspace, size_t workspace_bytes, int B, int H, int Sq, int Sk, int d,
                     float scale, int mask_mode, int window, int n_global,
                     const uint8_t* layout, int dtype, fa_stream_t stream) {
  fa_fwd_params a;  // the forward's checks cover q, k, v, sizes, mask and dtype
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = dq;  // any non-null 16-byte-aligned output passes the output check
  a.B = B;
  a.H = H;
  a.Sq = Sq;
  a.Sk = Sk;
  a.d = d;
  a.scale = scale;
  a.mask_mode = mask_mode;
  a.window = window;
  a.n_global = n_global;
  a.dtype = dtype;
  a.block_layout = layout;
  fa_status st = check_fwd(a);
  if (st != FA_OK) return st;
  if (Sq == 0 && Sk == 0) return FA_OK;
  if ((Sq > 0 && (!o || !dout || !lse || !dq)) || (Sk > 0 && (!dk || !dv)))
    return fail(FA_ERR_INVALID_ARG, "o, dout, lse, dq, dk and dv must be non-null");
  if (!aligned16(o) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(FA_ERR_INVALID_ARG, "o, dout, dq, dk and dv must be 16-byte aligned");
  if (lse && !aligned4(lse)) return fail(FA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const size_t need = bwd_workspace_bytes(B, H, Sq, d);
  if (Sq > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return fail(FA_ERR_INVALID_ARG, "workspace: %zu bytes, 16-byte aligned, needed", need);
  DeviceInfo dev;
  if ((st = device_info(&dev)) != FA_OK) return st;
  const int BH = B * H;
  const bool bf16 = dtype == FA_BF16;
  fa::BwdLaunch L;
  std::memset(&L, 0, sizeof L);
  fa::PrefillParams& p = L.p;
  p.BH = BH;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.mask_mode = mask_mode;
  p.window = (mask_mode == FA_MASK_CAUSAL_WINDOW || mask_mode == FA_MASK_BAND) ? window : 0;
  p.n_global = (mask_mode == FA_MASK_CAUSAL_WINDOW || mask_mode == FA_MASK_PREFIX_LM) ? n_global : 0;
  p.sl2 = scale * 1.4426950408889634f;
  p.status = dev.status;
  p.timeout_ns = 1000000000ull;
  if (mask_mode == FA_MASK_BLOCK_SPARSE) {  // one layout block is one backward tile (128 x 128)
    p.layout = layout;
    p.lnqb = (Sq + FA_LAYOUT_BLOCK - 1) / FA_LAYOUT_BLOCK;
    p.lnkb = (Sk + FA_LAYOUT_BLOCK - 1) / FA_LAYOUT_BLOCK;
  }
  L.b.lse = lse;
  L.b.dqacc = static_cast<float*>(workspace);
  L.b.dsum = static_cast<float*>(workspace) + static_cast<size_t>(BH) * ((Sq + 3) / 4) * 4 * d;
  L.b.dq = dq;
  L.b.dk = dk;
  L.b.dv = dv;
  L.b.scale = scale;
  {  // the dK/dV kernel's launch order: heads in groups whose CTAs make about two waves
    const int nkb = (Sk + 127) / 128;
    L.b.head_group = nkb > 0 ? std::min(BH, std::max(1, (2 * dev.sms + nkb - 1) / nkb)) : 1;
  }
  L.o = o;
  L.dout = dout;
  const void* qmap = Sq ? q : k;  // a map needs a valid address even when nothing is loaded
  const void* kmap = Sk ? k : q;
  const int box = fa::kBwdBoxRows;
  if ((st = make_map(&L.tmQ, qmap, bf16, d, Sq, BH, box)) != FA_OK) return st;
  if ((st = make_map(&L.tmdO, Sq ? dout : k, bf16, d, Sq, BH, box)) != FA_OK) return st;
  if ((st = make_map(&L.tmK, kmap, bf16, d, Sk, BH, box)) != FA_OK) return st;
  if ((st = make_map(&L.tmV, Sk ? v : q, bf16, d, Sk, BH, box)) != FA_OK) return st;
  cudaError_t e = fa::launch_backward(L, d, bf16, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  return FA_OK;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 size_t workspace_bytes, int B, int H, int Sq, int Sk, int d, float scale,
                 int mask_mode, int window, int n_global, int dtype, fa_stream_t stream) {
  if (mask_mode == FA_MASK_BLOCK_SPARSE)
    return fail(FA_ERR_UNSUPPORTED, "fa_bwd: a block layout goes through fa_bwd_block_sparse");
  return bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, Sq, Sk, d,
             scale, mask_mode, window, n_global, nullptr, dtype, stream);
}

fa_status fa_bwd_block_sparse(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              void* workspace, size_t workspace_bytes, int B, int H, int Sq,
                              int Sk, int d, float scale, const uint8_t* block_layout, int dtype,
                              fa_stream_t stream) {
  return bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H, Sq, Sk, d,
             scale, FA_MASK_BLOCK_SPARSE, 0, 0, block_layout, dtype, stream);
}

fa_status fa_merge_partials(const void* o_a, const float* lse_a, const void* o_b,
                            const float* lse_b, void* o, float* lse, int64_t rows, int d,
                            int dtype, fa_stream_t stream) {
  if (rows < 0) return fail(FA_ERR_INVALID_ARG, "rows must be >= 0");
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", d);
  if (dtype != FA_F16 && dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (rows == 0) return FA_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o)
    return fail(FA_ERR_INVALID_ARG, "o_a, lse_a, o_b, lse_b and o must be non-null");
  if (!aligned16(o_a) || !aligned16(o_b) || !aligned16(o))
    return fail(FA_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
  if (!aligned4(lse_a) || !aligned4(lse_b) || (lse && !aligned4(lse)))
    return fail(FA_ERR_INVALID_ARG, "LSE arrays must be 4-byte aligned");
  if (rows > (1LL << 40)) return fail(FA_ERR_INVALID_ARG, "too many rows");
  DeviceInfo dev;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_merge(o_a, lse_a, o_b, lse_b, o, lse, rows, d, dtype == FA_BF16,
                                   dev.sms, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return FA_OK;
}

fa_status fa_kv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                       const int32_t* block_table, const int32_t* ctx_lens,
                       const int32_t* new_lens, int B, int H, int T, int d, int page_size,
                       int max_pages_per_seq, int num_pages, int dtype, fa_stream_t stream) {
  if (B < 1 || H < 1 || T < 0 || max_pages_per_seq < 1 || num_pages < 1)
    return fail(FA_ERR_INVALID_ARG, "need B, H, max_pages_per_seq, num_pages >= 1 and T >= 0");
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", d);
  if (dtype != FA_F16 && dtype != FA_BF16) return fail(FA_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (page_size < 16 || page_size > 4096 || page_size % 16 != 0)
    return fail(FA_ERR_UNSUPPORTED, "page_size %d (a multiple of 16 in [16, 4096])", page_size);
  if (T == 0) return FA_OK;
  if (!k_new || !v_new || !k_pages || !v_pages || !block_table || !ctx_lens)
    return fail(FA_ERR_INVALID_ARG, "k_new, v_new, pools, block_table and ctx_lens must be non-null");
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages))
    return fail(FA_ERR_INVALID_ARG, "k_new, v_new and pools must be 16-byte aligned");
  if (!aligned4(block_table) || !aligned4(ctx_lens) || (new_lens && !aligned4(new_lens)))
    return fail(FA_ERR_INVALID_ARG, "block_table, ctx_lens and new_lens must be 4-byte aligned");
  const long long cap = static_cast<long long>(page_size) * max_pages_per_seq;
  if (cap > (1LL << 30) || static_cast<long long>(B) * H > (1LL << 31) - 1 ||
      static_cast<long long>(B) * H * T * d > (1LL << 46))
    return fail(FA_ERR_INVALID_ARG, "problem too large");
  DeviceInfo dev;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  fa::KvAppendParams p{block_table, ctx_lens, new_lens, B, H, T, d, page_size, max_pages_per_seq,
                       num_pages, dev.status};
  cudaError_t e = fa::launch_kv_append(k_new, v_new, k_pages, v_pages, p,
                                       reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return FA_OK;
}

fa_status fa_get_device_status(fa_stream_t stream) {
  DeviceInfo dev;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, dev.status, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device status word");
  const uint32_t zero = 0;
  e = cudaMemcpy(dev.status, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device status word");
  if (word & fa::FA_DEV_TIMEOUT) return fail(FA_ERR_TIMEOUT, "a kernel gave up on a pipeline wait");
  if (word & fa::FA_DEV_BAD_PAGE) return fail(FA_ERR_BAD_PAGE, "a block-table entry or context length was out of range");
  if (word & fa::FA_DEV_SMEM_BASE)
    return fail(FA_ERR_UNSUPPORTED, "a kernel's dynamic shared memory did not start close enough "
                "to a 1024-byte boundary for its layout; its outputs were not written");
  return FA_OK;
}

fa_status fa_selftest_timeout(uint32_t timeout_us, fa_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000u)
    return fail(FA_ERR_INVALID_ARG, "timeout_us must be in [1, 1000000]");
  DeviceInfo dev;
  fa_status st = device_info(&dev);
  if (st != FA_OK) return st;
  cudaError_t e = fa::launch_selftest_timeout(dev.status, static_cast<uint64_t>(timeout_us) * 1000u,
                                              reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return FA_OK;
}

}  // extern "C"
