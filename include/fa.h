/*
 * fa.h - FlashAttention forward for one NVIDIA GB300 (sm_103a): C ABI.
 *
 * What is computed. For every (batch b, head h) and query row i:
 *     O[b,h,i,:] = sum_j P_ij V[b,h,j,:],
 *     P_ij = exp(scale * Q_i.K_j) / sum_{t in Vis(i)} exp(scale * Q_i.K_t),  j in Vis(i),
 *     LSE[b,h,i] = ln sum_{t in Vis(i)} exp(scale * Q_i.K_t)      (natural log),
 * i.e. O = softmax(scale * Q K^T + mask) V, the definition in the ops-transformer
 * overview (gitcode.csdn.net, section 二.1 "FlashAttention算子", the traditional-
 * attention listing), computed the way its tiled loop describes: the score tile is
 * produced on chip and never written to memory, the running max and sum are
 * updated block by block (softmax denominator in FP32, zwxr.cn article section 5.1)
 * and the output is normalised once at the end.
 *
 * Masks (Vis(i)); queries are aligned to the LAST Sq key positions, delta = Sk - Sq:
 *   FA_MASK_NONE           every key.
 *   FA_MASK_CAUSAL         j <= i + delta                (ops-transformer overview,
 *                                                        section 四, causal=True).
 *   FA_MASK_CAUSAL_WINDOW  j <= i + delta and (i + delta - j < window or j < n_global):
 *                          a causal sliding window of `window` keys (the query's own
 *                          position included) plus the first `n_global` keys as
 *                          global tokens ("ascend-transformer-boost 实战" (ai6s.net),
 *                          scenario 3, window_size=2048, global_tokens=64).
 *   FA_MASK_BAND           |i + delta - j| <= window: a two-sided band, each query
 *                          seeing the keys within `window` positions of its own on
 *                          either side (the diagonal band of the zwxr.cn article on
 *                          ops-transformer, section 3.2); window >= 0.
 *   FA_MASK_PREFIX_LM      j <= i + delta or j < n_global: the first n_global keys (the
 *                          prefix) are seen by every query, the rest causally (the
 *                          prefix-LM variant named in "ascend-transformer-boost 实战",
 *                          scenario 3); n_global >= 0.
 *   FA_MASK_BLOCK_SPARSE   layout[h][i / 128][j / 128] != 0: a caller's block layout,
 *                          uint8 [H][ceil(Sq/128)][ceil(Sk/128)], one per head and the same
 *                          for every batch entry (the block-sparse variant that
 *                          "ascend-transformer-boost 实战" names beside prefix-LM, read as
 *                          the usual block layout). fa_fwd_ex only (params.block_layout).
 * A query that sees no key gets O = 0 and LSE = -inf.
 *
 * Conventions for every call:
 *   - Pointers are DEVICE pointers unless stated otherwise, 16-byte aligned, and
 *     owned by the caller. The library allocates no memory in any call.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and never synchronises the host.
 *   - Argument errors are detected on the host before anything is launched and
 *     return FA_ERR_INVALID_ARG or FA_ERR_UNSUPPORTED; nothing runs in that case.
 *   - Faults found on the device (a page-table entry out of range, a pipeline wait
 *     that ran past its time limit) are recorded in a device status word and
 *     reported by fa_get_device_status().
 *   - fa_last_error_string() describes the last non-FA_OK status of this thread.
 *   - The library looks up a few device addresses (its status word, the scratch of
 *     fa_decode_paged_noalloc) once per device and keeps them; a process that calls
 *     cudaDeviceReset must not call the library afterwards.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* same type as cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* a null pointer, a negative size, misalignment, ... */
  FA_ERR_UNSUPPORTED = 2, /* valid but not built: d not in {64,128}, an unknown dtype */
  FA_ERR_CUDA = 3,        /* a CUDA runtime call failed (see fa_last_error_string) */
  FA_ERR_TIMEOUT = 4,     /* a kernel gave up on a pipeline wait (device status) */
  FA_ERR_BAD_PAGE = 5     /* a block-table entry or context length was out of range */
} fa_status;

/* FA_F32: FP32 inputs and output, fa_fwd_ex over contiguous K/V only (see fa_fwd_params). */
enum { FA_F16 = 0, FA_BF16 = 1, FA_F32 = 2 };
enum {
  FA_MASK_NONE = 0,
  FA_MASK_CAUSAL = 1,
  FA_MASK_CAUSAL_WINDOW = 2,
  FA_MASK_BAND = 3,
  FA_MASK_PREFIX_LM = 4,
  FA_MASK_BLOCK_SPARSE = 5
};

/* Block size of a block-sparse layout (query rows x keys). */
#define FA_LAYOUT_BLOCK 128

/*
 * fa_fwd - attention forward (prefill) over contiguous BHSD tensors.
 *   q      [B, H, Sq, d]  dtype (fp16 or bf16), row-major (d fastest)
 *   k, v   [B, H, Sk, d]  dtype
 *   o      [B, H, Sq, d]  dtype, written (RN from the FP32 accumulator)
 *   lse    [B, H, Sq]     float32, natural log; may be NULL
 *   d      64 or 128;  B, H >= 1;  Sq, Sk >= 0. q and o may be NULL when Sq == 0 (the
 *          call then does nothing); k and v may be NULL when Sk == 0 (every row then
 *          sees no key).
 *   scale  the softmax scale (typically 1/sqrt(d))
 *   mask_mode / window / n_global as above: window >= 1 and n_global >= 0 for
 *          FA_MASK_CAUSAL_WINDOW, window >= 0 for FA_MASK_BAND, n_global >= 0 for
 *          FA_MASK_PREFIX_LM; a parameter the mode does not use is ignored.
 *   dtype  FA_F16 or FA_BF16 (added before `stream`: a signature without it could
 *          not tell fp16 inputs from bf16 inputs). FA_F32 needs a workspace and is taken
 *          by fa_fwd_ex only; fa_fwd returns FA_ERR_INVALID_ARG for it (Sq > 0).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Sq, int Sk, int d, float scale, int mask_mode, int window, int n_global,
                 int dtype, fa_stream_t stream);

/* Extended form of fa_fwd: tile size, grid size, time limit and a debug trace. */
typedef struct fa_fwd_params {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, H, Sq, Sk, d;
  float scale;
  int mask_mode, window, n_global, dtype;
  int block_n;        /* key-block size: 0 = default (128), else 64 or 128 */
  int block_m;        /* query rows per work item: 0 = fa_fwd_default_block_m(mask_mode),
                         else 64 (tensor-core tiles of 64 rows), 128, or 256 (two 128-row
                         tiles sharing every K/V tile) */
  int num_ctas;       /* persistent grid size: 0 = one CTA per SM */
  int group_heads;    /* (batch, head) pairs scheduled together: 0 = sized for L2 */
  uint32_t timeout_us; /* per-wait time limit: 0 = 1 s */
  /* Optional visit log, int32 [B*H, ceil(Sq/T), ceil(Sk/block_n)] with T the rows of a
   * tensor-core tile (128, or 64 when block_m is 64), zeroed by the caller. Every tile the
   * kernel computes for those T queries adds 16 + class (1 partial, 2 full); tiles the
   * mask skips stay 0. */
  int32_t* trace;
  /* FA_MASK_BLOCK_SPARSE: device pointer to the layout described above (owned by the
   * caller, read during the call); ignored for the other masks. */
  const uint8_t* block_layout;
  /* FA_F32 (FP32 q, k, v and o, same shapes): device scratch of at least
   * fa_fwd_workspace_size(...) bytes, 16-byte aligned, owned by the caller and overwritten
   * by the call; unused for 16-bit inputs. Each input element x is held there as
   * hi = bf16(x) and lo = bf16(x - hi) (hi + lo = x to 2^-16 relative), and every product
   * of the method (Q K^T and P V) is formed as hi*hi + hi*lo + lo*hi on the bf16 tensor
   * cores with FP32 accumulation, P being split the same way; block_n is 64 (0 or 64
   * accepted) and block_m 256 (0 or 256 accepted). Accuracy: the products' relative error
   * stays near 2^-15, far inside the 1e-3 bound on O that FP32 inputs are held to. */
  void* workspace;
  size_t workspace_bytes;
  /* Optional int32 [B*H, ceil(Sq/128)], zeroed by the caller: for every 128-query tile, the
   * number of (query row, key tile) steps at which the row's running maximum rose by more
   * than the lazy-rescale threshold (8 in log2 units) and its partial output and sum were
   * rescaled (the correction step of the per-block (m, l, O) recurrence, zwxr.cn article
   * on ops-transformer, section 3.1). For tests: it shows which inputs reach that step. */
  int32_t* rescale_count;
  /* Optional, FA_MASK_BLOCK_SPARSE: the same layout as block_layout in HOST memory (read
   * during the call). The device layout decides what is computed; this copy only plans the
   * work, weighing every work item by the key blocks its rows visit and handing the longest
   * items out first, where without it every item is weighed as dense. Results are the same,
   * bit for bit, whatever it holds (a wrong copy only costs balance). */
  const uint8_t* block_layout_host;
} fa_fwd_params;

fa_status fa_fwd_ex(const fa_fwd_params* params, fa_stream_t stream);

/* Bytes of workspace fa_fwd_ex needs: 4 * d * B * H * (Sq + 2 * Sk) for FA_F32 (a bf16
 * high and low plane of every Q, K and V element), 0 for FA_F16 / FA_BF16 and for
 * invalid sizes. */
size_t fa_fwd_workspace_size(int B, int H, int Sq, int Sk, int d, int dtype);

/* Query rows per tensor-core tile of the 128- and 256-row items (128): the row granularity of
 * the fa_fwd_ex trace; items of block_m = 64 use 64-row tiles, and so do their trace rows. */
int fa_fwd_block_m(void);

/* Query rows per work item that fa_fwd (and fa_fwd_ex with block_m = 0) uses for a mask:
 * 256 (two 128-row tiles sharing every K/V tile) except for FA_MASK_BAND, whose narrow
 * key ranges favour 128, and FA_MASK_BLOCK_SPARSE, where a 256-row item would visit the
 * union of two layout rows. fa_fwd_paged uses the same choice. Returns 0 for an unknown
 * mask. */
int fa_fwd_default_block_m(int mask_mode);

/*
 * fa_bwd - gradients of fa_fwd for an upstream gradient dout: with P the softmax of
 * fa_fwd (recomputed from the saved LSE, as the pages' remark on re-reading the scores in
 * the backward pass implies; zwxr.cn article on ops-transformer, section 3.1) and
 * D_i = dout_i . o_i,
 *     dv = P^T dout,  dS = P (dout v^T - D),  dq = scale dS k,  dk = scale dS^T q.
 *   q, o, dout, dq [B, H, Sq, d]; k, v, dk, dv [B, H, Sk, d]: dtype, contiguous, device
 *   lse        [B, H, Sq] float32, the natural-log LSE that fa_fwd returned with o
 *   workspace  device scratch, 16-byte aligned, owned by the caller: an FP32 dq
 *              accumulator of B*H*ceil(Sq/4)*4*d floats followed by D [B, H, Sq], i.e.
 *              B*H*(ceil(Sq/4)*4*d + Sq)*4 bytes; fa_bwd_workspace_size(B, H, Sq) returns
 *              that size for d = 128, enough for every supported d. Its contents on entry
 *              do not matter.
 *   d, scale, mask_mode / window / n_global, dtype as for fa_fwd; FA_MASK_BLOCK_SPARSE goes
 *   through fa_bwd_block_sparse (here it is FA_ERR_UNSUPPORTED). dq, dk and dv are written
 *   (RN from FP32 accumulators); a key no query sees gets dk = dv = 0, a query that sees no
 *   key dq = 0. dq sums the
 *   contributions of the key blocks with FP32 atomic additions, so its last bit can differ
 *   between runs; dk and dv are the same on every run.
 */
size_t fa_bwd_workspace_size(int B, int H, int Sq);
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace,
                 size_t workspace_bytes, int B, int H, int Sq, int Sk, int d, float scale,
                 int mask_mode, int window, int n_global, int dtype, fa_stream_t stream);

/*
 * fa_bwd_block_sparse - fa_bwd under FA_MASK_BLOCK_SPARSE: block_layout is the device layout
 * of the forward call, uint8 [H][ceil(Sq/128)][ceil(Sk/128)] (query i of head h sees key j
 * iff block_layout[h][i/128][j/128] != 0; read during the call). Every other argument as for
 * fa_bwd. A key no query sees gets dk = dv = 0, a query that sees no key dq = 0.
 */
fa_status fa_bwd_block_sparse(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              void* workspace, size_t workspace_bytes, int B, int H, int Sq,
                              int Sk, int d, float scale, const uint8_t* block_layout, int dtype,
                              fa_stream_t stream);

/*
 * fa_decode_paged - one query token per sequence against a paged KV cache
 * ("ascend-transformer-boost 实战" (ai6s.net), scenario 2: the cache is cut into
 * fixed-size pages, 256 tokens in the pages' example, and new pages are taken as a
 * sequence grows). The query of sequence b sits at position ctx_lens[b]-1 and sees
 * all ctx_lens[b] cached tokens; token t is stored in physical page
 * block_table[b, t / page_size] at offset t % page_size.
 *   q            [B, H, d]  dtype
 *   k_pages      [num_pages, H, page_size, d]  dtype (one (page, head) run is contiguous)
 *   v_pages      [num_pages, H, page_size, d]  dtype
 *   block_table  int32 [B, max_pages_per_seq]; entries past a sequence's last page
 *                are not read. An entry outside [0, num_pages) that would be read is
 *                skipped on the device and reported as FA_ERR_BAD_PAGE.
 *   ctx_lens     int32 [B], each in [0, page_size * max_pages_per_seq]; a value outside
 *                that range is clamped into it on the device and reported as
 *                FA_ERR_BAD_PAGE.
 *   o            [B, H, d]  dtype;  lse [B, H] float32 (may be NULL)
 *   d            64 or 128;  page_size a multiple of 16 in [16, 4096]
 *   workspace    device scratch of at least fa_decode_workspace_size(...) bytes,
 *                owned by the caller; its contents need no initialisation.
 * Two kernels run on `stream`: split-K partial attention over runs of pages, then
 * the merge of the partials. Pools that both start on a 32-byte boundary are read 32
 * bytes per access, others (16-byte aligned, as every pointer here must be) 16 bytes
 * per access; the two differ only in the order of their FP32 sums.
 */
fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                          const int32_t* block_table, const int32_t* ctx_lens, void* o, float* lse,
                          int B, int H, int d, int page_size, int max_pages_per_seq, int num_pages,
                          float scale, int dtype, void* workspace, size_t workspace_bytes,
                          fa_stream_t stream);

/* Bytes of workspace fa_decode_paged needs for these sizes (any split choice). */
size_t fa_decode_workspace_size(int B, int H, int d, int max_pages_per_seq, int page_size);

/* Extended form of fa_decode_paged: split size and debug traces. */
typedef struct fa_decode_params {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const int32_t* block_table;
  const int32_t* ctx_lens;
  void* o;
  float* lse;
  int B, H, d, page_size, max_pages_per_seq, num_pages;
  float scale;
  int dtype;
  void* workspace;
  size_t workspace_bytes;
  int pages_per_split; /* pages per split-K partial: 0 = default */
  /* Optional int32 [B*H, max_pages_per_seq], filled with -1 by the caller: the
   * physical page each logical page was read from. */
  int32_t* trace_pages;
  /* Optional int32 [B*H, ceil(max_pages_per_seq / pages_per_split), 2]: the token
   * range [t0, t1) of every split. */
  int32_t* trace_splits;
} fa_decode_params;

fa_status fa_decode_paged_ex(const fa_decode_params* params, fa_stream_t stream);

/* Pages per split that fa_decode_paged picks for these sizes. */
int fa_decode_default_pages_per_split(int B, int H, int max_pages_per_seq);

/*
 * fa_kv_append - write a chunk of new tokens into a paged KV cache ("ascend-transformer-
 * boost 实战" (ai6s.net), scenario 2: fixed-size pages, a new page taken as a sequence
 * grows). Token t < n_b of sequence b (n_b = new_lens[b], or T when new_lens is NULL) is
 * stored at position ctx_lens[b] + t: page block_table[b, pos / page_size], offset
 * pos % page_size. The caller puts the pages the chunk needs into the table beforehand
 * and adds n_b to ctx_lens afterwards (the call does not change ctx_lens). The slots of
 * the chunk's last page after its last token are set to zero, so every slot a paged
 * prefill may read past a sequence's end holds a finite value.
 *   k_new, v_new  [B, H, T, d] dtype (contiguous)
 *   k_pages, v_pages [num_pages, H, page_size, d] dtype, written in place
 *   block_table   int32 [B, max_pages_per_seq];  ctx_lens int32 [B];  new_lens int32 [B] or NULL
 *   d 64 or 128; page_size a multiple of 16 in [16, 4096].
 * A table entry outside [0, num_pages), or ctx + n_b beyond page_size*max_pages_per_seq,
 * is skipped on the device and reported as FA_ERR_BAD_PAGE.
 */
fa_status fa_kv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                       const int32_t* block_table, const int32_t* ctx_lens,
                       const int32_t* new_lens, int B, int H, int T, int d, int page_size,
                       int max_pages_per_seq, int num_pages, int dtype, fa_stream_t stream);

/*
 * fa_fwd_paged - chunked prefill against a paged KV cache: the Sq queries of sequence b
 * are its last Sq tokens, at key positions ctx_lens[b]-Sq .. ctx_lens[b]-1, and attend
 * to its ctx_lens[b] cached keys (K/V appended beforehand, e.g. with fa_kv_append) under
 * the given mask, exactly as fa_fwd with Sk = ctx_lens[b] would over the gathered keys.
 *   q, o          [B, H, Sq, d] dtype;  lse [B, H, Sq] float32 or NULL
 *   k_pages, v_pages, block_table, ctx_lens, page_size, max_pages_per_seq, num_pages
 *                 as for fa_decode_paged, except page_size: a multiple of 64 in [64, 4096]
 *                 (a key tile never crosses a page)
 *   mask_mode, window, n_global, scale, dtype as for fa_fwd.
 * The key tiles of a sequence's last page are read whole: slots past ctx_lens[b] must
 * hold finite values (fa_kv_append guarantees it). Lengths are read on the device; a
 * length above page_size*max_pages_per_seq is clamped and an out-of-range page is
 * replaced by page 0 and reported as FA_ERR_BAD_PAGE.
 */
fa_status fa_fwd_paged(const void* q, const void* k_pages, const void* v_pages,
                       const int32_t* block_table, const int32_t* ctx_lens, void* o, float* lse,
                       int B, int H, int Sq, int d, int page_size, int max_pages_per_seq,
                       int num_pages, float scale, int mask_mode, int window, int n_global,
                       int dtype, fa_stream_t stream);

/*
 * fa_fwd_paged_host_lens - fa_fwd_paged for a caller that also holds the context lengths in
 * HOST memory: ctx_lens_host[B] (int32, read during the call) should equal ctx_lens on the
 * device. The lengths on the device still decide what is computed; the host copy only
 * plans the work, weighing every (sequence, head, query block) item by the keys it visits
 * and handing the longest items out first, where fa_fwd_paged, which cannot read device
 * lengths without synchronising, weighs every item by the pool capacity
 * page_size*max_pages_per_seq. With sequences of different lengths that balances the SMs'
 * work; the results are the same as fa_fwd_paged's, bit for bit, whatever the host copy
 * holds (a wrong copy only costs balance). ctx_lens_host = NULL is fa_fwd_paged.
 */
fa_status fa_fwd_paged_host_lens(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table, const int32_t* ctx_lens,
                                 const int32_t* ctx_lens_host, void* o, float* lse, int B, int H,
                                 int Sq, int d, int page_size, int max_pages_per_seq,
                                 int num_pages, float scale, int mask_mode, int window,
                                 int n_global, int dtype, fa_stream_t stream);

/*
 * fa_merge_partials - combine two attention results that cover disjoint key sets of the
 * same queries (for example the text-to-text causal call and the text-to-vision cross
 * call of a multimodal layer). Splitting an attention into such calls is exact
 * ("ascend-transformer-boost 实战" (ai6s.net), scenario 4); with M = max(lse_a, lse_b)
 * and w_x = exp(lse_x - M):
 *     o = (w_a o_a + w_b o_b) / (w_a + w_b),   lse = M + ln(w_a + w_b).
 * A part whose LSE is -inf contributes nothing; two empty parts give o = 0, lse = -inf.
 *   o_a, o_b, o   [rows, d] dtype (for example [B,H,Sq,d] flattened); o may alias o_a
 *   lse_a, lse_b  [rows] float32 natural-log LSEs, as fa_fwd writes them
 *   lse           [rows] float32, may be NULL; must not overlap lse_a or lse_b
 *   d 64 or 128; dtype FA_F16 or FA_BF16.
 */
fa_status fa_merge_partials(const void* o_a, const float* lse_a, const void* o_b,
                            const float* lse_b, void* o, float* lse, int64_t rows, int d,
                            int dtype, fa_stream_t stream);

/*
 * fa_decode_paged_noalloc - fa_decode_paged for callers that cannot allocate device
 * memory. The pages have no counterpart for this call; it exists for users of this
 * library whose device memory is fixed when they start (a serving loop with a set
 * budget) or owned entirely by a host program that gives its plug-ins no allocator,
 * so they cannot provide the workspace fa_decode_paged needs.
 *   Arguments, layouts and results are those of fa_decode_paged without `workspace`
 *   and `workspace_bytes`; the caller still owns and passes every input and output.
 *   The split partials go to a scratch array built into the library: 16 MiB on every
 *   GPU that loads it, held until the process exits. The call allocates nothing.
 *   The split size is fa_decode_paged's default; the partials fit whenever
 *   B*H*(d+2)*4 bytes (one split per sequence) do, i.e. B*H <= 32263 at d = 128, and
 *   beyond that the call returns FA_ERR_INVALID_ARG and launches nothing.
 *   The first call on each device, with that device current, looks up the scratch
 *   array's device address and keeps it; make that first call before any stream
 *   capture. After cudaDeviceReset in this process that address is stale: calls made
 *   after a reset are not supported.
 *   Every call on a device shares the one array: calls whose kernels overlap on the
 *   GPU (for example on two streams) race and must be ordered by the caller.
 */
fa_status fa_decode_paged_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                  const int32_t* block_table, const int32_t* ctx_lens, void* o,
                                  float* lse, int B, int H, int d, int page_size,
                                  int max_pages_per_seq, int num_pages, float scale, int dtype,
                                  fa_stream_t stream);

/*
 * fa_get_device_status - synchronise `stream`, then read and clear the device
 * status word. Returns FA_OK, FA_ERR_BAD_PAGE or FA_ERR_TIMEOUT (FA_ERR_CUDA if the
 * stream itself failed). FA_ERR_UNSUPPORTED means that a backward kernel found its dynamic
 * shared memory starting more than 256 bytes past a 1024-byte boundary, which its layout
 * at d = 128 cannot absorb, and wrote nothing (dynamic shared memory starts on such a
 * boundary on the devices this library targets).
 */
fa_status fa_get_device_status(fa_stream_t stream);

/*
 * fa_selftest_timeout - launch one tiny kernel that waits on a pipeline barrier
 * nothing will ever complete, with the given time limit (microseconds, 1..10^6).
 * The wait runs out, the kernel records FA_ERR_TIMEOUT in the device status word
 * and returns; the context stays usable. For testing the failure path.
 */
fa_status fa_selftest_timeout(uint32_t timeout_us, fa_stream_t stream);

const char* fa_last_error_string(void);
int fa_version(void); /* major*10000 + minor*100 + patch */

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
