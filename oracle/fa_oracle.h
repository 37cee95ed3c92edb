/*
 * FP64 CPU oracle for FlashAttention forward (prefill and paged decode).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, includes or
 * calls this code; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it. It shares no source with the CUDA path.
 *
 * What it computes is the plain definition of attention that the pages start
 * from ("ops-transformer" overview on gitcode.csdn.net, section 二.1
 * "FlashAttention算子", the "traditional attention" listing):
 *     O = softmax(scale * Q K^T + mask) V,   per (batch, head),
 * with the score row materialised in double precision. The log-sum-exp
 * LSE_i = m_i + ln sum_j exp(s_ij - m_i) is returned beside O.
 *
 * Inputs are read as their exact stored values: 16-bit floats are decoded
 * bit by bit into doubles here, so input rounding is never counted as error.
 */
#ifndef FA_ORACLE_H
#define FA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types the oracle can read */
enum { OR_F16 = 0, OR_BF16 = 1, OR_F32 = 2, OR_F64 = 3 };
/* mask modes (same numbering as the library's public enum, chosen independently) */
enum { OR_MASK_NONE = 0, OR_MASK_CAUSAL = 1, OR_MASK_CAUSAL_WINDOW = 2, OR_MASK_BAND = 3,
       OR_MASK_PREFIX_LM = 4 };
/* tile classes */
enum { OR_TILE_EMPTY = 0, OR_TILE_PARTIAL = 1, OR_TILE_FULL = 2 };
/* online-recurrence variants (see or_online_attention) */
enum { OR_REC_UNNORMALISED = 0, OR_REC_NORMALISED = 1, OR_REC_LITERAL_P2 = 2 };

double or_elem(const void* base, int64_t idx, int dtype);
void or_decode(const void* src, double* dst, int64_t n, int dtype);

int or_visible(int64_t i, int64_t j, int64_t Sq, int64_t Sk, int mask_mode,
               int64_t window, int64_t n_global);
int64_t or_count_visible(int64_t Sq, int64_t Sk, int mask_mode, int64_t window,
                         int64_t n_global);
int or_tile_class(int64_t mb, int64_t nb, int64_t BM, int64_t BN, int64_t Sq,
                  int64_t Sk, int mask_mode, int64_t window, int64_t n_global);

int or_attention(const void* q, const void* k, const void* v, int dtype,
                 double* o, double* lse, int64_t B, int64_t H, int64_t Sq,
                 int64_t Sk, int64_t d, double scale, int mask_mode,
                 int64_t window, int64_t n_global, const int64_t* rows,
                 int64_t nrows, double* max_psum_err, int nthreads);

int or_online_attention(const void* q, const void* k, const void* v, int dtype,
                        double* o, double* lse, int64_t B, int64_t H,
                        int64_t Sq, int64_t Sk, int64_t d, double scale,
                        int mask_mode, int64_t window, int64_t n_global,
                        int64_t block_n, double tau, int variant);

/* Rescale events of the lazy online recurrence (threshold tau, natural-log
   units), summed per tile of tile_rows query rows: counts and near-threshold
   decisions (|margin| < eps), each int64 [B*H*ceil(Sq/tile_rows)]. layout may
   be NULL (closed-form mask) or a block layout as in or_attention_layout. */
int or_rescale_events(const void* q, const void* k, int dtype, int64_t B, int64_t H,
                      int64_t Sq, int64_t Sk, int64_t d, double scale, int mask_mode,
                      int64_t window, int64_t n_global, const uint8_t* layout, int64_t blk,
                      int64_t block_n, double tau, int64_t tile_rows, double eps,
                      int64_t* counts, int64_t* near, int nthreads);

int or_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                    int dtype, const int32_t* block_table,
                    const int32_t* ctx_lens, double* o, double* lse, int64_t B,
                    int64_t H, int64_t d, int64_t page_size,
                    int64_t max_pages_per_seq, int64_t num_pages, double scale,
                    const int64_t* bh_list, int64_t n_bh, int nthreads);

int or_attention_paged(const void* q, const void* k_pages, const void* v_pages, int dtype,
                       const int32_t* block_table, const int32_t* ctx_lens, double* o,
                       double* lse, int64_t B, int64_t H, int64_t Sq, int64_t d,
                       int64_t page_size, int64_t max_pages_per_seq, int64_t num_pages,
                       double scale, int mask_mode, int64_t window, int64_t n_global,
                       int nthreads);

/* Attention under a block-sparse layout uint8 [H][ceil(Sq/blk)][ceil(Sk/blk)] shared by
   every batch entry: query i of head h sees key j iff its block is non-zero. rows as in
   or_attention (NULL: every row). */
int or_attention_layout(const void* q, const void* k, const void* v, int dtype,
                        double* o, double* lse, int64_t B, int64_t H, int64_t Sq,
                        int64_t Sk, int64_t d, double scale, const uint8_t* layout,
                        int64_t blk, const int64_t* rows, int64_t nrows, int nthreads);
int64_t or_count_visible_layout(int64_t H, int64_t Sq, int64_t Sk, const uint8_t* layout,
                                int64_t blk);
int or_tile_class_layout(int64_t h, int64_t mb, int64_t nb, int64_t BM, int64_t BN,
                         int64_t Sq, int64_t Sk, const uint8_t* layout, int64_t blk);

/* Gradients dq [B,H,Sq,d], dk and dv [B,H,Sk,d] (FP64) of attention for the upstream
   gradient dout [B,H,Sq,d] (same dtype as q, k, v), by the chain rule. */
int or_attention_backward(const void* q, const void* k, const void* v, const void* dout,
                          int dtype, double* dq, double* dk, double* dv, int64_t B, int64_t H,
                          int64_t Sq, int64_t Sk, int64_t d, double scale, int mask_mode,
                          int64_t window, int64_t n_global, int nthreads);
int or_attention_backward_layout(const void* q, const void* k, const void* v, const void* dout,
                                 int dtype, double* dq, double* dk, double* dv, int64_t B,
                                 int64_t H, int64_t Sq, int64_t Sk, int64_t d, double scale,
                                 const unsigned char* layout, int64_t blk, int nthreads);

void or_combine_partials(const double* m, const double* l, const double* acc,
                         int64_t nsplit, int64_t d, double* o, double* lse);

void or_decode_split_tokens(int64_t ctx_len, int64_t page_size,
                            int64_t pages_per_split, int64_t split,
                            int64_t* t0, int64_t* t1);

#ifdef __cplusplus
}
#endif
#endif
