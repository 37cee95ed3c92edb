/*
 * FP64 CPU oracle for FlashAttention forward. TEST INFRASTRUCTURE ONLY: the
 * product library never links or calls it (see fa_oracle.h).
 *
 * Page references used below:
 *   [ops-transformer]  "ops-transformer" operator-library overview
 *                      (gitcode.csdn.net), section 二.1 "FlashAttention算子":
 *                      the traditional-attention listing and the tiled
 *                      online-softmax loop with a single final normalisation.
 *   [Ascend-FA]        zwxr.cn article on ops-transformer, section 3.1
 *                      "FlashAttention的昇腾魔改": per-block recurrence for
 *                      (m, l, O); section 5.1: softmax denominator in FP32.
 *   [boost]            "ascend-transformer-boost 实战" (ai6s.net):
 *                      scenario 2 (paged KV cache, 256-token pages),
 *                      scenario 3 (sliding window 2048 + 64 global tokens),
 *                      scenario 4 (splitting one attention into several
 *                      calls is mathematically equivalent).
 *
 * Parity status of each function (what pins it, in tests/test_oracle_pins.py):
 *   or_elem/or_decode      pinned against numpy's IEEE half / bf16 decoding
 *   or_visible             pinned by hand-enumerated small masks and closed-form
 *                          pair counts
 *   or_count_visible       pinned by closed-form pair counts
 *   or_tile_class          pinned by hand-classified small grids
 *   or_attention           pinned by closed forms (constant scores, one-hot,
 *                          causal row 0, hand-worked examples), invariances,
 *                          special cases and a library routine (torch SDPA in
 *                          float64 with an explicit boolean mask)
 *   or_online_attention    pinned against or_attention and against the closed
 *                          forms; the literal page-2 update is shown to differ
 *   or_decode_paged        pinned by special cases (ctx = 1, identity table)
 *   or_attention_paged     pinned against or_attention on gathered keys (identity and
 *                          permuted tables) and against or_decode_paged (Sq = 1)
 *   or_combine_partials    pinned by split invariance against unsplit softmax
 *   or_decode_split_tokens pinned by partition invariants (cover, disjoint)
 *   or_attention_layout    pinned against or_attention (all-ones layout = no mask;
 *                          block 1 with a lower-triangular layout = causal), against
 *                          torch SDPA in float64 with the layout expanded into an
 *                          explicit boolean mask, and by key-block permutation
 *                          invariance
 *   or_count_visible_layout / or_tile_class_layout
 *                          pinned by closed-form counts and hand-classified grids
 *   or_attention_backward  pinned by central finite differences of or_attention in
 *                          FP64, by torch autograd on SDPA in float64 with an explicit
 *                          mask, and by closed forms (zero queries: dK = 0; a row with one
 *                          visible key: dQ = 0; rows of dS sum to 0)
 *   or_attention_backward_layout
 *                          pinned by torch autograd on SDPA in float64 with the layout
 *                          expanded into an explicit mask, against or_attention_backward
 *                          (block 1 with a lower-triangular layout = causal), and per head
 *                          (heads with different layouts)
 */
#include "fa_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* element decoding: the exact value of each stored input element       */
/* ------------------------------------------------------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_bits_value(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1.f) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_value(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

double or_elem(const void* base, int64_t idx, int dtype) {
    switch (dtype) {
    case OR_F16: return half_bits_value(((const uint16_t*)base)[idx]);
    case OR_BF16: return bf16_bits_value(((const uint16_t*)base)[idx]);
    case OR_F32: return (double)((const float*)base)[idx];
    default: return ((const double*)base)[idx];
    }
}

void or_decode(const void* src, double* dst, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) dst[i] = or_elem(src, i, dtype);
}

static size_t elem_size(int dtype) {
    return dtype == OR_F64 ? 8 : dtype == OR_F32 ? 4 : 2;
}

/* ------------------------------------------------------------------ */
/* the mask                                                            */
/* ------------------------------------------------------------------ */

/*
 * Vis(i): which keys j query i may attend to. Queries and keys are aligned at
 * the bottom-right (delta = Sk - Sq), so query i sits at key position i+delta.
 *   NONE           every key.
 *   CAUSAL         j <= i+delta                    ([ops-transformer] section 四,
 *                                                   causal=True).
 *   CAUSAL_WINDOW  j <= i+delta and (i+delta-j < window or j < n_global)
 *                  ([boost] scenario 3: a sliding window plus global tokens
 *                  such as BOS, read causally: the window holds `window` keys
 *                  counting the query's own position; the global tokens are
 *                  the first n_global key positions).
 *   BAND           |i+delta - j| <= window: the diagonal band of [Ascend-FA]
 *                  section 3.2, each token seeing the tokens within +-w of it.
 *   PREFIX_LM      j <= i+delta or j < n_global: the first n_global keys (the
 *                  prefix) are seen by every query, the rest causally (the
 *                  prefix-LM variant [boost] scenario 3 lists by name; the
 *                  pages define it no further).
 */
int or_visible(int64_t i, int64_t j, int64_t Sq, int64_t Sk, int mask_mode,
               int64_t window, int64_t n_global) {
    int64_t pos = i + (Sk - Sq);
    if (i < 0 || i >= Sq || j < 0 || j >= Sk) return 0;
    if (mask_mode == OR_MASK_NONE) return 1;
    if (mask_mode == OR_MASK_BAND) return (j - pos <= window) && (pos - j <= window);
    if (mask_mode == OR_MASK_PREFIX_LM) return (j <= pos) || (j < n_global);
    if (j > pos) return 0;
    if (mask_mode == OR_MASK_CAUSAL) return 1;
    return (pos - j < window) || (j < n_global);
}

int64_t or_count_visible(int64_t Sq, int64_t Sk, int mask_mode, int64_t window,
                         int64_t n_global) {
    int64_t total = 0;
    for (int64_t i = 0; i < Sq; ++i)
        for (int64_t j = 0; j < Sk; ++j)
            total += or_visible(i, j, Sq, Sk, mask_mode, window, n_global);
    return total;
}

/*
 * Class of the (mb, nb) tile of BM query rows x BN key columns, by brute force
 * over its pairs. A pair outside [0,Sq) x [0,Sk) counts as not visible, so a
 * tile that hangs over the end of either sequence is never FULL.
 */
int or_tile_class(int64_t mb, int64_t nb, int64_t BM, int64_t BN, int64_t Sq,
                  int64_t Sk, int mask_mode, int64_t window, int64_t n_global) {
    int64_t vis = 0;
    for (int64_t i = mb * BM; i < mb * BM + BM; ++i)
        for (int64_t j = nb * BN; j < nb * BN + BN; ++j)
            vis += or_visible(i, j, Sq, Sk, mask_mode, window, n_global);
    if (vis == 0) return OR_TILE_EMPTY;
    if (vis == BM * BN) return OR_TILE_FULL;
    return OR_TILE_PARTIAL;
}

/* ------------------------------------------------------------------ */
/* attention by its definition                                         */
/* ------------------------------------------------------------------ */

/*
 * One query row against an explicit list of key/value rows, by the definition:
 *   s_j = scale * sum_c q_c k_jc,  m = max_j s_j,
 *   P_j = exp(s_j - m) / sum_t exp(s_t - m),  O = sum_j P_j v_j,
 *   LSE = m + ln sum_t exp(s_t - m).
 * An empty list gives O = 0 and LSE = -inf.
 * krows[t] / vrows[t] point at the t-th key / value row (already decoded).
 */
static void attend_row(const double* q, const double* const* krows,
                       const double* const* vrows, int64_t n, int64_t d,
                       double scale, double* s, double* o, double* lse,
                       double* psum_err) {
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        *psum_err = 0.0;
        return;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += q[c] * krows[t][c];
        s[t] = scale * dot;
        if (s[t] > m) m = s[t];
    }
    double z = 0.0;
    for (int64_t t = 0; t < n; ++t) z += exp(s[t] - m);
    double psum = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        double p = exp(s[t] - m) / z;
        psum += p;
        for (int64_t c = 0; c < d; ++c) o[c] += p * vrows[t][c];
    }
    *lse = m + log(z);
    *psum_err = fabs(1.0 - psum);
}

static int cmp_i64(const void* a, const void* b) {
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

/*
 * Attention over [B,H,Sq,d] queries and [B,H,Sk,d] keys/values (contiguous).
 * rows == NULL: every row; o is [B,H,Sq,d] and lse [B,H,Sq].
 * otherwise rows[r] = (b*H + h)*Sq + i and o is [nrows,d], lse [nrows].
 * max_psum_err (may be NULL) receives max over rows of |1 - sum_j P_j|.
 * The work is split by (batch, head): each slice of K and V is decoded once.
 * Returns 0, or -1 on a bad argument.
 */
int or_attention(const void* q, const void* k, const void* v, int dtype,
                 double* o, double* lse, int64_t B, int64_t H, int64_t Sq,
                 int64_t Sk, int64_t d, double scale, int mask_mode,
                 int64_t window, int64_t n_global, const int64_t* rows,
                 int64_t nrows, double* max_psum_err, int nthreads) {
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || d <= 0) return -1;
    if (mask_mode < OR_MASK_NONE || mask_mode > OR_MASK_PREFIX_LM) return -1;
    if (mask_mode == OR_MASK_CAUSAL_WINDOW && (window < 1 || n_global < 0)) return -1;
    if (mask_mode == OR_MASK_BAND && window < 0) return -1;
    if (mask_mode == OR_MASK_PREFIX_LM && n_global < 0) return -1;
    int64_t n_out = rows ? nrows : B * H * Sq;
    /* order[r] = output index r, sorted by the row it asks for, so that the rows
       of one (batch, head) are contiguous */
    int64_t* order = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)(n_out > 0 ? n_out : 1));
    for (int64_t r = 0; r < n_out; ++r) {
        int64_t row = rows ? rows[r] : r;
        if (row < 0 || row >= B * H * Sq) {
            free(order);
            return -1;
        }
        order[2 * r] = row;
        order[2 * r + 1] = r;
    }
    qsort(order, (size_t)n_out, 2 * sizeof(int64_t), cmp_i64);
    double worst = 0.0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(max : worst)
#endif
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        size_t skd = (size_t)(Sk > 0 ? Sk : 1) * (size_t)d;
        double* kd = (double*)malloc(sizeof(double) * skd);
        double* vd = (double*)malloc(sizeof(double) * skd);
        double* s = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1));
        const double** kr = (const double**)malloc(sizeof(double*) * (size_t)(Sk > 0 ? Sk : 1));
        const double** vr = (const double**)malloc(sizeof(double*) * (size_t)(Sk > 0 ? Sk : 1));
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bh = 0; bh < B * H; ++bh) {
            /* the output rows that belong to this (batch, head) */
            int64_t lo = 0, hi = n_out;
            while (lo < hi) {
                int64_t mid = (lo + hi) / 2;
                if (order[2 * mid] < bh * Sq) lo = mid + 1; else hi = mid;
            }
            int64_t first = lo;
            if (first >= n_out || order[2 * first] >= (bh + 1) * Sq) continue;
            or_decode((const char*)k + (size_t)(bh * Sk * d) * elem_size(dtype), kd, Sk * d, dtype);
            or_decode((const char*)v + (size_t)(bh * Sk * d) * elem_size(dtype), vd, Sk * d, dtype);
            for (int64_t r = first; r < n_out && order[2 * r] < (bh + 1) * Sq; ++r) {
                int64_t row = order[2 * r], out = order[2 * r + 1];
                int64_t i = row - bh * Sq;
                for (int64_t c = 0; c < d; ++c) qrow[c] = or_elem(q, row * d + c, dtype);
                int64_t n = 0;
                for (int64_t j = 0; j < Sk; ++j)
                    if (or_visible(i, j, Sq, Sk, mask_mode, window, n_global)) {
                        kr[n] = kd + j * d;
                        vr[n] = vd + j * d;
                        ++n;
                    }
                double err;
                attend_row(qrow, kr, vr, n, d, scale, s, o + out * d, lse + out, &err);
                if (err > worst) worst = err;
            }
        }
        free(qrow);
        free(kd);
        free(vd);
        free(s);
        free(kr);
        free(vr);
    }
    free(order);
    if (max_psum_err) *max_psum_err = worst;
    return 0;
}

/* ------------------------------------------------------------------ */
/* the blocked online recurrence, in the pages' order                  */
/* ------------------------------------------------------------------ */

/*
 * The tiled loop of [ops-transformer] 二.1 for every row: walk the keys in
 * blocks of block_n, keep a running maximum m and running sum l, and fold each
 * block into the output. Three forms of the per-block update:
 *
 *   OR_REC_UNNORMALISED  ([ops-transformer]: statistics updated per block,
 *       one normalisation at the end). The accumulator and l share a
 *       reference maximum m_ref; when a block raises the running maximum by
 *       more than tau (natural-log units) both are multiplied by
 *       exp(m_ref - m_new) and m_ref moves up. tau = 0 rescales on every
 *       increase. p_j = exp(s_j - m_ref); l += sum p; acc += sum p_j v_j;
 *       at the end O = acc / l, LSE = m_ref + ln l.
 *   OR_REC_NORMALISED    ([Ascend-FA] 3.1 read with its lost factor restored):
 *       m_new = max(m, block max); l_new = exp(m - m_new) l + sum exp(s - m_new);
 *       O = (l exp(m - m_new) O + sum exp(s_j - m_new) v_j) / l_new.
 *   OR_REC_LITERAL_P2    ([Ascend-FA] 3.1 as printed): the old-output term is
 *       divided by l_new without the factor l. Kept only so that a test can
 *       show this printed form is not the softmax.
 *
 * Output layout as or_attention with rows == NULL.
 */
int or_online_attention(const void* q, const void* k, const void* v, int dtype,
                        double* o, double* lse, int64_t B, int64_t H,
                        int64_t Sq, int64_t Sk, int64_t d, double scale,
                        int mask_mode, int64_t window, int64_t n_global,
                        int64_t block_n, double tau, int variant) {
    if (block_n < 1 || d <= 0 || B < 0 || H < 0 || Sq < 0 || Sk < 0) return -1;
    double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)block_n);
    int* vis = (int*)malloc(sizeof(int) * (size_t)block_n);
    for (int64_t bh = 0; bh < B * H; ++bh) {
        for (int64_t i = 0; i < Sq; ++i) {
            int64_t row = bh * Sq + i;
            for (int64_t c = 0; c < d; ++c) {
                qrow[c] = or_elem(q, row * d + c, dtype);
                acc[c] = 0.0;
            }
            double m = -INFINITY, l = 0.0;
            for (int64_t j0 = 0; j0 < Sk; j0 += block_n) {
                int64_t nb = (Sk - j0 < block_n) ? Sk - j0 : block_n;
                double bmax = -INFINITY;
                for (int64_t t = 0; t < nb; ++t) {
                    int64_t j = j0 + t;
                    vis[t] = or_visible(i, j, Sq, Sk, mask_mode, window, n_global);
                    if (!vis[t]) continue;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c)
                        dot += qrow[c] * or_elem(k, (bh * Sk + j) * d + c, dtype);
                    s[t] = scale * dot;
                    if (s[t] > bmax) bmax = s[t];
                }
                if (bmax == -INFINITY) continue; /* nothing visible in this block */
                double m_new = bmax > m ? bmax : m;
                if (variant == OR_REC_UNNORMALISED) {
                    if (m == -INFINITY) {
                        m = m_new; /* first visible block: m is the reference */
                    } else if (m_new - m > tau) {
                        double a = exp(m - m_new);
                        l *= a;
                        for (int64_t c = 0; c < d; ++c) acc[c] *= a;
                        m = m_new;
                    }
                    for (int64_t t = 0; t < nb; ++t) {
                        if (!vis[t]) continue;
                        double p = exp(s[t] - m);
                        l += p;
                        for (int64_t c = 0; c < d; ++c)
                            acc[c] += p * or_elem(v, (bh * Sk + j0 + t) * d + c, dtype);
                    }
                } else {
                    double a = (m == -INFINITY) ? 0.0 : exp(m - m_new);
                    double bsum = 0.0;
                    for (int64_t t = 0; t < nb; ++t)
                        if (vis[t]) bsum += exp(s[t] - m_new);
                    double l_new = a * l + bsum;
                    double keep = (variant == OR_REC_NORMALISED) ? l * a / l_new : a / l_new;
                    for (int64_t c = 0; c < d; ++c) {
                        double pv = 0.0;
                        for (int64_t t = 0; t < nb; ++t)
                            if (vis[t])
                                pv += exp(s[t] - m_new) *
                                      or_elem(v, (bh * Sk + j0 + t) * d + c, dtype);
                        acc[c] = acc[c] * keep + pv / l_new;
                    }
                    m = m_new;
                    l = l_new;
                }
            }
            double* orow = o + row * d;
            if (l == 0.0) {
                for (int64_t c = 0; c < d; ++c) orow[c] = 0.0;
                lse[row] = -INFINITY;
            } else if (variant == OR_REC_UNNORMALISED) {
                for (int64_t c = 0; c < d; ++c) orow[c] = acc[c] / l;
                lse[row] = m + log(l);
            } else {
                for (int64_t c = 0; c < d; ++c) orow[c] = acc[c];
                lse[row] = m + log(l);
            }
        }
    }
    free(qrow);
    free(acc);
    free(s);
    free(vis);
    return 0;
}

static int layout_visible(const uint8_t* layout, int64_t h, int64_t i, int64_t j,
                          int64_t nqb, int64_t nkb, int64_t blk);
static int layout_blk_bad(const uint8_t* layout, int64_t blk) { return layout && blk <= 0; }

/*
 * How often the lazy form of the recurrence above (OR_REC_UNNORMALISED with
 * threshold tau > 0, natural-log units) rescales: for every row, walk the keys
 * in blocks of block_n in ascending order, skip the blocks in which the row sees
 * no key, take the first visible block's maximum as the reference m, and count a
 * rescale at every later block whose maximum exceeds m + tau (m then moves up
 * to it). This is the correction step of the per-block (m, l, O) update
 * ([Ascend-FA] 3.1, O * exp(m - m_new)), taken only when the maximum has risen
 * far enough. Scores are s_j = scale * q . k_j in FP64 from the stored input
 * values.
 *
 * The counts are summed per tile of tile_rows consecutive query rows of one
 * (batch, head): counts[bh * ntiles + i / tile_rows], ntiles = ceil(Sq /
 * tile_rows). near[...] counts, likewise, the decisions whose margin
 * |(block max - m) - tau| is below eps: a computation in lower precision may
 * take those the other way. layout != NULL selects the block-sparse visibility
 * (blocks of blk, as or_attention_layout; mask_mode is then ignored).
 * Returns 0, or -1 on a bad argument.
 */
int or_rescale_events(const void* q, const void* k, int dtype, int64_t B, int64_t H,
                      int64_t Sq, int64_t Sk, int64_t d, double scale, int mask_mode,
                      int64_t window, int64_t n_global, const uint8_t* layout, int64_t blk,
                      int64_t block_n, double tau, int64_t tile_rows, double eps,
                      int64_t* counts, int64_t* near, int nthreads) {
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || d <= 0 || block_n < 1 || tile_rows < 1)
        return -1;
    if (!(tau > 0.0) || layout_blk_bad(layout, blk)) return -1;
    const int64_t ntiles = (Sq + tile_rows - 1) / tile_rows;
    const int64_t nqb = layout ? (Sq + blk - 1) / blk : 0, nkb = layout ? (Sk + blk - 1) / blk : 0;
    for (int64_t t = 0; t < B * H * ntiles; ++t) counts[t] = near[t] = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        double* kd = (double*)malloc(sizeof(double) * (size_t)(Sk > 0 ? Sk : 1) * (size_t)d);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bh = 0; bh < B * H; ++bh) {
            const int64_t h = bh % (H > 0 ? H : 1);
            or_decode((const char*)k + (size_t)(bh * Sk * d) * elem_size(dtype), kd, Sk * d, dtype);
            for (int64_t i = 0; i < Sq; ++i) {
                for (int64_t c = 0; c < d; ++c) qrow[c] = or_elem(q, (bh * Sq + i) * d + c, dtype);
                double m = -INFINITY;
                int64_t n_ev = 0, n_near = 0;
                for (int64_t j0 = 0; j0 < Sk; j0 += block_n) {
                    const int64_t j1 = (j0 + block_n < Sk) ? j0 + block_n : Sk;
                    double bmax = -INFINITY;
                    for (int64_t j = j0; j < j1; ++j) {
                        const int vis = layout ? layout_visible(layout, h, i, j, nqb, nkb, blk)
                                               : or_visible(i, j, Sq, Sk, mask_mode, window,
                                                            n_global);
                        if (!vis) continue;
                        double dot = 0.0;
                        for (int64_t c = 0; c < d; ++c) dot += qrow[c] * kd[j * d + c];
                        if (scale * dot > bmax) bmax = scale * dot;
                    }
                    if (bmax == -INFINITY) continue; /* the row sees nothing here */
                    if (m == -INFINITY) {
                        m = bmax;
                        continue;
                    }
                    if (fabs((bmax - m) - tau) < eps) ++n_near;
                    if (bmax - m > tau) {
                        ++n_ev;
                        m = bmax;
                    }
                }
                const int64_t t = bh * ntiles + i / tile_rows;
#ifdef _OPENMP
#pragma omp atomic
#endif
                counts[t] += n_ev;
#ifdef _OPENMP
#pragma omp atomic
#endif
                near[t] += n_near;
            }
        }
        free(qrow);
        free(kd);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* paged-KV decode                                                     */
/* ------------------------------------------------------------------ */

/*
 * Decode over a paged KV cache ([boost] scenario 2: the cache is split into
 * fixed-size pages, 256 tokens each in the pages' example). Sequence b has
 * ctx_lens[b] cached tokens; token t lives in physical page
 * block_table[b*max_pages_per_seq + t/page_size] at offset t % page_size.
 * Pools are [num_pages, H, page_size, d]; q and o are [B,H,d]; lse [B,H].
 * The single new query sits at position ctx-1 and sees every cached token,
 * so the result is the definition above over the gathered rows.
 * bh_list == NULL: all B*H pairs; else only bh_list[r] = b*H + h, packed.
 * Returns 0, or -1 if a needed table entry is out of range.
 */
int or_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                    int dtype, const int32_t* block_table,
                    const int32_t* ctx_lens, double* o, double* lse, int64_t B,
                    int64_t H, int64_t d, int64_t page_size,
                    int64_t max_pages_per_seq, int64_t num_pages, double scale,
                    const int64_t* bh_list, int64_t n_bh, int nthreads) {
    if (B < 0 || H < 0 || d <= 0 || page_size <= 0) return -1;
    int64_t n_out = bh_list ? n_bh : B * H;
    int64_t max_ctx = page_size * max_pages_per_seq;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
#endif
    {
        size_t cap = (size_t)(max_ctx > 0 ? max_ctx : 1);
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * cap);
        double* kd = (double*)malloc(sizeof(double) * cap * (size_t)d);
        double* vd = (double*)malloc(sizeof(double) * cap * (size_t)d);
        const double** kr = (const double**)malloc(sizeof(double*) * cap);
        const double** vr = (const double**)malloc(sizeof(double*) * cap);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < n_out; ++r) {
            int64_t bh = bh_list ? bh_list[r] : r;
            if (bh < 0 || bh >= B * H) {
                bad = 1;
                continue;
            }
            int64_t b = bh / H, h = bh % H;
            int64_t ctx = ctx_lens[b];
            if (ctx < 0 || ctx > max_ctx) {
                bad = 1;
                continue;
            }
            /* gather: token t of sequence b, head h, into row t of kd / vd */
            int64_t n = 0;
            for (int64_t t = 0; t < ctx; ++t) {
                int64_t page = block_table[b * max_pages_per_seq + t / page_size];
                if (page < 0 || page >= num_pages) {
                    bad = 1;
                    break;
                }
                int64_t src = ((page * H + h) * page_size + t % page_size) * d;
                for (int64_t c = 0; c < d; ++c) {
                    kd[t * d + c] = or_elem(k_pages, src + c, dtype);
                    vd[t * d + c] = or_elem(v_pages, src + c, dtype);
                }
                kr[n] = kd + t * d;
                vr[n] = vd + t * d;
                ++n;
            }
            if (n != ctx) continue;
            for (int64_t c = 0; c < d; ++c) qrow[c] = or_elem(q, bh * d + c, dtype);
            double err;
            attend_row(qrow, kr, vr, n, d, scale, s, o + r * d, lse + r, &err);
        }
        free(qrow);
        free(s);
        free(kd);
        free(vd);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * Prefill against a paged cache: sequence b holds ctx_lens[b] keys in pages (as in
 * or_decode_paged) and its Sq queries are its last Sq tokens, so query i of sequence b
 * is row i of an attention with Sq queries and Sk = ctx_lens[b] keys under the given
 * mask (bottom-right alignment, as or_visible). q and o are [B,H,Sq,d], lse [B,H,Sq].
 * Returns 0, or -1 if a needed table entry is out of range.
 */
int or_attention_paged(const void* q, const void* k_pages, const void* v_pages, int dtype,
                       const int32_t* block_table, const int32_t* ctx_lens, double* o,
                       double* lse, int64_t B, int64_t H, int64_t Sq, int64_t d,
                       int64_t page_size, int64_t max_pages_per_seq, int64_t num_pages,
                       double scale, int mask_mode, int64_t window, int64_t n_global,
                       int nthreads) {
    if (B < 0 || H < 0 || Sq < 0 || d <= 0 || page_size <= 0) return -1;
    int64_t max_ctx = page_size * max_pages_per_seq;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
#endif
    {
        size_t cap = (size_t)(max_ctx > 0 ? max_ctx : 1);
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * cap);
        double* kd = (double*)malloc(sizeof(double) * cap * (size_t)d);
        double* vd = (double*)malloc(sizeof(double) * cap * (size_t)d);
        const double** kr = (const double**)malloc(sizeof(double*) * cap);
        const double** vr = (const double**)malloc(sizeof(double*) * cap);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bh = 0; bh < B * H; ++bh) {
            int64_t b = bh / H, h = bh % H;
            int64_t ctx = ctx_lens[b];
            if (ctx < 0 || ctx > max_ctx) {
                bad = 1;
                continue;
            }
            /* gather this sequence's keys and values for head h, in position order */
            int ok = 1;
            for (int64_t t = 0; t < ctx && ok; ++t) {
                int64_t page = block_table[b * max_pages_per_seq + t / page_size];
                if (page < 0 || page >= num_pages) {
                    ok = 0;
                    break;
                }
                int64_t src = ((page * H + h) * page_size + t % page_size) * d;
                for (int64_t c = 0; c < d; ++c) {
                    kd[t * d + c] = or_elem(k_pages, src + c, dtype);
                    vd[t * d + c] = or_elem(v_pages, src + c, dtype);
                }
            }
            if (!ok) {
                bad = 1;
                continue;
            }
            for (int64_t i = 0; i < Sq; ++i) {
                int64_t row = bh * Sq + i;
                for (int64_t c = 0; c < d; ++c) qrow[c] = or_elem(q, row * d + c, dtype);
                int64_t n = 0;
                for (int64_t j = 0; j < ctx; ++j)
                    if (or_visible(i, j, Sq, ctx, mask_mode, window, n_global)) {
                        kr[n] = kd + j * d;
                        vr[n] = vd + j * d;
                        ++n;
                    }
                double err;
                attend_row(qrow, kr, vr, n, d, scale, s, o + row * d, lse + row, &err);
            }
        }
        free(qrow);
        free(s);
        free(kd);
        free(vd);
        free(kr);
        free(vr);
    }
    return bad ? -1 : 0;
}

/*
 * Merge softmax partials computed over disjoint key subsets. Split s holds
 *   m_s = max of its scores, l_s = sum exp(s_j - m_s), acc_s = sum exp(s_j - m_s) v_j.
 * The merged result is the same recurrence as the per-block update of
 * [ops-transformer] 二.1 / [Ascend-FA] 3.1, applied across splits:
 *   M = max m_s;  L = sum l_s exp(m_s - M);  O = sum exp(m_s - M) acc_s / L;
 *   LSE = M + ln L.  Splits with l_s = 0 contribute nothing; if all are empty,
 *   O = 0 and LSE = -inf.
 */
void or_combine_partials(const double* m, const double* l, const double* acc,
                         int64_t nsplit, int64_t d, double* o, double* lse) {
    double M = -INFINITY;
    for (int64_t s = 0; s < nsplit; ++s)
        if (l[s] > 0.0 && m[s] > M) M = m[s];
    for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double L = 0.0;
    for (int64_t s = 0; s < nsplit; ++s)
        if (l[s] > 0.0) L += l[s] * exp(m[s] - M);
    for (int64_t s = 0; s < nsplit; ++s) {
        if (!(l[s] > 0.0)) continue;
        double w = exp(m[s] - M) / L;
        for (int64_t c = 0; c < d; ++c) o[c] += w * acc[s * d + c];
    }
    *lse = M + log(L);
}

/*
 * The token range [t0, t1) that decode split `split` covers when a sequence
 * of ctx_len tokens is cut into runs of pages_per_split whole pages.
 */
void or_decode_split_tokens(int64_t ctx_len, int64_t page_size,
                            int64_t pages_per_split, int64_t split, int64_t* t0,
                            int64_t* t1) {
    int64_t span = page_size * pages_per_split;
    int64_t a = split * span, b = a + span;
    *t0 = a < ctx_len ? a : ctx_len;
    *t1 = b < ctx_len ? b : ctx_len;
}

/* ------------------------------------------------------------------ */
/* block-sparse layouts                                                */
/* ------------------------------------------------------------------ */

/*
 * Block-sparse attention: [boost] scenario 3 names block-sparse FlashAttention as
 * a variant beside prefix-LM and defines it no further. It is read here as the
 * usual block layout: query i of head h sees key j iff
 *     layout[(h * nqb + i / blk) * nkb + j / blk] != 0,
 * with nqb = ceil(Sq / blk) and nkb = ceil(Sk / blk); one layout serves every
 * batch entry. No alignment between query and key positions is involved.
 */
static int layout_visible(const uint8_t* layout, int64_t h, int64_t i, int64_t j,
                          int64_t nqb, int64_t nkb, int64_t blk) {
    return layout[(h * nqb + i / blk) * nkb + j / blk] != 0;
}

/*
 * Attention under a block layout, by the definition (attend_row), for every row
 * (rows == NULL; o [B,H,Sq,d], lse [B,H,Sq]) or for rows[r] = (b*H + h)*Sq + i
 * (o [nrows,d], lse [nrows]). Returns 0, or -1 on a bad argument.
 */
int or_attention_layout(const void* q, const void* k, const void* v, int dtype,
                        double* o, double* lse, int64_t B, int64_t H, int64_t Sq,
                        int64_t Sk, int64_t d, double scale, const uint8_t* layout,
                        int64_t blk, const int64_t* rows, int64_t nrows, int nthreads) {
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || d <= 0 || blk <= 0) return -1;
    if (!layout && B * H * Sq > 0) return -1;
    const int64_t nqb = (Sq + blk - 1) / blk, nkb = (Sk + blk - 1) / blk;
    const int64_t n_out = rows ? nrows : B * H * Sq;
    for (int64_t r = 0; r < n_out; ++r)
        if (rows && (rows[r] < 0 || rows[r] >= B * H * Sq)) return -1;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        const size_t cap = (size_t)(Sk > 0 ? Sk : 1);
        double* qrow = (double*)malloc(sizeof(double) * (size_t)d);
        double* kd = (double*)malloc(sizeof(double) * cap * (size_t)d);
        double* vd = (double*)malloc(sizeof(double) * cap * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * cap);
        const double** kr = (const double**)malloc(sizeof(double*) * cap);
        const double** vr = (const double**)malloc(sizeof(double*) * cap);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 16)
#endif
        for (int64_t r = 0; r < n_out; ++r) {
            const int64_t row = rows ? rows[r] : r;
            const int64_t bh = row / Sq, i = row % Sq, h = bh % H;
            for (int64_t c = 0; c < d; ++c) qrow[c] = or_elem(q, row * d + c, dtype);
            int64_t n = 0;
            for (int64_t j = 0; j < Sk; ++j) {
                if (!layout_visible(layout, h, i, j, nqb, nkb, blk)) continue;
                for (int64_t c = 0; c < d; ++c) {
                    kd[n * d + c] = or_elem(k, (bh * Sk + j) * d + c, dtype);
                    vd[n * d + c] = or_elem(v, (bh * Sk + j) * d + c, dtype);
                }
                kr[n] = kd + n * d;
                vr[n] = vd + n * d;
                ++n;
            }
            double err;
            attend_row(qrow, kr, vr, n, d, scale, s, o + r * d, lse + r, &err);
        }
        free(qrow);
        free(kd);
        free(vd);
        free(s);
        free(kr);
        free(vr);
    }
    return 0;
}

/* Visible (query, key) pairs of all H heads under a layout, by brute force. */
int64_t or_count_visible_layout(int64_t H, int64_t Sq, int64_t Sk, const uint8_t* layout,
                                int64_t blk) {
    const int64_t nqb = (Sq + blk - 1) / blk, nkb = (Sk + blk - 1) / blk;
    int64_t n = 0;
    for (int64_t h = 0; h < H; ++h)
        for (int64_t i = 0; i < Sq; ++i)
            for (int64_t j = 0; j < Sk; ++j) n += layout_visible(layout, h, i, j, nqb, nkb, blk);
    return n;
}

/* Class of the BM x BN tile (mb, nb) of head h under a layout, by brute force over
 * its pairs (rows and keys past the ends count as not visible). */
int or_tile_class_layout(int64_t h, int64_t mb, int64_t nb, int64_t BM, int64_t BN,
                         int64_t Sq, int64_t Sk, const uint8_t* layout, int64_t blk) {
    const int64_t nqb = (Sq + blk - 1) / blk, nkb = (Sk + blk - 1) / blk;
    int64_t vis = 0;
    for (int64_t i = mb * BM; i < mb * BM + BM; ++i)
        for (int64_t j = nb * BN; j < nb * BN + BN; ++j)
            if (i < Sq && j < Sk) vis += layout_visible(layout, h, i, j, nqb, nkb, blk);
    if (vis == 0) return OR_TILE_EMPTY;
    if (vis == BM * BN) return OR_TILE_FULL;
    return OR_TILE_PARTIAL;
}

/* ------------------------------------------------------------------ */
/* backward                                                            */
/* ------------------------------------------------------------------ */

/*
 * Gradients of O = softmax(scale Q K^T + mask) V for an upstream gradient dO: the
 * backward pass that the pages' remark on re-reading the scores refers to (they print
 * no formula), written out by the chain rule per (batch, head) and row i:
 *   s_ij = scale Q_i.K_j and P_ij = exp(s_ij - LSE_i) over the visible j,
 *   dV_j += P_ij dO_i,   dP_ij = dO_i.V_j,   D_i = sum_j P_ij dP_ij,
 *   dS_ij = P_ij (dP_ij - D_i),   dQ_i = scale sum_j dS_ij K_j,   dK_j += scale dS_ij Q_i.
 * Inputs q, k, v, dout share one dtype; dq [B,H,Sq,d], dk and dv [B,H,Sk,d] are FP64.
 * A row that sees no key contributes nothing. Returns 0, or -1 on a bad argument.
 */
static int backward_impl(const void* q, const void* k, const void* v, const void* dout,
                         int dtype, double* dq, double* dk, double* dv, int64_t B, int64_t H,
                         int64_t Sq, int64_t Sk, int64_t d, double scale, int mask_mode,
                         int64_t window, int64_t n_global, const unsigned char* layout,
                         int64_t blk, int nthreads) {
    const int64_t lnq = layout ? (Sq + blk - 1) / blk : 0, lnk = layout ? (Sk + blk - 1) / blk : 0;
    memset(dq, 0, sizeof(double) * (size_t)(B * H * Sq * d));
    memset(dk, 0, sizeof(double) * (size_t)(B * H * Sk * d));
    memset(dv, 0, sizeof(double) * (size_t)(B * H * Sk * d));
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        const size_t kc = (size_t)(Sk > 0 ? Sk : 1);
        double* qd = (double*)malloc(sizeof(double) * (size_t)(Sq > 0 ? Sq : 1) * (size_t)d);
        double* gd = (double*)malloc(sizeof(double) * (size_t)(Sq > 0 ? Sq : 1) * (size_t)d);
        double* kd = (double*)malloc(sizeof(double) * kc * (size_t)d);
        double* vd = (double*)malloc(sizeof(double) * kc * (size_t)d);
        double* s = (double*)malloc(sizeof(double) * kc);
        double* dp = (double*)malloc(sizeof(double) * kc);
        int64_t* vis = (int64_t*)malloc(sizeof(int64_t) * kc);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t bh = 0; bh < B * H; ++bh) {
            or_decode((const char*)q + (size_t)(bh * Sq * d) * elem_size(dtype), qd, Sq * d, dtype);
            or_decode((const char*)dout + (size_t)(bh * Sq * d) * elem_size(dtype), gd, Sq * d,
                      dtype);
            or_decode((const char*)k + (size_t)(bh * Sk * d) * elem_size(dtype), kd, Sk * d, dtype);
            or_decode((const char*)v + (size_t)(bh * Sk * d) * elem_size(dtype), vd, Sk * d, dtype);
            double* dqb = dq + bh * Sq * d;
            double* dkb = dk + bh * Sk * d;
            double* dvb = dv + bh * Sk * d;
            for (int64_t i = 0; i < Sq; ++i) {
                const double* qi = qd + i * d;
                const double* gi = gd + i * d;
                int64_t n = 0;
                double m = -INFINITY;
                for (int64_t j = 0; j < Sk; ++j) {
                    const int seen =
                        layout ? layout[((bh % H) * lnq + i / blk) * lnk + j / blk] != 0
                               : or_visible(i, j, Sq, Sk, mask_mode, window, n_global);
                    if (!seen) continue;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += qi[c] * kd[j * d + c];
                    vis[n] = j;
                    s[n] = scale * dot;
                    if (s[n] > m) m = s[n];
                    ++n;
                }
                if (n == 0) continue;
                double z = 0.0;
                for (int64_t t = 0; t < n; ++t) z += exp(s[t] - m);
                const double lse = m + log(z);
                double D = 0.0;
                for (int64_t t = 0; t < n; ++t) {
                    const int64_t j = vis[t];
                    s[t] = exp(s[t] - lse); /* P_ij */
                    double g = 0.0;
                    for (int64_t c = 0; c < d; ++c) g += gi[c] * vd[j * d + c];
                    dp[t] = g;
                    D += s[t] * g;
                }
                for (int64_t t = 0; t < n; ++t) {
                    const int64_t j = vis[t];
                    const double p = s[t], ds = p * (dp[t] - D);
                    for (int64_t c = 0; c < d; ++c) {
                        dvb[j * d + c] += p * gi[c];
                        dqb[i * d + c] += scale * ds * kd[j * d + c];
                        dkb[j * d + c] += scale * ds * qi[c];
                    }
                }
            }
        }
        free(qd);
        free(gd);
        free(kd);
        free(vd);
        free(s);
        free(dp);
        free(vis);
    }
    return 0;
}

int or_attention_backward(const void* q, const void* k, const void* v, const void* dout,
                          int dtype, double* dq, double* dk, double* dv, int64_t B, int64_t H,
                          int64_t Sq, int64_t Sk, int64_t d, double scale, int mask_mode,
                          int64_t window, int64_t n_global, int nthreads) {
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || d <= 0) return -1;
    if (mask_mode < OR_MASK_NONE || mask_mode > OR_MASK_PREFIX_LM) return -1;
    if (mask_mode == OR_MASK_CAUSAL_WINDOW && (window < 1 || n_global < 0)) return -1;
    if (mask_mode == OR_MASK_BAND && window < 0) return -1;
    if (mask_mode == OR_MASK_PREFIX_LM && n_global < 0) return -1;
    return backward_impl(q, k, v, dout, dtype, dq, dk, dv, B, H, Sq, Sk, d, scale, mask_mode,
                         window, n_global, NULL, 1, nthreads);
}

/*
 * The same gradients under a block layout (as or_attention_layout): query i of head h sees
 * key j iff layout[h][i / blk][j / blk] != 0, layout uint8 [H][ceil(Sq/blk)][ceil(Sk/blk)].
 * Returns 0, or -1 on a bad argument.
 */
int or_attention_backward_layout(const void* q, const void* k, const void* v, const void* dout,
                                 int dtype, double* dq, double* dk, double* dv, int64_t B,
                                 int64_t H, int64_t Sq, int64_t Sk, int64_t d, double scale,
                                 const unsigned char* layout, int64_t blk, int nthreads) {
    if (B < 0 || H < 0 || Sq < 0 || Sk < 0 || d <= 0 || blk < 1 || !layout) return -1;
    return backward_impl(q, k, v, dout, dtype, dq, dk, dv, B, H, Sq, Sk, d, scale, OR_MASK_NONE,
                         0, 0, layout, blk, nthreads);
}
