/*
 * pagedkv_oracle.c -- plain, slow fp64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file.  Its users are the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark.  It shares no code, header, table or
 * constant with the CUDA library: it has its own element decoders, its own
 * enums and its own address arithmetic, all written from the three
 * FlashInfer API pages:
 *
 *   [prefill] flashinfer.prefill.cudnn_batch_prefill_with_kv_cache
 *   [decode]  flashinfer.decode.trtllm_batch_decode_with_kv_cache
 *   [append]  flashinfer.page.append_paged_kv_cache
 *
 * Every function is the definition written out: no tiling, no splitting, no
 * online softmax.  Floating-point work is in double; 16-bit inputs are
 * widened exactly.  Sums run over keys in logical order.
 *
 * Return values are bit masks of ORC_E_* (0 = clean); the same conditions
 * are documented for the CUDA library's device error word.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_NHD 0 /* page = [page_size][num_kv_heads][head_dim] */
#define ORC_HND 1 /* page = [num_kv_heads][page_size][head_dim] */

#define ORC_FP16 0
#define ORC_BF16 1
#define ORC_E4M3 2 /* 8-bit float cache elements (OCP FP8 E4M3) */

#define ORC_E_PAGE 1  /* physical page id outside [0, max_num_pages)       */
#define ORC_E_POS 2   /* position / page slot outside the request's pages  */
#define ORC_E_BATCH 4 /* batch index outside [0, B)                        */
#define ORC_E_QLEN 8  /* kv length shorter than the query length           */

/* ---- exact widening of 16-bit floats ------------------------------------ */

static double orc_from_bf16(uint16_t bits)
{
    /* bfloat16 is the upper half of an IEEE binary32 */
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_from_fp16(uint16_t bits)
{
    /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits */
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int mant = bits & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24); /* subnormal: mant * 2^-14 * 2^-10 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25); /* (1.m) * 2^(e-15) */
    return sign ? -v : v;
}

static double orc_from_e4m3(uint8_t bits)
{
    /* OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no
     * infinities, exponent 15 with mantissa 7 is NaN, the largest normal is
     * 1.75 * 2^8 = 448 */
    int sign = (bits >> 7) & 1;
    int expo = (bits >> 3) & 0xf;
    int mant = bits & 0x7;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -9); /* subnormal: mant/8 * 2^-6 */
    else if (expo == 15 && mant == 7)
        v = NAN;
    else
        v = ldexp((double)(8 + mant), expo - 10); /* (1.m) * 2^(e-7) */
    return sign ? -v : v;
}

/* element i of an array of 16-bit (fp16 / bf16) or 8-bit (e4m3) floats */
static double orc_elem(const void *p, int64_t i, int dtype)
{
    if (dtype == ORC_E4M3)
        return orc_from_e4m3(((const uint8_t *)p)[i]);
    const uint16_t *h = (const uint16_t *)p;
    return dtype == ORC_BF16 ? orc_from_bf16(h[i]) : orc_from_fp16(h[i]);
}

/* Element offset of (page, kv head, slot, d) inside one cache tensor
 * ([decode] kv_cache shapes; [append] paged_kv_cache shapes). */
static int64_t orc_kv_offset(int layout, int64_t page, int64_t page_stride,
                             int head, int slot, int d, int num_kv_heads,
                             int page_size, int head_dim)
{
    int64_t within;
    if (layout == ORC_HND)
        within = ((int64_t)head * page_size + slot) * head_dim + d;
    else
        within = ((int64_t)slot * num_kv_heads + head) * head_dim + d;
    return page * page_stride + within;
}

/* ---- [append] example helpers ------------------------------------------- */

/* kv length of request b from its page count and last-page fill:
 * (pages - 1) * page_size + last_page_len   ([append] worked example). */
int orc_seq_lens(const int32_t *kv_indptr, const int32_t *kv_last_page_len,
                 int B, int page_size, int32_t *seq_lens)
{
    for (int b = 0; b < B; ++b) {
        int pages = kv_indptr[b + 1] - kv_indptr[b];
        seq_lens[b] = pages > 0 ? (pages - 1) * page_size + kv_last_page_len[b] : 0;
    }
    return 0;
}

/* Request index and absolute position of each appended entry.  The page
 * table already counts the appended tokens ([append] note), so the n_b new
 * tokens of request b occupy the last n_b positions of its sequence.
 * Entries not covered by append_indptr are set to -1. */
int orc_batch_indices_positions(const int32_t *append_indptr,
                                const int32_t *seq_lens, int B, int64_t nnz,
                                int32_t *batch_indices, int32_t *positions)
{
    for (int64_t i = 0; i < nnz; ++i) {
        batch_indices[i] = -1;
        positions[i] = -1;
    }
    for (int b = 0; b < B; ++b) {
        int64_t start = append_indptr[b];
        int64_t n = (int64_t)append_indptr[b + 1] - start;
        for (int64_t k = 0; k < n; ++k) {
            int64_t i = start + k;
            if (i < 0 || i >= nnz)
                continue;
            batch_indices[i] = b;
            positions[i] = (int32_t)(seq_lens[b] - n + k);
        }
    }
    return 0;
}

/* ---- [append] scatter ---------------------------------------------------- */

/* Copy the bits of append_key[i] / append_value[i] into the page slot that
 * (batch_indices[i], positions[i]) addresses through kv_indptr/kv_indices.
 * Entries whose addressing is out of range are skipped and flagged. */
int orc_append(const void *append_key, const void *append_value,
               int64_t nnz, const int32_t *batch_indices,
               const int32_t *positions, void *k_cache, void *v_cache,
               int64_t page_stride, int64_t max_num_pages,
               const int32_t *kv_indices, const int32_t *kv_indptr,
               const int32_t *kv_last_page_len, int B, int num_kv_heads,
               int head_dim, int page_size, int layout, int elem_bytes)
{
    int err = 0;
    for (int64_t i = 0; i < nnz; ++i) {
        int b = batch_indices[i];
        int p = positions[i];
        if (b < 0 || b >= B) {
            err |= ORC_E_BATCH;
            continue;
        }
        int pages = kv_indptr[b + 1] - kv_indptr[b];
        int len = pages > 0 ? (pages - 1) * page_size + kv_last_page_len[b] : 0;
        if (p < 0 || p >= len) {
            err |= ORC_E_POS;
            continue;
        }
        int64_t page = kv_indices[kv_indptr[b] + p / page_size];
        if (page < 0 || page >= max_num_pages) {
            err |= ORC_E_PAGE;
            continue;
        }
        int slot = p % page_size;
        for (int h = 0; h < num_kv_heads; ++h)
            for (int d = 0; d < head_dim; ++d) {
                int64_t dst = orc_kv_offset(layout, page, page_stride, h, slot, d,
                                            num_kv_heads, page_size, head_dim);
                int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim + d;
                memcpy((char *)k_cache + dst * elem_bytes,
                       (const char *)append_key + src * elem_bytes, elem_bytes);
                memcpy((char *)v_cache + dst * elem_bytes,
                       (const char *)append_value + src * elem_bytes, elem_bytes);
            }
    }
    return err;
}

/* ---- one attention row --------------------------------------------------- */

/* o[0:d_vo] = out_scale * sum_{j in [lo, hi]} e^{s_j - M} v_j / den and
 * lse = M + log den, with s_j = scale * <q, k_j>, den = sum e^{s_j - M}
 * (+ e^{sink - M} when has_sink), M the largest term.  Every stored element
 * is dequantised by its tensor's factor first (q_mul * q, k_mul * k,
 * v_mul * v; 1 for 16-bit tensors).  The query row is elements q_off ..
 * q_off + d_qk - 1 of q.  Keys are read through the block table row `bt` of
 * one request.  An empty key set without a sink gives o = 0 and lse = -inf. */
static int orc_attend_row(const void *q, int64_t q_off, int dtype, double q_mul,
                          double k_mul, double v_mul, const void *k_cache,
                          const void *v_cache, int kv_dtype, int64_t k_page_stride,
                          int64_t v_page_stride, int64_t max_num_pages,
                          const int32_t *bt, int kvh, int num_kv_heads,
                          int page_size, int d_qk, int d_vo, int layout,
                          int64_t lo, int64_t hi, double scale, double out_scale,
                          int has_sink, double sink, double *o, double *lse,
                          double *s /* scratch, >= hi - lo + 1 */)
{
    int err = 0;
    int64_t n = hi >= lo ? hi - lo + 1 : 0;
    double m = has_sink ? sink : -INFINITY;
    for (int64_t jj = 0; jj < n; ++jj) {
        int64_t j = lo + jj;
        int64_t page = bt[j / page_size];
        if (page < 0 || page >= max_num_pages) {
            err |= ORC_E_PAGE;
            s[jj] = -INFINITY;
            continue;
        }
        int slot = (int)(j % page_size);
        double dot = 0.0;
        for (int d = 0; d < d_qk; ++d) {
            int64_t off = orc_kv_offset(layout, page, k_page_stride, kvh, slot, d,
                                        num_kv_heads, page_size, d_qk);
            dot += (q_mul * orc_elem(q, q_off + d, dtype)) * (k_mul * orc_elem(k_cache, off, kv_dtype));
        }
        s[jj] = scale * dot;
        if (s[jj] > m)
            m = s[jj];
    }
    for (int d = 0; d < d_vo; ++d)
        o[d] = 0.0;
    if (m == -INFINITY) { /* no key and no sink */
        *lse = -INFINITY;
        return err;
    }
    double den = has_sink ? exp(sink - m) : 0.0;
    for (int64_t jj = 0; jj < n; ++jj) {
        if (s[jj] == -INFINITY)
            continue;
        int64_t j = lo + jj;
        int64_t page = bt[j / page_size];
        int slot = (int)(j % page_size);
        double w = exp(s[jj] - m);
        den += w;
        for (int d = 0; d < d_vo; ++d) {
            int64_t off = orc_kv_offset(layout, page, v_page_stride, kvh, slot, d,
                                        num_kv_heads, page_size, d_vo);
            o[d] += w * (v_mul * orc_elem(v_cache, off, kv_dtype));
        }
    }
    for (int d = 0; d < d_vo; ++d)
        o[d] = out_scale * o[d] / den;
    *lse = m + log(den);
    return err;
}

/* ---- [decode] batch decode ----------------------------------------------- */

/* For request b, query token t < Q and qo head h (query row b*Q + t):
 *   kv head    = h / (num_qo_heads / num_kv_heads)
 *   position   p = seq_lens[b] - Q + t   (the Q tokens are the last ones)
 * With cum_seq_lens_q (the decode page's variable-length queries) request b
 * has Q = cum_seq_lens_q[b+1] - cum_seq_lens_q[b] tokens at rows
 * cum_seq_lens_q[b] + t, and q_len_per_req is unused.
 *   keys       max(0, p - window_left) <= j <= p  (window_left = -1: j >= 0)
 *   logits     s_j = bmm1_scale * <q, k_j>
 *   out        bmm2_scale * softmax-weighted sum of v_j, where the softmax
 *              denominator also holds e^{sinks[h]} when sinks != NULL
 *   lse        log of that denominator.
 * out: [rows, num_qo_heads, head_dim], lse: [rows, num_qo_heads] (may be
 * NULL), rows = B*Q or cum_seq_lens_q[B].
 * scratch: caller buffer of at least max_seq_len doubles per thread slot
 * (threads * max_seq_len when OpenMP is used; pass n_scratch_threads). */
int orc_decode(const uint16_t *query, const void *k_cache,
               const void *v_cache, int64_t page_stride,
               int64_t max_num_pages, const int32_t *block_tables,
               int block_table_stride, const uint32_t *seq_lens, int B,
               int max_seq_len, double bmm1_scale, double bmm2_scale,
               int window_left, const float *sinks, int q_len_per_req,
               const int32_t *cum_seq_lens_q, int num_qo_heads,
               int num_kv_heads, int head_dim, int page_size, int layout,
               int dtype, int kv_dtype, double *out, double *lse, double *scratch,
               int n_scratch_threads, int num_threads)
{
    int err = 0;
    int group = num_qo_heads / num_kv_heads;
    int64_t tokens = cum_seq_lens_q ? cum_seq_lens_q[B] : (int64_t)B * q_len_per_req;
    int64_t rows = tokens * num_qo_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err) num_threads(num_threads)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        if (tid >= n_scratch_threads)
            tid = 0; /* never happens when the caller sizes scratch */
        double *s = scratch + (int64_t)tid * (max_seq_len + 1);
        int h = (int)(r % num_qo_heads);
        int64_t row = r / num_qo_heads; /* query row */
        int b, t, Q;
        if (cum_seq_lens_q) {
            /* the request whose rows [cum[b], cum[b+1]) hold this row */
            int lo_b = 0, hi_b = B - 1;
            while (lo_b < hi_b) {
                int mid = (lo_b + hi_b + 1) / 2;
                if (cum_seq_lens_q[mid] <= row)
                    lo_b = mid;
                else
                    hi_b = mid - 1;
            }
            b = lo_b;
            Q = cum_seq_lens_q[b + 1] - cum_seq_lens_q[b];
            t = (int)(row - cum_seq_lens_q[b]);
        } else {
            Q = q_len_per_req;
            b = (int)(row / Q);
            t = (int)(row % Q);
        }
        int64_t L = seq_lens[b];
        int64_t p = L - Q + t;
        int64_t lo = 0, hi = p;
        if (L < Q)
            err |= ORC_E_QLEN;
        if (window_left >= 0 && p - window_left > 0)
            lo = p - window_left;
        double lse_r;
        err |= orc_attend_row(query, r * head_dim, dtype, 1.0, 1.0, 1.0, k_cache, v_cache, kv_dtype,
                              page_stride, page_stride, max_num_pages,
                              block_tables + (int64_t)b * block_table_stride,
                              h / group, num_kv_heads, page_size, head_dim,
                              head_dim, layout, lo, hi, bmm1_scale, bmm2_scale,
                              sinks != NULL, sinks ? (double)sinks[h] : 0.0,
                              out + r * head_dim, &lse_r, s);
        if (lse)
            lse[r] = lse_r;
    }
    return err;
}

/* ---- [prefill] causal ragged batch prefill -------------------------------- */

/* For request b with q_b = actual_seq_lens_q[b] query tokens and
 * kv_b = actual_seq_lens_kv[b] keys, query i (packed row cu_q[b] + i, cu_q
 * the exclusive prefix sum of q lengths) sits at absolute position
 * kv_b - q_b + i; with causal it attends keys j <= that position, otherwise
 * every j < kv_b.  out = softmax(scale * q k^T) v over those keys and
 * lse = log sum_j e^{scale * <q, k_j>} (natural log).  out: [total_q,
 * num_qo_heads, d_vo], lse: [total_q, num_qo_heads].
 * q is stored as q_dtype, the caches as kv_dtype (16-bit, or E4M3 with one
 * byte per element); q, k and v above are the stored values times the
 * page's q_scale, k_scale and v_scale (1 for 16-bit tensors). */
int orc_prefill(const void *q, const void *k_cache,
                const void *v_cache, int64_t k_page_stride,
                int64_t v_page_stride, int64_t max_num_pages, double scale,
                const int32_t *seq_lens_q, const int32_t *seq_lens_kv,
                const int32_t *block_tables, int block_table_stride, int B,
                int causal, int num_qo_heads, int num_kv_heads, int d_qk,
                int d_vo, int page_size, int layout, int q_dtype, int kv_dtype,
                double q_scale, double k_scale, double v_scale, double *out,
                double *lse, double *scratch, int scratch_len,
                int n_scratch_threads, int num_threads)
{
    int err = 0;
    int group = num_qo_heads / num_kv_heads;
    int64_t total_q = 0;
    for (int b = 0; b < B; ++b)
        total_q += seq_lens_q[b];
    int64_t rows = total_q * num_qo_heads;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 4) reduction(| : err) num_threads(num_threads)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        if (tid >= n_scratch_threads)
            tid = 0;
        double *s = scratch + (int64_t)tid * scratch_len;
        int h = (int)(r % num_qo_heads);
        int64_t tok = r / num_qo_heads;
        /* find the request that owns packed token `tok` */
        int b = 0;
        int64_t start = 0;
        while (b < B && tok >= start + seq_lens_q[b]) {
            start += seq_lens_q[b];
            ++b;
        }
        int64_t i = tok - start;
        int64_t qb = seq_lens_q[b], kvb = seq_lens_kv[b];
        if (kvb < qb)
            err |= ORC_E_QLEN;
        int64_t pos = kvb - qb + i;
        int64_t hi = causal ? (pos < kvb - 1 ? pos : kvb - 1) : kvb - 1;
        double lse_r;
        err |= orc_attend_row(q, r * d_qk, q_dtype, q_scale, k_scale, v_scale, k_cache, v_cache, kv_dtype,
                              k_page_stride, v_page_stride, max_num_pages,
                              block_tables + (int64_t)b * block_table_stride,
                              h / group, num_kv_heads, page_size, d_qk, d_vo,
                              layout, 0, hi, scale, 1.0, 0, 0.0,
                              out + r * d_vo, &lse_r, s);
        lse[r] = lse_r;
    }
    return err;
}

/* ---- merge of partial results over disjoint key sets ----------------------- */

/* lse = log sum_i e^{lse_i}; o = sum_i e^{lse_i - lse} o_i.  Used to check
 * that softmax over a partition of the keys recombines to the whole. */
int orc_merge(const double *o_parts, const double *lse_parts, int n_parts,
              int dim, double *o, double *lse)
{
    double m = -INFINITY;
    for (int i = 0; i < n_parts; ++i)
        if (lse_parts[i] > m)
            m = lse_parts[i];
    for (int d = 0; d < dim; ++d)
        o[d] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return 0;
    }
    double den = 0.0;
    for (int i = 0; i < n_parts; ++i)
        den += exp(lse_parts[i] - m);
    double total = m + log(den);
    for (int i = 0; i < n_parts; ++i) {
        double w = exp(lse_parts[i] - total);
        for (int d = 0; d < dim; ++d)
            o[d] += w * o_parts[(int64_t)i * dim + d];
    }
    *lse = total;
    return 0;
}

/* Widen n 16-bit values (exposes the decoders above to the tests). */
int orc_widen16(const void *src, int64_t n, int dtype, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = orc_elem(src, i, dtype);
    return 0;
}

int orc_has_openmp(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 0;
#endif
}
