/*
 * pagedkv.h -- C ABI of libpagedkv.so: attention over a paged KV cache on
 * NVIDIA GB300 (sm_103a).
 *
 * The operations follow three FlashInfer API pages:
 *   [append]  flashinfer.page.append_paged_kv_cache (signature, parameters,
 *             worked example, note that the space is reserved beforehand);
 *   [decode]  flashinfer.decode.trtllm_batch_decode_with_kv_cache
 *             (signature and parameter list);
 *   [prefill] flashinfer.prefill.cudnn_batch_prefill_with_kv_cache
 *             (signature, parameter list, returns, note on head sizes).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is caller-owned.  Tensor arguments are DEVICE
 *    pointers on the current CUDA device; scalars are passed by value.  The
 *    library allocates and frees no memory and keeps no per-call state; its
 *    only globals are a launch counter for diagnostics, the limit of its
 *    bounded waits (pkv_set_wait_limit_ns) and the fixed scratch array of
 *    paged_decode_noalloc.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All device work is enqueued on it and the call returns without
 *    synchronising.  Argument errors are detected on the host and returned
 *    before anything is launched.
 *  - Return value: a pkv_status.  PKV_ERR_CUDA means a launch failed; the
 *    CUDA error is left for cudaGetLastError-style inspection by the caller.
 *  - `err_word` (optional, may be NULL) is one device int32.  Kernels OR
 *    PKV_DEV_ERR_* bits into it when an index read from device memory is out
 *    of range; the offending read or write is skipped and nothing traps.  The
 *    caller clears it.
 *  - 16-bit elements: dtype PKV_F16 (IEEE half) or PKV_BF16.  Attention
 *    accumulates in fp32 and rounds the output to nearest-even in the input
 *    dtype; LSE is fp32, natural log.  An 8-bit (OCP FP8 E4M3) K/V cache:
 *    PKV_E4M3 for paged_append, PKV_F16_E4M3 / PKV_BF16_E4M3 for decode (the
 *    query and output stay 16-bit; the caller folds the K and V scales into
 *    bmm1_scale / bmm2_scale, as the decode page's fused scales do), and
 *    paged_prefill_fp8 for the prefill (E4M3 query and/or caches with the
 *    prefill page's q_scale / k_scale / v_scale).
 *  - Layouts (both pages list the same two):
 *      PKV_HND: a page is [num_kv_heads][page_size][head_dim];
 *      PKV_NHD: a page is [page_size][num_kv_heads][head_dim].
 *    There is no default: the decode page defaults to HND, the append page
 *    to NHD, so the caller always says which.
 *  - A cache is passed as two base pointers (K pages, V pages) and a page
 *    stride in elements.  The 5-D form [pages, 2, ...] is k = base,
 *    v = base + num_kv_heads * page_size * head_dim, stride = 2 * that; the
 *    tuple form is two tensors with stride num_kv_heads*page_size*head_dim.
 *    Element (page, head, slot, d) lives at
 *      HND: page * stride + (head * page_size + slot) * head_dim + d
 *      NHD: page * stride + (slot * num_kv_heads + head) * head_dim + d.
 *  - Alignment: every 16-bit tensor base and page stride must be a multiple
 *    of 16 bytes (8 elements), else PKV_ERR_INVALID_ARG.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_NULL = 1,        /* a required pointer is NULL                   */
    PKV_ERR_INVALID_ARG = 2, /* bad enum, size, ratio or alignment           */
    PKV_ERR_UNSUPPORTED = 3, /* valid but not compiled (head dim, page size) */
    PKV_ERR_WORKSPACE = 4,   /* workspace smaller than the size query says   */
    PKV_ERR_CUDA = 5         /* a kernel launch failed                       */
} pkv_status;

enum { PKV_NHD = 0, PKV_HND = 1 };
enum {
    PKV_F16 = 0,
    PKV_BF16 = 1,
    PKV_E4M3 = 2,      /* 8-bit float (OCP FP8 E4M3) cache elements: paged_append   */
    PKV_F16_E4M3 = 3,  /* decode: fp16 query/out over an E4M3 K/V cache            */
    PKV_BF16_E4M3 = 4  /* decode: bf16 query/out over an E4M3 K/V cache            */
};

/* bits of the device error word */
#define PKV_DEV_ERR_PAGE 1    /* physical page id outside [0, max_num_pages)        */
#define PKV_DEV_ERR_POS 2     /* append position outside the request's reserved pages */
#define PKV_DEV_ERR_BATCH 4   /* append batch index outside [0, batch_size)         */
#define PKV_DEV_ERR_QLEN 8    /* kv length shorter than the query length            */
#define PKV_DEV_ERR_TIMEOUT 16 /* a bounded pipeline wait gave up; output invalid   */
#define PKV_DEV_ERR_LEN 32    /* a length exceeds the stated maximum; it is clamped  */
#define PKV_DEV_ERR_BOUNDS 64 /* debug build only: a derived offset left its buffer  */

/* Human-readable name of a pkv_status value (static string). */
const char *pkv_status_string(int status);

/* Number of kernels this library has launched in this process. */
unsigned long long pkv_kernel_launches(void);

/*
 * pkv_debug_bounds -- 1 for the debug build of the library (compiled with
 * -DPKV_DEBUG_BOUNDS=1: libpagedkv_debug.so), 0 for the release build.  Both
 * check every index they read from device memory (page ids, batch indices,
 * positions, lengths; the PKV_DEV_ERR_* bits above).  The debug build also
 * range-checks every offset the kernels derive from those indices -- cache
 * rows, query and output rows, workspace partials, block-table entries,
 * tensor-map coordinates and shared-memory page lists -- before the access;
 * a violation sets PKV_DEV_ERR_BOUNDS and the access is skipped.  The
 * results of both builds are otherwise identical.  A diagnostic aid of this
 * library (the pages have none), in place of a memory checker.
 */
int pkv_debug_bounds(void);

/*
 * pkv_set_wait_limit_ns -- time limit, in nanoseconds, of every bounded
 * pipeline wait (an mbarrier wait for copied data, for the tensor core or
 * for another warp of the CTA) in the kernels of paged_append and
 * paged_prefill launched after the call; 0 restores the default of one
 * second.  Returns the previous limit.  Process-wide (every thread and
 * device).  A wait that runs out sets PKV_DEV_ERR_TIMEOUT in the call's
 * error word; the CTA then stops its work, waits for the copies and MMAs
 * it had already issued, frees its tensor memory and exits, so the device
 * stays usable and the next call runs normally, but the outputs of that
 * call are incomplete.  It exists to detect a stalled pipeline (and to test
 * that detection with a limit no wait can meet); the pages have no
 * counterpart.
 */
unsigned long long pkv_set_wait_limit_ns(unsigned long long ns);

/*
 * paged_seq_lens -- [append] worked example, `get_seq_lens` and the comments
 * "45 = (3 - 1) * 16 + 13" ...: the kv length of each request from its page
 * count and the fill of its last page,
 *   seq_lens[b] = (kv_indptr[b+1] - kv_indptr[b] - 1) * page_size
 *                 + kv_last_page_len[b]          (0 for a request with no page).
 *   kv_indptr [batch_size+1], kv_last_page_len [batch_size], seq_lens
 *   [batch_size] (output); all int32, device.
 */
int paged_seq_lens(const int32_t *kv_indptr, const int32_t *kv_last_page_len,
                   int32_t batch_size, int32_t page_size, int32_t *seq_lens,
                   void *stream);

/*
 * paged_batch_indices_positions -- [append] worked example,
 * `get_batch_indices_positions` and its printed output: for appended entry
 * i of request b (append_indptr[b] <= i < append_indptr[b+1]),
 *   batch_indices[i] = b,
 *   positions[i] = seq_lens[b] - (append_indptr[b+1] - append_indptr[b])
 *                  + (i - append_indptr[b]),
 * i.e. the new tokens are the last ones of each sequence because seq_lens
 * already counts them ([append] note).  Entries i >= append_indptr[batch_size]
 * get -1 in both outputs.  append_indptr must be non-decreasing.
 *   append_indptr [batch_size+1], seq_lens [batch_size]; outputs [nnz];
 *   int32, device.
 */
int paged_batch_indices_positions(const int32_t *append_indptr,
                                  const int32_t *seq_lens, int32_t batch_size,
                                  int64_t nnz, int32_t *batch_indices,
                                  int32_t *positions, void *stream);

/*
 * paged_append -- [append] signature and parameters: scatter nnz new tokens
 * into their reserved page slots.  For entry i with b = batch_indices[i],
 * p = positions[i]:
 *   page = kv_indices[kv_indptr[b] + p / page_size], slot = p % page_size,
 *   k_cache[page, head, slot, :] = append_key[i, head, :]  (HND indexing; NHD
 *   analogous), and the same for append_value into v_cache.
 * Bits are copied unchanged (dtype only fixes the element size; both 16-bit
 * types are accepted).  Nothing else in the pool is written.
 *   append_key/value: [nnz, num_kv_heads, head_dim], contiguous.
 *   batch_indices, positions: [nnz] int32 (from the helper above or the caller).
 *   kv_indices [kv_indptr[batch_size]], kv_indptr [batch_size+1],
 *   kv_last_page_len [batch_size]: int32.
 * Device errors: b outside [0, batch_size) -> PKV_DEV_ERR_BATCH; p outside
 * [0, seq_len(b)) -> PKV_DEV_ERR_POS; page outside [0, max_num_pages) ->
 * PKV_DEV_ERR_PAGE; the entry is skipped.  A copy that does not complete
 * within the wait limit (1 s; pkv_set_wait_limit_ns) -> PKV_DEV_ERR_TIMEOUT
 * and the CTA stops (its remaining entries are not written).  Duplicate
 * (b, p) pairs race.
 * dtype: PKV_F16 / PKV_BF16 (2-byte elements) or PKV_E4M3 (1-byte).
 * Host errors: a head row (head_dim elements) not a multiple of 16 bytes or
 * page_size <= 0 -> PKV_ERR_INVALID_ARG; a head row above 8 KB ->
 * PKV_ERR_UNSUPPORTED.
 */
int paged_append(const void *append_key, const void *append_value, int64_t nnz,
                 const int32_t *batch_indices, const int32_t *positions,
                 void *k_cache, void *v_cache, int64_t page_stride,
                 int64_t max_num_pages, const int32_t *kv_indices,
                 const int32_t *kv_indptr, const int32_t *kv_last_page_len,
                 int32_t batch_size, int32_t num_kv_heads, int32_t head_dim,
                 int32_t page_size, int32_t layout, int32_t dtype,
                 int32_t *err_word, void *stream);

/*
 * paged_decode_workspace_size -- bytes of device workspace paged_decode needs
 * for these sizes (split-KV partial outputs and their LSEs).  The decode
 * page asks for a caller-provided workspace; this query sizes it exactly.
 * Returns 0 for invalid sizes.
 */
size_t paged_decode_workspace_size(int32_t batch_size, int32_t q_len_per_req,
                                   int32_t num_qo_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_seq_len,
                                   int32_t page_size, int32_t window_left);

/*
 * paged_decode -- [decode] signature and parameters (query, kv_cache,
 * workspace_buffer, block_tables, seq_lens, max_seq_len, bmm1_scale,
 * bmm2_scale, window_left, sinks, kv_layout, q_len_per_req).  For request b
 * with L = seq_lens[b] keys, query token t < Q = q_len_per_req (row b*Q + t
 * of query/out) and qo head h:
 *   kv head   = h / (num_qo_heads / num_kv_heads)      (consecutive groups)
 *   position  p = L - Q + t        (the Q tokens are the last Q of the
 *             sequence, causal among themselves)
 *   keys      j with max(0, p - window_left) <= j <= p; window_left = -1
 *             means all j <= p ("left, inclusive" window)
 *   logits    s_j = bmm1_scale * <q, k_j>   (natural-exp softmax)
 *   out       bmm2_scale * sum_j e^{s_j} v_j / (sum_j e^{s_j} + e^{sinks[h]})
 *             (the sink term only when sinks != NULL; it has no value row)
 *   lse       log(sum_j e^{s_j} + e^{sinks[h]})      (optional output)
 * Key j of request b lives in page block_tables[b * block_table_stride +
 * j / page_size], slot j % page_size; table entries at or beyond
 * ceil(L / page_size) are never read.  An empty key set gives out = 0 and
 * lse = -inf (lse = sink with a sink).
 *   query/out: [batch_size*Q, num_qo_heads, head_dim] contiguous, dtype.
 *   seq_lens: [batch_size] uint32 (decode page: "uint32 1D tensor"), each
 *   <= max_seq_len.  sinks: [num_qo_heads] fp32 or NULL.  lse:
 *   [batch_size*Q, num_qo_heads] fp32 or NULL.
 *   workspace: >= paged_decode_workspace_size(...) bytes, 256-byte aligned.
 *   block_table_stride >= ceil(max_seq_len / page_size), else
 *   PKV_ERR_INVALID_ARG.  A seq_lens entry above max_seq_len sets
 *   PKV_DEV_ERR_LEN and is treated as max_seq_len.
 * Supported: head_dim 128; page_size a power of two in [8, 256];
 * num_qo_heads % num_kv_heads == 0 with (num_qo_heads/num_kv_heads) * Q <= 64.
 * Device errors: bad page id -> PKV_DEV_ERR_PAGE (key treated as absent);
 * L < Q -> PKV_DEV_ERR_QLEN (rows with p < 0 see no key).
 */
int paged_decode(const void *query, const void *k_cache, const void *v_cache,
                 int64_t page_stride, int64_t max_num_pages, void *workspace,
                 size_t workspace_bytes, const int32_t *block_tables,
                 int32_t block_table_stride, const uint32_t *seq_lens,
                 int32_t batch_size, int32_t max_seq_len, float bmm1_scale,
                 float bmm2_scale, int32_t window_left, const float *sinks,
                 int32_t q_len_per_req, int32_t num_qo_heads,
                 int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                 int32_t layout, int32_t dtype, void *out, float *lse,
                 int32_t *err_word, void *stream);

/*
 * paged_decode_varlen -- [decode] with variable-length queries: the page's
 * cum_seq_lens_q ([batch_size + 1] int32, device) and max_q_len.  Request b
 * has Q_b = cum_seq_lens_q[b+1] - cum_seq_lens_q[b] query tokens, at rows
 * cum_seq_lens_q[b] + t (t < Q_b) of query/out/lse; they are the last Q_b
 * positions of its kv sequence (p = L - Q_b + t), causal among themselves,
 * with everything else as in paged_decode.  num_tokens is the number of
 * rows query/out hold (the page's num_tokens); max_q_len bounds every Q_b
 * and sizes the workspace (paged_decode_workspace_size with q_len_per_req =
 * max_q_len).  The uniform case is cum_seq_lens_q[b] = b * q_len_per_req.
 * Device errors: an entry with cum[b] < 0, Q_b < 0, Q_b > max_q_len or
 * cum[b+1] > num_tokens -> PKV_DEV_ERR_QLEN and the request is skipped.
 * Host errors: cum_seq_lens_q NULL -> PKV_ERR_NULL; num_tokens < 0 ->
 * PKV_ERR_INVALID_ARG; others as paged_decode (max_q_len in the role of
 * q_len_per_req).
 */
int paged_decode_varlen(const void *query, int64_t num_tokens, const void *k_cache,
                        const void *v_cache, int64_t page_stride, int64_t max_num_pages,
                        void *workspace, size_t workspace_bytes,
                        const int32_t *block_tables, int32_t block_table_stride,
                        const uint32_t *seq_lens, int32_t batch_size, int32_t max_seq_len,
                        float bmm1_scale, float bmm2_scale, int32_t window_left,
                        const float *sinks, int32_t max_q_len,
                        const int32_t *cum_seq_lens_q, int32_t num_qo_heads,
                        int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                        int32_t layout, int32_t dtype, void *out, float *lse,
                        int32_t *err_word, void *stream);

/*
 * paged_decode_ex -- [decode] with the two remaining options of the page's
 * decode call: bmm1_scale / bmm2_scale given as float32 device tensors, and
 * enable_pdl.
 *  - bmm1_scale_dev / bmm2_scale_dev: NULL, or a device pointer to one fp32
 *    value that replaces the host bmm1_scale / bmm2_scale.  The kernels read
 *    it when they run (not when the call is made), so a CUDA graph captured
 *    once follows later writes to that value; the caller keeps it alive until
 *    the call's kernels finish.
 *  - enable_pdl != 0: the first kernel of the call is launched as a
 *    programmatic dependent of the stream's previous kernel (the page's
 *    programmatic dependent launch); it starts its prologue early and waits
 *    for that kernel's memory before touching any input.  0: an ordinary
 *    launch.  Results are identical either way.
 *  - cum_seq_lens_q NULL: uniform queries, max_q_len tokens per request
 *    (paged_decode with q_len_per_req = max_q_len; num_tokens must be at
 *    least batch_size * max_q_len).  Otherwise as paged_decode_varlen.
 * Everything else, including errors, is as paged_decode_varlen.
 */
int paged_decode_ex(const void *query, int64_t num_tokens, const void *k_cache,
                    const void *v_cache, int64_t page_stride, int64_t max_num_pages,
                    void *workspace, size_t workspace_bytes,
                    const int32_t *block_tables, int32_t block_table_stride,
                    const uint32_t *seq_lens, int32_t batch_size, int32_t max_seq_len,
                    float bmm1_scale, float bmm2_scale, const float *bmm1_scale_dev,
                    const float *bmm2_scale_dev, int32_t window_left, const float *sinks,
                    int32_t max_q_len, const int32_t *cum_seq_lens_q,
                    int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t page_size, int32_t layout, int32_t dtype, int32_t enable_pdl,
                    void *out, float *lse, int32_t *err_word, void *stream);

/*
 * paged_decode_noalloc -- paged_decode without a caller workspace.  The API
 * pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory where they call decode (a plugin inside another
 * runtime's execution step, which owns the device memory and forbids
 * allocation there; a latency-critical loop that cannot take cudaMalloc's
 * device-wide synchronisation; a process that reserves all device memory up
 * front).  Arguments, results and device errors are those of paged_decode
 * minus `workspace` / `workspace_bytes`; it allocates and frees nothing.
 *  - The split partials go to a fixed array of PKV_NOALLOC_SCRATCH_BYTES in
 *    the library's device image; every GPU that loads the library holds one
 *    copy until the process exits.  Sizes whose
 *    paged_decode_workspace_size(...) exceeds it are rejected with
 *    PKV_ERR_WORKSPACE before anything is launched (use paged_decode then).
 *  - The first call in each CUDA context (so on each device, and again after
 *    a cudaDeviceReset, which creates a new context in which the array may
 *    sit elsewhere) looks up the array's device address
 *    (cudaGetSymbolAddress, with that context current) and caches it, keyed
 *    by the context's unique id; make that first call before any stream
 *    capture.
 *  - All calls share the one array and it keeps the last call's contents;
 *    nothing in it needs to start at zero.  Calls that overlap on the GPU
 *    (concurrent streams, or host threads on one device) race on it:
 *    serialise them.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)
int paged_decode_noalloc(const void *query, const void *k_cache,
                         const void *v_cache, int64_t page_stride,
                         int64_t max_num_pages, const int32_t *block_tables,
                         int32_t block_table_stride, const uint32_t *seq_lens,
                         int32_t batch_size, int32_t max_seq_len,
                         float bmm1_scale, float bmm2_scale, int32_t window_left,
                         const float *sinks, int32_t q_len_per_req,
                         int32_t num_qo_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t page_size, int32_t layout,
                         int32_t dtype, void *out, float *lse, int32_t *err_word,
                         void *stream);

/*
 * paged_prefill_workspace_size -- bytes of device workspace paged_prefill
 * needs (packed query offsets and the work list of query tiles).  The
 * prefill page's workspace_buffer plays the same role.
 */
size_t paged_prefill_workspace_size(int32_t batch_size, int32_t num_qo_heads,
                                    int32_t max_token_per_sequence,
                                    int32_t max_sequence_kv);

/*
 * paged_prefill -- [prefill] signature, parameters and returns (q, k_cache,
 * v_cache, scale, workspace_buffer, max_token_per_sequence, max_sequence_kv,
 * actual_seq_lens_q, actual_seq_lens_kv, block_tables, causal, return_lse
 * = true, out, lse).  Request b has q_b = actual_seq_lens_q[b] query tokens,
 * packed at rows cu_q[b] .. cu_q[b] + q_b - 1 of q/out/lse (cu_q the
 * exclusive prefix sum of the q lengths), and kv_b = actual_seq_lens_kv[b]
 * keys.  Query i sits at position kv_b - q_b + i (the queries are the last
 * q_b tokens); with causal it sees keys j <= that position, otherwise all
 * j < kv_b.  With kvh = h / (num_qo_heads / num_kv_heads):
 *   out[row, h, :] = softmax_j(scale * <q[row, h], k_j>) v_j
 *   lse[row, h]    = log sum_j e^{scale * <q[row, h], k_j>}   (natural log)
 *   q: [total_q, num_qo_heads, d_qk]; out: [total_q, num_qo_heads, d_vo];
 *   total_q is the row count of q/out/lse (rows past it are neither read
 *   nor written even if the lengths say otherwise);
 *   lse: [total_q, num_qo_heads] fp32 (required: the page says return_lse
 *   must be true).  k_cache pages hold d_qk-wide rows, v_cache pages d_vo-wide
 *   rows, each with its own page stride.  actual_seq_lens_q/kv: [batch_size]
 *   int32 on the device.  max_token_per_sequence / max_sequence_kv bound them.
 *   workspace: >= paged_prefill_workspace_size(...) bytes, 256-byte aligned.
 *   block_table_stride >= ceil(max_sequence_kv / page_size), else
 *   PKV_ERR_INVALID_ARG.  A length above its maximum sets PKV_DEV_ERR_LEN
 *   and is clamped to it.
 * Supported (prefill page note): d_qk in {128, 192}, d_vo = 128; page_size a
 * power of two in [8, 256]; num_qo_heads % num_kv_heads == 0.
 * Errors: PKV_ERR_CUDA also when the driver rejects a TMA tensor map.
 * Device errors additionally include PKV_DEV_ERR_TIMEOUT if a pipeline wait
 * gave up (see pkv_set_wait_limit_ns; rows of the CTAs that stopped are
 * then left unwritten).
 * Device errors: bad page id -> PKV_DEV_ERR_PAGE; kv_b < q_b ->
 * PKV_DEV_ERR_QLEN (rows that see no key get out = 0, lse = -inf).
 * block_tables = NULL (the page's non-paged case): k_cache / v_cache are
 * contiguous [max_num_pages rows, num_kv_heads, d] tensors (token-major, so
 * layout must be PKV_NHD), k_page_stride / v_page_stride are their row
 * strides in elements, request b's keys are rows cu_kv[b] + j (cu_kv the
 * exclusive prefix sum of the kv lengths), and page_size /
 * block_table_stride are ignored.
 */
int paged_prefill(const void *q, int64_t total_q, const void *k_cache,
                  const void *v_cache,
                  int64_t k_page_stride, int64_t v_page_stride,
                  int64_t max_num_pages, float scale, void *workspace,
                  size_t workspace_bytes, int32_t max_token_per_sequence,
                  int32_t max_sequence_kv, const int32_t *actual_seq_lens_q,
                  const int32_t *actual_seq_lens_kv, const int32_t *block_tables,
                  int32_t block_table_stride, int32_t batch_size, int32_t causal,
                  int32_t num_qo_heads, int32_t num_kv_heads, int32_t d_qk,
                  int32_t d_vo, int32_t page_size, int32_t layout, int32_t dtype,
                  void *out, float *lse, int32_t *err_word, void *stream);

/*
 * paged_prefill_ex -- paged_prefill with the prefill page's batch offsets
 * (batch_offsets_q, batch_offsets_o, batch_offsets_k, batch_offsets_v:
 * [batch_size] int32 on the device, each optional).  The page gives no unit;
 * they are read as token rows: request b's queries are rows
 * batch_offsets_q[b] + i of q, its outputs and LSEs rows
 * batch_offsets_o[b] + i of out / lse, and (contiguous K/V only) its keys /
 * values rows batch_offsets_k[b] + j / batch_offsets_v[b] + j.  A NULL array
 * keeps the packed placement of paged_prefill.  Output rows outside
 * [0, total_q) are not written (the debug build, pkv_debug_bounds, also sets
 * PKV_DEV_ERR_BOUNDS for them).  Host errors: K/V offsets together with a
 * block table -> PKV_ERR_INVALID_ARG; the rest as paged_prefill.
 */
int paged_prefill_ex(const void *q, int64_t total_q, const void *k_cache,
                     const void *v_cache,
                     int64_t k_page_stride, int64_t v_page_stride,
                     int64_t max_num_pages, float scale, void *workspace,
                     size_t workspace_bytes, int32_t max_token_per_sequence,
                     int32_t max_sequence_kv, const int32_t *actual_seq_lens_q,
                     const int32_t *actual_seq_lens_kv, const int32_t *block_tables,
                     int32_t block_table_stride, int32_t batch_size, int32_t causal,
                     int32_t num_qo_heads, int32_t num_kv_heads, int32_t d_qk,
                     int32_t d_vo, int32_t page_size, int32_t layout, int32_t dtype,
                     void *out, float *lse, const int32_t *batch_offsets_q,
                     const int32_t *batch_offsets_o, const int32_t *batch_offsets_k,
                     const int32_t *batch_offsets_v, int32_t *err_word, void *stream);

/*
 * paged_prefill_fp8 -- [prefill] with the page's q_scale, k_scale and
 * v_scale: the query and/or the paged caches hold E4M3 (OCP FP8, one byte
 * per element) values, dequantised as q_scale * q, k_scale * k and
 * v_scale * v.  The output is out_dtype (PKV_F16 or PKV_BF16, the page's
 * o_data_type); lse is the log-sum-exp of the dequantised logits.
 *  - q_dtype: PKV_E4M3 or out_dtype; kv_dtype: PKV_E4M3 or out_dtype.
 *  - q_scale, k_scale, v_scale: NULL (1) or a device pointer to one fp32
 *    value, read when the kernels run (a captured graph follows later
 *    writes).
 *  - Page strides are in elements (bytes for E4M3); E4M3 caches need
 *    16-byte aligned bases and page strides that are multiples of 16.
 *  - Paged caches only (block_tables non-NULL); packed rows (no batch
 *    offsets).
 *  - workspace: >= paged_prefill_fp8_workspace_size(...) bytes, 256-byte
 *    aligned.  With an E4M3 query and E4M3 caches at d_qk = d_vo = 128 the
 *    attention kernel reads the E4M3 bytes as they are (QK as E4M3 x E4M3
 *    tensor-core MMAs, V tiles widened exactly to fp16 in shared memory, P
 *    in fp16) and the workspace is the plain prefill's.  Otherwise the E4M3
 *    inputs are widened (exactly: every E4M3 value is an fp16 and a bf16
 *    value) into it before the attention kernel: the query rows, and the
 *    caches packed request by request, for which it reserves
 *    batch_size * max_sequence_kv keys.
 * Device errors as paged_prefill (a page id outside the pool flags
 * PKV_DEV_ERR_PAGE and its keys read as zeros).  Host errors: a dtype other
 * than those above or no block table -> PKV_ERR_INVALID_ARG; misaligned
 * E4M3 caches -> PKV_ERR_INVALID_ARG; the rest as paged_prefill.
 */
size_t paged_prefill_fp8_workspace_size(int32_t batch_size, int32_t num_qo_heads,
                                        int32_t num_kv_heads,
                                        int32_t max_token_per_sequence,
                                        int32_t max_sequence_kv, int64_t total_q,
                                        int32_t d_qk, int32_t d_vo, int32_t q_dtype,
                                        int32_t kv_dtype);
int paged_prefill_fp8(const void *q, int64_t total_q, const void *k_cache,
                      const void *v_cache, int64_t k_page_stride,
                      int64_t v_page_stride, int64_t max_num_pages, float scale,
                      const float *q_scale, const float *k_scale, const float *v_scale,
                      void *workspace, size_t workspace_bytes,
                      int32_t max_token_per_sequence, int32_t max_sequence_kv,
                      const int32_t *actual_seq_lens_q,
                      const int32_t *actual_seq_lens_kv, const int32_t *block_tables,
                      int32_t block_table_stride, int32_t batch_size, int32_t causal,
                      int32_t num_qo_heads, int32_t num_kv_heads, int32_t d_qk,
                      int32_t d_vo, int32_t page_size, int32_t layout, int32_t q_dtype,
                      int32_t kv_dtype, int32_t out_dtype, void *out, float *lse,
                      int32_t *err_word, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
