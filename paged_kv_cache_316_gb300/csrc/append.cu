// append.cu -- index helpers and the paged append scatter.
//
// Follows flashinfer.page.append_paged_kv_cache: its parameter list (the
// (batch_indices, positions) COO form of the new tokens and the
// kv_indptr / kv_indices / kv_last_page_len page table), its worked example
// (get_seq_lens, get_batch_indices_positions) and its note that the page
// table already covers the appended tokens.
#include "pkv_common.cuh"

namespace pkv {

// seq_lens[b] = (pages_b - 1) * page_size + last_page_len[b]   (0 pages -> 0)
__global__ void seq_lens_kernel(const int32_t *__restrict__ kv_indptr,
                                const int32_t *__restrict__ last, int B, int page_size,
                                int32_t *__restrict__ out) {
    int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int pages = kv_indptr[b + 1] - kv_indptr[b];
    out[b] = pages > 0 ? (pages - 1) * page_size + last[b] : 0;
}

// Entry i belongs to the last request b with append_indptr[b] <= i; its
// position counts back from the end of that request's sequence.
__global__ void batch_pos_kernel(const int32_t *__restrict__ indptr,
                                 const int32_t *__restrict__ seq_lens, int B, int64_t nnz,
                                 int32_t *__restrict__ bi, int32_t *__restrict__ pos) {
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= nnz) return;
    if (B <= 0 || i < indptr[0] || i >= indptr[B]) {
        bi[i] = -1;
        pos[i] = -1;
        return;
    }
    int l = 0, r = B - 1;
    while (l < r) {
        int mid = (l + r + 1) >> 1;
        if (indptr[mid] <= i) l = mid;
        else r = mid - 1;
    }
    int start = indptr[l];
    int n = indptr[l + 1] - start;
    bi[i] = l;
    pos[i] = seq_lens[l] - n + static_cast<int>(i - start);
}

struct AppendParams {
    const uint4 *key;    // [nnz, H, D] 16-bit elements, viewed as 16-byte chunks
    const uint4 *value;
    int64_t nnz;
    const int32_t *batch_indices;
    const int32_t *positions;
    uint16_t *k_cache;
    uint16_t *v_cache;
    int64_t page_stride;  // elements
    int64_t max_num_pages;
    const int32_t *kv_indices;
    const int32_t *kv_indptr;
    const int32_t *kv_last_page_len;
    int B, H, D, page_size;
    int chunks_per_row;  // H * D / 8 (16-byte chunks in one token's K row)
    int tokens_per_cta;
    int32_t *err;
};

constexpr int kAppendThreads = 256;
constexpr int kAppendUnroll = 4;

// Each CTA copies `tokens_per_cta` whole tokens (K row then V row, H*D
// elements each) as 16-byte chunks: every thread first issues up to
// kAppendUnroll streaming loads, then the matching stores, so a warp keeps
// 2 KB in flight per round.  Source reads are contiguous; destination rows
// are contiguous H*D runs (NHD) or D-element runs page_size*D apart (HND).
template <int LAYOUT>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(AppendParams p) {
    const int two_ch = 2 * p.chunks_per_row;
    const int per_cta = p.tokens_per_cta * two_ch;
    const int dchunks = p.D >> 3;
    const int64_t tok0 = static_cast<int64_t>(blockIdx.x) * p.tokens_per_cta;
    for (int base = 0; base < per_cta; base += kAppendThreads * kAppendUnroll) {
        uint4 val[kAppendUnroll];
        uint4 *dst[kAppendUnroll];
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u) {
            dst[u] = nullptr;
            int li = base + u * kAppendThreads + threadIdx.x;
            if (li >= per_cta) continue;
            int tl = li / two_ch;
            int rem = li - tl * two_ch;
            int64_t tok = tok0 + tl;
            if (tok >= p.nnz) continue;
            bool is_v = rem >= p.chunks_per_row;
            int c = is_v ? rem - p.chunks_per_row : rem;
            bool leader = rem == 0;
            int b = p.batch_indices[tok];
            if (b < 0 || b >= p.B) {
                if (leader) set_err(p.err, PKV_DEV_ERR_BATCH);
                continue;
            }
            int first = p.kv_indptr[b];
            int pages = p.kv_indptr[b + 1] - first;
            int len = pages > 0 ? (pages - 1) * p.page_size + p.kv_last_page_len[b] : 0;
            int pos = p.positions[tok];
            if (pos < 0 || pos >= len) {
                if (leader) set_err(p.err, PKV_DEV_ERR_POS);
                continue;
            }
            int64_t page = p.kv_indices[first + pos / p.page_size];
            if (page < 0 || page >= p.max_num_pages) {
                if (leader) set_err(p.err, PKV_DEV_ERR_PAGE);
                continue;
            }
            int slot = pos % p.page_size;
            int h = c / dchunks;
            int dc = c - h * dchunks;
            const uint4 *src = (is_v ? p.value : p.key) + tok * p.chunks_per_row + c;
            val[u] = __ldcs(src);
            uint16_t *cache = is_v ? p.v_cache : p.k_cache;
            int64_t off = kv_row_offset<LAYOUT>(page, p.page_stride, h, slot, p.H, p.page_size, p.D) +
                          static_cast<int64_t>(dc) * 8;
            dst[u] = reinterpret_cast<uint4 *>(cache + off);
        }
#pragma unroll
        for (int u = 0; u < kAppendUnroll; ++u)
            if (dst[u]) __stcs(dst[u], val[u]);
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" int paged_seq_lens(const int32_t *kv_indptr, const int32_t *kv_last_page_len,
                              int32_t batch_size, int32_t page_size, int32_t *seq_lens,
                              void *stream) {
    if (batch_size < 0 || page_size <= 0) return PKV_ERR_INVALID_ARG;
    if (batch_size == 0) return PKV_OK;
    if (!kv_indptr || !kv_last_page_len || !seq_lens) return PKV_ERR_NULL;
    int threads = 256, blocks = (batch_size + threads - 1) / threads;
    seq_lens_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
        kv_indptr, kv_last_page_len, batch_size, page_size, seq_lens);
    note_launches(1);
    return launch_status();
}

extern "C" int paged_batch_indices_positions(const int32_t *append_indptr,
                                             const int32_t *seq_lens, int32_t batch_size,
                                             int64_t nnz, int32_t *batch_indices,
                                             int32_t *positions, void *stream) {
    if (batch_size < 0 || nnz < 0) return PKV_ERR_INVALID_ARG;
    if (nnz == 0) return PKV_OK;
    if (!append_indptr || !seq_lens || !batch_indices || !positions) return PKV_ERR_NULL;
    int threads = 256;
    int64_t blocks = (nnz + threads - 1) / threads;
    if (blocks > 0x7fffffff) return PKV_ERR_INVALID_ARG;
    batch_pos_kernel<<<static_cast<unsigned>(blocks), threads, 0,
                       static_cast<cudaStream_t>(stream)>>>(append_indptr, seq_lens, batch_size,
                                                            nnz, batch_indices, positions);
    note_launches(1);
    return launch_status();
}

extern "C" int paged_append(const void *append_key, const void *append_value, int64_t nnz,
                            const int32_t *batch_indices, const int32_t *positions,
                            void *k_cache, void *v_cache, int64_t page_stride,
                            int64_t max_num_pages, const int32_t *kv_indices,
                            const int32_t *kv_indptr, const int32_t *kv_last_page_len,
                            int32_t batch_size, int32_t num_kv_heads, int32_t head_dim,
                            int32_t page_size, int32_t layout, int32_t dtype,
                            int32_t *err_word, void *stream) {
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (nnz < 0 || batch_size < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
        max_num_pages < 0 || page_stride <= 0)
        return PKV_ERR_INVALID_ARG;
    if (head_dim % 8) return PKV_ERR_INVALID_ARG;
    if (page_stride < static_cast<int64_t>(num_kv_heads) * page_size * head_dim)
        return PKV_ERR_INVALID_ARG;
    if (nnz == 0) return PKV_OK;
    if (!append_key || !append_value || !batch_indices || !positions || !k_cache || !v_cache ||
        !kv_indices || !kv_indptr || !kv_last_page_len)
        return PKV_ERR_NULL;
    if (!aligned16(append_key) || !aligned16(append_value) || !aligned16(k_cache) ||
        !aligned16(v_cache) || (page_stride % 8))
        return PKV_ERR_INVALID_ARG;

    AppendParams p;
    p.key = static_cast<const uint4 *>(append_key);
    p.value = static_cast<const uint4 *>(append_value);
    p.nnz = nnz;
    p.batch_indices = batch_indices;
    p.positions = positions;
    p.k_cache = static_cast<uint16_t *>(k_cache);
    p.v_cache = static_cast<uint16_t *>(v_cache);
    p.page_stride = page_stride;
    p.max_num_pages = max_num_pages;
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.kv_last_page_len = kv_last_page_len;
    p.B = batch_size;
    p.H = num_kv_heads;
    p.D = head_dim;
    p.page_size = page_size;
    p.chunks_per_row = num_kv_heads * head_dim / 8;
    p.err = err_word;
    int target = kAppendThreads * kAppendUnroll;
    p.tokens_per_cta = 2 * p.chunks_per_row >= target ? 1 : target / (2 * p.chunks_per_row);
    int64_t blocks = (nnz + p.tokens_per_cta - 1) / p.tokens_per_cta;
    if (blocks > 0x7fffffff) return PKV_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (layout == PKV_HND)
        append_kernel<PKV_HND><<<static_cast<unsigned>(blocks), kAppendThreads, 0, st>>>(p);
    else
        append_kernel<PKV_NHD><<<static_cast<unsigned>(blocks), kAppendThreads, 0, st>>>(p);
    note_launches(1);
    return launch_status();
}
