// append.cu -- index helpers and the paged append scatter.
//
// Follows flashinfer.page.append_paged_kv_cache: its parameter list (the
// (batch_indices, positions) COO form of the new tokens and the
// kv_indptr / kv_indices / kv_last_page_len page table), its worked example
// (get_seq_lens, get_batch_indices_positions) and its note that the page
// table already covers the appended tokens.
#include "pkv_common.cuh"
#include "sm103_ptx.cuh"

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
    const uint8_t *key;    // [nnz, H, D] 16-bit elements
    const uint8_t *value;
    int64_t nnz;
    const int32_t *batch_indices;
    const int32_t *positions;
    uint8_t *k_cache;
    uint8_t *v_cache;
    int esize;  // bytes per element: 2 (fp16 / bf16) or 1 (e4m3)
    int64_t page_stride;  // elements
    int64_t max_num_pages;
    int64_t kv_extent;  // elements a cache pointer spans: (max_num_pages - 1) * page_stride + one page
    const int32_t *kv_indices;
    const int32_t *kv_indptr;
    const int32_t *kv_last_page_len;
    int B, H, D, page_size;
    int heads_per_piece;   // whole heads per copied piece (piece <= kApSlotBytes)
    int pieces_per_row;    // ceil(H / heads_per_piece)
    int64_t tokens_per_cta;
    int32_t *err;
    unsigned long long wait_ns;  // limit of the bounded copy waits
};

constexpr int kApSlots = 6;            // shared-memory ring of one CTA
constexpr int kApSlotBytes = 8192;     // largest piece of a token row
constexpr int kApCtasPerSm = 4;

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;\n" ::"l"(
                     reinterpret_cast<uint64_t>(dst)),
                 "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;\n" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory"); }

// Destination of one token: element offset of head 0 of its K (and V) row in
// the pool, or -1 when its request, position or page is out of range (the
// matching bit goes to the error word and the token is skipped).
template <int LAYOUT>
__device__ __forceinline__ int64_t append_dst(const AppendParams &p, int64_t tok) {
    if (tok >= p.nnz) return -1;
    const int b = p.batch_indices[tok];
    if (b < 0 || b >= p.B) {
        set_err(p.err, PKV_DEV_ERR_BATCH);
        return -1;
    }
    const int first = p.kv_indptr[b];
    const int pages = p.kv_indptr[b + 1] - first;
    const int len = pages > 0 ? (pages - 1) * p.page_size + p.kv_last_page_len[b] : 0;
    const int pos = p.positions[tok];
    if (pos < 0 || pos >= len) {
        set_err(p.err, PKV_DEV_ERR_POS);
        return -1;
    }
    if (kDebugBounds && !dbg_in(first + pos / p.page_size, 1, p.kv_indptr[p.B], p.err)) return -1;
    const int64_t page = p.kv_indices[first + pos / p.page_size];
    if (page < 0 || page >= p.max_num_pages) {
        set_err(p.err, PKV_DEV_ERR_PAGE);
        return -1;
    }
    const int64_t dst = kv_row_offset<LAYOUT>(page, p.page_stride, 0, pos % p.page_size, p.H, p.page_size, p.D);
    // the token's whole row: H * D contiguous elements (NHD) or H head rows
    // page_size * D apart (HND)
    const int64_t span = LAYOUT == PKV_NHD ? static_cast<int64_t>(p.H) * p.D
                                           : static_cast<int64_t>(p.H - 1) * p.page_size * p.D + p.D;
    return dbg_in(dst, span, p.kv_extent, p.err) ? dst : -1;
}

// One warp per CTA copies a contiguous run of tokens with the bulk-copy
// engine: every token row (K, then V; H*D 16-bit elements) is cut into
// pieces of whole heads of at most kApSlotBytes, each loaded from the new
// tokens into a slot of a shared-memory ring and stored from there into its
// page (one store for NHD, where a token's heads are contiguous; one per
// head for HND).  Loads run kApSlots-1 pieces ahead of the stores; a slot is
// reloaded once the store that read it has finished reading.  The lanes
// resolve the destinations of 32 tokens at a time (lane i: token i), two
// groups ahead of need; one elect.sync leader issues every copy.
template <int LAYOUT>
__global__ void __launch_bounds__(32) append_kernel(AppendParams p) {
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t full[kApSlots];
    const int lane = threadIdx.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * p.tokens_per_cta;
    const int64_t t1 = min(p.nnz, t0 + p.tokens_per_cta);
    if (t0 >= t1) return;
    const bool leader = elect_one();
    const int leader_lane = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
    if (leader) {
        for (int s = 0; s < kApSlots; ++s) mbar_init(smem_u32(&full[s]), 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint32_t ring_s = smem_u32(ring);
    const int npr = p.pieces_per_row;
    const int64_t per_tok = 2 * npr;
    const int64_t total = (t1 - t0) * per_tok;
    const int64_t row_elems = static_cast<int64_t>(p.H) * p.D;
    // destinations of tokens gA .. gA+31 (lane i: gA + i) and of the next 32
    int64_t gA = t0;
    int64_t dA = append_dst<LAYOUT>(p, gA + lane);
    int64_t dB = append_dst<LAYOUT>(p, gA + 32 + lane);
    auto dst_of = [&](int64_t tok) -> int64_t {  // warp-uniform tok
        const int64_t i = tok - gA;
        const int64_t a = __shfl_sync(0xffffffffu, dA, static_cast<int>(i & 31));
        const int64_t b = __shfl_sync(0xffffffffu, dB, static_cast<int>(i & 31));
        return i < 32 ? a : b;
    };
    // piece j: token, row (0 = K, 1 = V), first head and head count
    auto piece = [&](int64_t j, int64_t &tok, int &row, int &h0, int &nh) {
        tok = t0 + j / per_tok;
        const int r = static_cast<int>(j % per_tok);
        row = r / npr;
        h0 = (r % npr) * p.heads_per_piece;
        nh = min(p.heads_per_piece, p.H - h0);
    };
    // (debug build) the piece's heads lie inside the row and its bytes fit a
    // ring slot; both sides skip a piece that fails
    auto piece_in = [&](int h0, int nh) {
        return dbg_in(h0, nh, p.H, p.err) && dbg_in(0, static_cast<int64_t>(nh) * p.D * p.esize, kApSlotBytes, p.err);
    };
    auto issue_load = [&](int64_t j) {
        int64_t tok;
        int row, h0, nh;
        piece(j, tok, row, h0, nh);
        const int64_t dst = dst_of(tok);
        const int s = static_cast<int>(j % kApSlots);
        const uint32_t bar = smem_u32(&full[s]);
        if (leader) {
            if (dst >= 0 && piece_in(h0, nh)) {
                const uint32_t bytes = static_cast<uint32_t>(nh) * p.D * p.esize;
                mbar_expect_tx(bar, bytes);
                const uint8_t *src = (row ? p.value : p.key) + (tok * row_elems + static_cast<int64_t>(h0) * p.D) * p.esize;
                bulk_load(ring_s + s * kApSlotBytes, src, bytes, bar);
            } else {
                mbar_arrive(bar);  // nothing to copy: complete the phase
            }
        }
    };
    bool ok = true;
    volatile int no_abort = 0;
    int64_t jl = 0;
    for (; jl < total && jl < kApSlots - 1; ++jl) issue_load(jl);
    int64_t js = 0;
    for (; js < total; ++js) {
        int64_t tok;
        int row, h0, nh;
        piece(js, tok, row, h0, nh);
        if (tok - gA >= 32) {  // the store side left group A: shift, resolve the next group
            gA += 32;
            dA = dB;
            dB = append_dst<LAYOUT>(p, gA + 32 + lane);
        }
        const int64_t dst = dst_of(tok);
        const int s = static_cast<int>(js % kApSlots);
        if (leader) {
            if (!mbar_wait(smem_u32(&full[s]), static_cast<uint32_t>((js / kApSlots) & 1), &no_abort, p.wait_ns)) {
                set_err(p.err, PKV_DEV_ERR_TIMEOUT);
                ok = false;
            } else if (dst >= 0 && piece_in(h0, nh)) {
                uint8_t *cache = row ? p.v_cache : p.k_cache;
                const uint32_t src = ring_s + s * kApSlotBytes;
                const uint32_t hb = static_cast<uint32_t>(p.D) * p.esize;
                if (LAYOUT == PKV_NHD) {
                    bulk_store(cache + (dst + static_cast<int64_t>(h0) * p.D) * p.esize, src, nh * hb);
                } else {
                    for (int h = 0; h < nh; ++h)
                        bulk_store(cache + (dst + static_cast<int64_t>(h0 + h) * p.page_size * p.D) * p.esize,
                                   src + h * hb, hb);
                }
            }
            bulk_commit();
        }
        if (!__shfl_sync(0xffffffffu, ok, leader_lane)) break;
        if (jl < total) {
            if (leader) bulk_wait_read1();  // the store that last read slot jl % kApSlots is done reading
            issue_load(jl);
            ++jl;
        }
    }
    // A wait that gave up left the loads of pieces js .. jl-1 in flight (at
    // most one per slot): they land in this CTA's shared memory, so wait for
    // them before it exits; then for the stores.
    if (leader && !ok)
        for (int64_t j = js; j < jl; ++j)
            mbar_wait_drain(smem_u32(&full[j % kApSlots]), static_cast<uint32_t>((j / kApSlots) & 1));
    if (leader) bulk_wait_all();
}

}  // namespace pkv

using namespace pkv;

extern "C" int paged_seq_lens(const int32_t *kv_indptr, const int32_t *kv_last_page_len,
                              int32_t batch_size, int32_t page_size, int32_t *seq_lens,
                              void *stream) {
    const CallRange nvtx_range("paged_seq_lens");
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
    const CallRange nvtx_range("paged_batch_indices_positions");
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
    const CallRange nvtx_range("paged_append");
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16 && dtype != PKV_E4M3) return PKV_ERR_INVALID_ARG;
    const int esize = dtype == PKV_E4M3 ? 1 : 2;  // bytes per element; bits are copied unchanged
    if (nnz < 0 || batch_size < 0 || num_kv_heads <= 0 || head_dim <= 0 || page_size <= 0 ||
        max_num_pages < 0 || page_stride <= 0)
        return PKV_ERR_INVALID_ARG;
    if ((head_dim * esize) % 16) return PKV_ERR_INVALID_ARG;  // 16-byte head rows
    if (head_dim * esize > kApSlotBytes) return PKV_ERR_UNSUPPORTED;  // one head must fit a ring slot
    if (page_stride < static_cast<int64_t>(num_kv_heads) * page_size * head_dim)
        return PKV_ERR_INVALID_ARG;
    if (nnz == 0) return PKV_OK;
    if (!append_key || !append_value || !batch_indices || !positions || !k_cache || !v_cache ||
        !kv_indices || !kv_indptr || !kv_last_page_len)
        return PKV_ERR_NULL;
    if (!aligned16(append_key) || !aligned16(append_value) || !aligned16(k_cache) ||
        !aligned16(v_cache) || ((page_stride * esize) % 16))
        return PKV_ERR_INVALID_ARG;

    AppendParams p;
    p.key = static_cast<const uint8_t *>(append_key);
    p.value = static_cast<const uint8_t *>(append_value);
    p.nnz = nnz;
    p.batch_indices = batch_indices;
    p.positions = positions;
    p.k_cache = static_cast<uint8_t *>(k_cache);
    p.v_cache = static_cast<uint8_t *>(v_cache);
    p.esize = esize;
    p.page_stride = page_stride;
    p.max_num_pages = max_num_pages;
    p.kv_extent = max_num_pages > 0 ? (max_num_pages - 1) * page_stride +
                                          static_cast<int64_t>(num_kv_heads) * page_size * head_dim
                                    : 0;
    p.kv_indices = kv_indices;
    p.kv_indptr = kv_indptr;
    p.kv_last_page_len = kv_last_page_len;
    p.B = batch_size;
    p.H = num_kv_heads;
    p.D = head_dim;
    p.page_size = page_size;
    p.heads_per_piece = head_dim * esize >= kApSlotBytes ? 1 : min(num_kv_heads, kApSlotBytes / (head_dim * esize));
    p.pieces_per_row = (num_kv_heads + p.heads_per_piece - 1) / p.heads_per_piece;
    p.err = err_word;
    p.wait_ns = wait_limit_ns();
    const int64_t ctas_max = static_cast<int64_t>(num_sms()) * kApCtasPerSm;
    p.tokens_per_cta = (nnz + ctas_max - 1) / ctas_max;
    const int64_t blocks = (nnz + p.tokens_per_cta - 1) / p.tokens_per_cta;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t smem = static_cast<size_t>(kApSlots) * kApSlotBytes;
    // the ring plus the static barriers exceed the default 48 KB per block
    auto kern = layout == PKV_HND ? append_kernel<PKV_HND> : append_kernel<PKV_NHD>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    kern<<<static_cast<unsigned>(blocks), 32, smem, st>>>(p);
    note_launches(1);
    return launch_status();
}
