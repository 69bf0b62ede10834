// decode.cu -- split-KV GQA batch decode over a paged KV cache.
//
// Computes what flashinfer.decode.trtllm_batch_decode_with_kv_cache
// documents (parameters query, kv_cache, workspace_buffer, block_tables,
// seq_lens, max_seq_len, bmm1_scale, bmm2_scale, window_left, sinks,
// kv_layout, q_len_per_req): for every request, kv head and split of its
// visible key range, one CTA streams the split's K/V rows through a
// cp.async ring in shared memory and keeps an online softmax; a second
// kernel merges the splits by their log-sum-exp and adds the sink term.
//
// Row packing: the group = Hqo / Hkv query heads that share a kv head and
// the Q query tokens of a request form R = group * Q rows, padded to
// 16 * MT rows of one mma.sync m16n8k16 A operand, so each K/V row read
// from HBM feeds every query row that needs it.
#include <math.h>

#include <type_traits>

#include "pkv_common.cuh"

namespace pkv {

constexpr int kDecD = 128;                        // head_dim
constexpr int kDecTile = 64;                      // keys per pipeline stage
// Ring depth and CTAs per SM.  One row tile (up to 16 packed query rows): 3
// CTAs per SM with a 2-stage ring; more row tiles need more registers: 2
// CTAs per SM, 3 stages.  An E4M3 stage is half as large, so its ring is 4
// stages deep at the same CTA counts.
template <int MT, bool KV8 = false>
struct DecCfg {
    static constexpr int STAGES = KV8 ? 4 : (MT == 1 ? 2 : 3);
    static constexpr int CTAS = MT == 1 ? 3 : 2;
};
constexpr int kDecThreads = 128;
constexpr int kDecRowBytes = kDecD * 2;           // one K or V row
constexpr int kDecTileBytes = kDecTile * kDecRowBytes;
constexpr int kDecStageBytes = 2 * kDecTileBytes; // K tile then V tile
// An E4M3 cache is staged as 128-byte rows (K then V, 8 KB each per tile),
// 16-byte chunk c of row r at chunk c ^ (r & 7), and the MMA fragments are
// widened straight from those bytes (no 16-bit copy of the tile).
constexpr int kDec8RowBytes = kDecD;
constexpr int kDec8TileBytes = kDecTile * kDec8RowBytes;
template <bool KV8>
struct DecSmem {
    static constexpr int STAGE = KV8 ? 2 * kDec8TileBytes : kDecStageBytes;  // one ring stage
};
__device__ __forceinline__ int swz8(int r, int c) { return r * kDec8RowBytes + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ float2 unpack2_bf16(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}
constexpr int kDecMinPage = 8;                    // smallest supported page size
constexpr int kDecMaxChunk = 5120;                // largest split (keys)
constexpr int kDecMaxPages = kDecMaxChunk / kDecMinPage + 2;  // page ids one split can touch

struct DecodeParams {
    const void *q;
    const void *k;
    const void *v;
    int64_t page_stride;
    int64_t max_num_pages;
    const int32_t *block_tables;
    int64_t bt_stride;
    const uint32_t *seq_lens;
    int B;
    int max_seq_len;
    float scale_log2;  // bmm1_scale * log2(e): logits in base-2 units
    // device-resident fp32 bmm1 / bmm2 scales (NULL: the host values), read
    // when the kernels run, so a captured graph follows their current value
    const float *bmm1_dev, *bmm2_dev;
    float bmm2;
    int window_left;
    const float *sinks;
    int Q, Hqo, Hkv, group, R;  // Q: query tokens per request (the largest, with cu_q)
    const int32_t *cu_q;        // [B+1] variable-length query rows, or NULL (rows b*Q + t)
    int64_t num_tokens;         // query / out rows the caller holds
    int64_t kv_extent;  // elements a cache pointer spans: (max_num_pages - 1) * page_stride + one page
    int64_t ws_rows;    // partial rows of the workspace (B * Hkv * n_split_max * R)
    int page_shift;
    int chunk;        // keys per split
    int n_split_max;  // split slots per (request, kv head) in the workspace
    void *out;
    float *lse;
    float *ws_o;      // [B][Hkv][n_split_max][R][128] normalised partial outputs
    float *ws_lse;    // [B][Hkv][n_split_max][R] partial log2-sum-exp
    int32_t *err;
};

// Lowest visible key `lo` of a request and how its range [lo, L) is cut into
// splits: from `first` = lo rounded down to a 64-key tile, split s covers
// keys [max(lo, first + s * chunk), min(L, first + (s + 1) * chunk)).  An
// empty request keeps one split so its rows are written.
__host__ __device__ inline void decode_split_geometry(int L, int Q, int window_left, int chunk,
                                                      int &lo, int &first, int &n_split) {
    lo = 0;
    if (window_left >= 0) {
        lo = L - Q - window_left;
        if (lo < 0) lo = 0;
    }
    first = lo & ~(kDecTile - 1);
    n_split = L <= lo ? 1 : (L - first + chunk - 1) / chunk;
}

// Barrier over the MT warps that share a slice of keys (warps kg*MT ..
// kg*MT + MT - 1): a warp sync for one, __syncthreads for all four, else the
// named barrier 1 + kg.
template <int MT>
__device__ __forceinline__ void key_group_sync(int kg) {
    if constexpr (MT == 1) {
        __syncwarp();
    } else if constexpr (MT * 32 == kDecThreads) {
        __syncthreads();
    } else {
        asm volatile("bar.sync %0, %1;\n" ::"r"(1 + kg), "n"(MT * 32) : "memory");
    }
}

template <typename T>
__device__ __forceinline__ void store4(T *dst, float a, float b, float c, float d) {
    uint2 v;
    v.x = pack2<T>(a, b);
    v.y = pack2<T>(c, d);
    *reinterpret_cast<uint2 *>(dst) = v;
}

// SW (an E4M3 cache and at most 8 query rows): the MMAs take the keys as
// their 16-row side, S^T = K Q^T and O^T = V^T P^T (see the tile loop).
template <typename T, int MT, int LAYOUT, bool KV8, bool SW = false>
__global__ void __launch_bounds__(kDecThreads, DecCfg<MT, KV8>::CTAS) decode_split_kernel(const DecodeParams p) {
    constexpr int kDecStages = DecCfg<MT, KV8>::STAGES;
    constexpr int STAGE_BYTES = DecSmem<KV8>::STAGE;
    // the MMA element type: over an E4M3 cache always fp16 (E4M3 widens to
    // fp16 in one instruction; a bf16 query is brought to fp16 exactly, see
    // below)
    using TM = typename std::conditional<KV8, __half, T>::type;
    static_assert(!SW || (KV8 && MT == 1), "swapped operands: E4M3 cache, one row tile");
    constexpr int NKG = 4 / MT;          // warps that split the keys of a tile
    constexpr int KPW = kDecTile / NKG;  // keys per warp per tile
    constexpr int NT = KPW / 8;          // 8-key score tiles per warp
    constexpr int ROWS = 16 * MT;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *q_s = smem + kDecStages * STAGE_BYTES;
    uint8_t *kvalid = q_s + ROWS * kDecRowBytes;
    float *comb_m = reinterpret_cast<float *>(kvalid + kDecStages * kDecTile);
    float *comb_l = comb_m + NKG * ROWS;
    int *pages_s = reinterpret_cast<int *>(comb_l + NKG * ROWS);  // the split's page ids
    __shared__ int any_bad[4];  // per key group: a row of its slice was on a bad page

    // launched as a dependent of the stream's previous kernel (enable_pdl):
    // wait for it before reading anything it may have written
    pdl_wait();
    const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = warp % MT, kg = warp / MT;
    const int gtid = tid - kg * MT * 32;  // thread index within the key group
    const int kw0 = kg * KPW;             // the group's key slice of every tile
    const uint32_t L_in = p.seq_lens[b];
    const int L = L_in > static_cast<uint32_t>(p.max_seq_len) ? p.max_seq_len : static_cast<int>(L_in);
    if (L_in > static_cast<uint32_t>(p.max_seq_len) && s == 0 && kvh == 0 && threadIdx.x == 0)
        set_err(p.err, PKV_DEV_ERR_LEN);
    // this request's query tokens: Q at rows b*Q + t, or Q_b at rows
    // cu_q[b] + t (an inconsistent entry -- decreasing, longer than the
    // planned maximum, or past the caller's rows -- is flagged and skipped)
    int Q = p.Q;
    int64_t qrow0 = static_cast<int64_t>(b) * p.Q;
    if (p.cu_q) {
        const int c0 = p.cu_q[b], c1 = p.cu_q[b + 1];
        Q = c1 - c0;
        qrow0 = c0;
        if (c0 < 0 || Q < 0 || Q > p.Q || c1 > p.num_tokens) {
            if (s == 0 && kvh == 0 && threadIdx.x == 0) set_err(p.err, PKV_DEV_ERR_QLEN);
            Q = 0;
        }
        if (Q == 0) return;  // uniform over the CTA: before any barrier
    }
    const int R = p.group * Q;  // query rows of this (request, kv head)
    int lo, first, n_split;
    decode_split_geometry(L, Q, p.window_left, p.chunk, lo, first, n_split);
    if (s >= n_split) return;
    if (L < Q && s == 0 && kvh == 0 && tid == 0) set_err(p.err, PKV_DEV_ERR_QLEN);
    const int k_begin = max(lo, first + s * p.chunk);
    const int k_end = min(L, first + (s + 1) * p.chunk);
    // tiles start on 64-key boundaries (a window's first key need not): the
    // rows before k_begin are zero-filled and masked like rows past the end
    const int k_tile0 = k_begin & ~(kDecTile - 1);
    const int n_tiles = k_end > k_begin ? (k_end - k_tile0 + kDecTile - 1) / kDecTile : 0;

    const T *kc = static_cast<const T *>(p.k);
    const T *vc = static_cast<const T *>(p.v);
    const uint8_t *kc8 = static_cast<const uint8_t *>(p.k);  // E4M3 cache (KV8)
    const uint8_t *vc8 = static_cast<const uint8_t *>(p.v);
    const int32_t *bt = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
    const int S = 1 << p.page_shift;
    if (tid < 4) any_bad[tid] = 0;
    // page ids of the split, fetched once (coalesced) so that the per-tile
    // address computation does not wait on global memory; -1 marks an id
    // outside the pool
    const int first_page = k_begin >> p.page_shift;
    const int n_pages = k_end > k_begin ? ((k_end - 1) >> p.page_shift) - first_page + 1 : 0;
    for (int i = tid; i < n_pages; i += kDecThreads) {
        const bool in_bt = dbg_in(first_page + i, 1, (p.max_seq_len + S - 1) >> p.page_shift, p.err);
        int page = in_bt ? bt[first_page + i] : -1;
        if (in_bt && (page < 0 || page >= p.max_num_pages)) {
            set_err(p.err, PKV_DEV_ERR_PAGE);
            page = -1;
        }
        if (dbg_in(i, 1, kDecMaxPages, p.err)) pages_s[i] = page;
    }
    __syncthreads();

    // K and V rows of a tile.  Every key group loads (and later widens) only
    // the KPW rows of its own key slice, the only rows its warps read, so a
    // tile needs no barrier wider than the group.  16 consecutive lanes copy
    // one 256-byte row: every warp instruction moves two whole rows.  Rows
    // past the split end or on an out-of-range page are zero-filled and never
    // read from global memory; kvalid records which rows hold a key.
    // A thread's rows of a tile are RSTEP apart; when they all lie before the
    // split end on one page (the common case), the page is looked up once
    // and the row address advances by a fixed step.
    constexpr int LPR = KV8 ? 8 : 16;                 // lanes per row
    constexpr int RSTEP = MT * 32 / LPR;              // rows between a thread's rows
    constexpr int NLOAD = KPW * LPR / (MT * 32);      // rows per thread per tile
    const int64_t row_step = (LAYOUT == PKV_HND ? kDecD : static_cast<int64_t>(p.Hkv) * kDecD) * RSTEP;
    auto load_tile = [&](int stage, int j0) {
        const uint32_t dst = smem_u32(smem + stage * STAGE_BYTES);
        {
            const int r0 = kw0 + gtid / LPR, c = gtid % LPR;
            const int jA = j0 + r0, jZ = jA + (NLOAD - 1) * RSTEP;
            const int pi = (jA >> p.page_shift) - first_page;
            const int page = jA >= k_begin && jZ < k_end && (jA >> p.page_shift) == (jZ >> p.page_shift) &&
                                     dbg_in(pi, 1, kDecMaxPages, p.err)
                                 ? pages_s[pi]
                                 : -1;
            if (__all_sync(0xffffffffu, page >= 0)) {
                const int64_t off = kv_row_offset<LAYOUT>(page, p.page_stride, kvh, jA & (S - 1), p.Hkv, S, kDecD);
#pragma unroll
                for (int k = 0; k < NLOAD; ++k) {
                    const int r = r0 + k * RSTEP;
                    if (c == 0) kvalid[stage * kDecTile + r] = 1;
                    if constexpr (KV8) {
                        const int64_t e = off + k * row_step + c * 16;
                        const bool in = dbg_in(e, 16, p.kv_extent, p.err);
                        cp_async_16(dst + swz8(r, c), in ? kc8 + e : kc8, in);
                        cp_async_16(dst + kDec8TileBytes + swz8(r, c), in ? vc8 + e : vc8, in);
                    } else {
                        const uint32_t o = swz(r, c, kDecRowBytes);
                        const int64_t e = off + k * row_step + c * 8;
                        const bool in = dbg_in(e, 8, p.kv_extent, p.err);
                        cp_async_16(dst + o, in ? kc + e : kc, in);
                        cp_async_16(dst + kDecTileBytes + o, in ? vc + e : vc, in);
                    }
                }
                return;
            }
        }
        if constexpr (KV8) {
            // 128-byte E4M3 rows: 8 consecutive lanes copy one row
#pragma unroll
            for (int k = 0; k < KPW * 8 / (MT * 32); ++k) {
                const int idx = k * MT * 32 + gtid;
                const int r = kw0 + (idx >> 3), c = idx & 7;
                const int j = j0 + r;
                bool ok = j >= k_begin && j < k_end;
                const uint8_t *ks = kc8, *vs = vc8;
                if (ok) {
                    const int pi = (j >> p.page_shift) - first_page;
                    const int page = dbg_in(pi, 1, kDecMaxPages, p.err) ? pages_s[pi] : -1;
                    if (page < 0) {
                        ok = false;
                        any_bad[kg] = 1;
                    } else {
                        const int64_t off = kv_row_offset<LAYOUT>(page, p.page_stride, kvh, j & (S - 1), p.Hkv,
                                                                  S, kDecD) + c * 16;
                        ok = dbg_in(off, 16, p.kv_extent, p.err);
                        if (ok) {
                            ks = kc8 + off;
                            vs = vc8 + off;
                        }
                    }
                }
                if (c == 0) kvalid[stage * kDecTile + r] = ok ? 1 : 0;
                cp_async_16(dst + swz8(r, c), ks, ok);
                cp_async_16(dst + kDec8TileBytes + swz8(r, c), vs, ok);
            }
        } else {
#pragma unroll
        for (int k = 0; k < KPW * 16 / (MT * 32); ++k) {
            const int idx = k * MT * 32 + gtid;
            const int r = kw0 + (idx >> 4), c = idx & 15;
            const int j = j0 + r;
            bool ok = j >= k_begin && j < k_end;
            const T *ks = kc, *vs = vc;
            if (ok) {
                const int pi = (j >> p.page_shift) - first_page;
                const int page = dbg_in(pi, 1, kDecMaxPages, p.err) ? pages_s[pi] : -1;
                if (page < 0) {
                    ok = false;
                    any_bad[kg] = 1;
                } else {
                    const int64_t off = kv_row_offset<LAYOUT>(page, p.page_stride, kvh, j & (S - 1), p.Hkv,
                                                              S, kDecD) + c * 8;
                    ok = dbg_in(off, 8, p.kv_extent, p.err);
                    if (ok) {
                        ks = kc + off;
                        vs = vc + off;
                    }
                }
            }
            if (c == 0) kvalid[stage * kDecTile + r] = ok ? 1 : 0;
            const uint32_t o = swz(r, c, kDecRowBytes);
            cp_async_16(dst + o, ks, ok);
            cp_async_16(dst + kDecTileBytes + o, vs, ok);
        }
        }
    };

    // query rows r = t * group + i  ->  query[(b*Q + t), kvh*group + i, :]
    const T *qp = static_cast<const T *>(p.q);
    for (int idx = tid; idx < ROWS * 16; idx += kDecThreads) {
        int r = idx >> 4, c = idx & 15;
        bool ok = r < R;
        const T *src = qp;
        if (ok) {
            int t = r / p.group, i = r - t * p.group;
            const int64_t e = ((qrow0 + t) * p.Hqo + kvh * p.group + i) * kDecD + c * 8;
            ok = dbg_in(e, 8, p.num_tokens * p.Hqo * kDecD, p.err);
            if (ok) src = qp + e;
        }
        cp_async_16(smem_u32(q_s) + swz(r, c, kDecRowBytes), src, ok);
    }
    cp_async_commit();
#pragma unroll
    for (int st = 0; st < kDecStages - 1; ++st) {
        if (st < n_tiles) load_tile(st, k_tile0 + st * kDecTile);
        cp_async_commit();
    }
    cp_async_wait<kDecStages - 1>();
    __syncthreads();

    float scale_log2 = p.bmm1_dev ? __ldg(p.bmm1_dev) * kLog2e : p.scale_log2;
    const float bmm2 = p.bmm2_dev ? __ldg(p.bmm2_dev) : p.bmm2;
    if constexpr (KV8 && !std::is_same<T, __half>::value) {
        // bf16 query -> fp16 for the fp16 MMAs: scaled by 2^e so that the
        // largest |q| of the CTA lies in [2^14, 2^15) -- every bf16 value of
        // the rows then converts exactly unless it falls below fp16's normal
        // range, 2^29 under that largest element -- with 2^-e moved into the
        // logit scale (powers of two, exact)
        __shared__ float qmax_s[kDecThreads / 32];
        float mx = 0.f;
        for (int idx = tid; idx < ROWS * 16; idx += kDecThreads) {
            const uint4 v = *reinterpret_cast<const uint4 *>(q_s + swz(idx >> 4, idx & 15, kDecRowBytes));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = unpack2_bf16(w[i]);
                mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0) qmax_s[warp] = mx;
        __syncthreads();
        mx = fmaxf(fmaxf(qmax_s[0], qmax_s[1]), fmaxf(qmax_s[2], qmax_s[3]));
        int e = 0;
        if (mx > 0.f && isfinite(mx)) {
            int ex;
            frexpf(mx, &ex);  // mx in [2^(ex-1), 2^ex)
            e = min(max(15 - ex, -100), 100);  // (beyond that the row is all but zero)
        }
        const float up = ldexpf(1.f, e);
        scale_log2 = ldexpf(scale_log2, -e);
        __syncthreads();  // every warp has its max before the tile is rewritten
        for (int idx = tid; idx < ROWS * 16; idx += kDecThreads) {
            uint4 *a = reinterpret_cast<uint4 *>(q_s + swz(idx >> 4, idx & 15, kDecRowBytes));
            const uint4 v = *a;
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = unpack2_bf16(w[i]);
                h[i] = pack2<__half>(f.x * up, f.y * up);
            }
            *a = make_uint4(h[0], h[1], h[2], h[3]);
        }
        __syncthreads();
    }

    uint32_t qa[8][4];
    if constexpr (SW) {
        // B operand of the swapped QK (Q^T, k = head dim, n = query row):
        // lane (g, c) holds row g, dims 32c + 4kk + {0, 1} and {2, 3} of
        // k-step kk (the permuted order of the K rows, below)
        const int gq = lane >> 2, cq = lane & 3;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int dim = cq * 32 + kk * 4;
            const uint2 lo = *reinterpret_cast<const uint2 *>(q_s + swz(gq, dim >> 3, kDecRowBytes) + (dim & 7) * 2);
            qa[kk][0] = lo.x;
            qa[kk][1] = lo.y;
        }
    } else if constexpr (KV8) {
        // Over an E4M3 cache the head dimension is taken in a permuted order,
        // the same for Q and K (a dot product does not depend on it): the k
        // pairs {2c, 2c+1} and {2c+8, 2c+9} of k-step kk are the dims
        // 32c + 4kk + {0,1} and {2,3}, so that one 32-bit word of a K row
        // holds both halves of a B fragment.
        const int gq = lane >> 2, cq = lane & 3;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int dim = cq * 32 + kk * 4;
            const uint2 lo = *reinterpret_cast<const uint2 *>(q_s + swz(16 * mt + gq, dim >> 3, kDecRowBytes) +
                                                              (dim & 7) * 2);
            const uint2 hi = *reinterpret_cast<const uint2 *>(q_s + swz(16 * mt + gq + 8, dim >> 3, kDecRowBytes) +
                                                              (dim & 7) * 2);
            qa[kk][0] = lo.x;
            qa[kk][1] = hi.x;
            qa[kk][2] = lo.y;
            qa[kk][3] = hi.y;
        }
    } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            ldsm_x4(qa[kk], smem_u32(q_s) + swz(16 * mt + (lane & 15), 2 * kk + (lane >> 4), kDecRowBytes));
    }

    // the two rows this lane holds in every accumulator fragment
    const int r0 = 16 * mt + (lane >> 2), r1 = r0 + 8;
    const int t0 = min(r0 / p.group, Q - 1), t1 = min(r1 / p.group, Q - 1);
    const int pos0 = L - Q + t0, pos1 = L - Q + t1;
    const int lo0 = p.window_left >= 0 ? max(0, pos0 - p.window_left) : 0;
    const int lo1 = p.window_left >= 0 ? max(0, pos1 - p.window_left) : 0;
    const int lo_max = p.window_left >= 0 ? max(0, L - 1 - p.window_left) : 0;
    const int hi_min = min(L - Q, k_end - 1);
    // (swapped operands: lane (g, c) holds query rows 2c and 2c + 1)
    const int sr0 = 2 * (lane & 3), sr1 = sr0 + 1;
    const int spos0 = L - Q + min(sr0 / p.group, Q - 1), spos1 = L - Q + min(sr1 / p.group, Q - 1);
    const int slo0 = p.window_left >= 0 ? max(0, spos0 - p.window_left) : 0;
    const int slo1 = p.window_left >= 0 ? max(0, spos1 - p.window_left) : 0;

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int it = 0; it < n_tiles; ++it) {
        cp_async_wait<kDecStages - 2>();
        key_group_sync<MT>(kg);  // the slice landed; the group is done with the stage reloaded next
        {
            int nxt = it + kDecStages - 1;
            if (nxt < n_tiles) load_tile(nxt % kDecStages, k_tile0 + nxt * kDecTile);
            cp_async_commit();
        }
        const int stage = it % kDecStages;
        const int j0 = k_tile0 + it * kDecTile;
        const uint32_t kb = smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t vb = kb + kDecTileBytes;
        const uint8_t *k8 = smem + stage * STAGE_BYTES;  // E4M3 K rows (KV8)
        const uint8_t *v8 = k8 + kDec8TileBytes;         // E4M3 V rows (KV8)

        if constexpr (SW) {
            // Swapped operands for at most 8 query rows: S^T (the warp's 16
            // keys x 8 rows) = K Q^T and O^T (128 dims x 8 rows) += V^T P^T,
            // so that the keys fill the MMA's 16-row side and half as many
            // MMAs cover a tile.  Lane (g, c) = (lane / 4, lane % 4) holds
            // the scores of keys kw0 + g and kw0 + g + 8 for query rows 2c
            // and 2c + 1; rows at or beyond R are padding, masked out.
            const int g = lane >> 2, c = lane & 3;
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};  // even / odd k-steps
            {
                // A = K rows kw0 + g and kw0 + g + 8: the word at byte
                // 32c + 4kk of a row holds dims 32c + 4kk .. + 3, both halves
                // of the lane's A fragment of k-step kk (the permuted order
                // the Q fragments follow)
                const uint4 u0 = *reinterpret_cast<const uint4 *>(k8 + swz8(kw0 + g, 2 * c));
                const uint4 u1 = *reinterpret_cast<const uint4 *>(k8 + swz8(kw0 + g, 2 * c + 1));
                const uint4 v0 = *reinterpret_cast<const uint4 *>(k8 + swz8(kw0 + g + 8, 2 * c));
                const uint4 v1 = *reinterpret_cast<const uint4 *>(k8 + swz8(kw0 + g + 8, 2 * c + 1));
                const uint32_t wa[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
                const uint32_t wb[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t a[4] = {widen_e4m3x2<TM>(wa[kk] & 0xffffu), widen_e4m3x2<TM>(wb[kk] & 0xffffu),
                                           widen_e4m3x2<TM>(wa[kk] >> 16), widen_e4m3x2<TM>(wb[kk] >> 16)};
                    if (kk & 1)
                        mma16816<TM>(sb, a, qa[kk][0], qa[kk][1]);
                    else
                        mma16816<TM>(sa, a, qa[kk][0], qa[kk][1]);
                }
            }
            // element e: key kw0 + g + 8 (e / 2), query row 2c + (e % 2)
            float sv[4];
            const bool interior = !any_bad[kg] && j0 >= lo_max && j0 + kDecTile - 1 <= hi_min;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = (sa[e] + sb[e]) * scale_log2;
                const int jj = kw0 + g + 8 * (e >> 1), j = j0 + jj;
                bool vis = (e & 1 ? sr1 : sr0) < R;
                if (!interior)
                    vis = vis && kvalid[stage * kDecTile + jj] &&
                          (e & 1 ? (j >= slo1 && j <= spos1) : (j >= slo0 && j <= spos0));
                sv[e] = vis ? x : -INFINITY;
            }
            // row maxima over the warp's 16 keys (the lanes of one c)
            float mx0 = fmaxf(sv[0], sv[2]), mx1 = fmaxf(sv[1], sv[3]);
#pragma unroll
            for (int o_ = 4; o_ < 32; o_ <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o_));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o_));
            }
            const float mn0 = mx0 > m0 + 8.f ? mx0 : m0, mn1 = mx1 > m1 + 8.f ? mx1 : m1;
            const float base0 = mn0 == -INFINITY ? 0.f : mn0;
            const float base1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = fast_exp2(m0 - base0), al1 = fast_exp2(m1 - base1);
            const float p0 = fast_exp2(sv[0] - base0), p1 = fast_exp2(sv[1] - base1);
            const float p2 = fast_exp2(sv[2] - base0), p3 = fast_exp2(sv[3] - base1);
            l0 = l0 * al0 + (p0 + p2);  // (this lane's keys; summed over g at the end)
            l1 = l1 * al1 + (p1 + p3);
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[i][0] *= al0;
                    o[i][2] *= al0;
                    o[i][1] *= al1;
                    o[i][3] *= al1;
                }
            }
            // B = P^T (k = the warp's 16 keys, n = query row): lane (g, c)
            // needs row g's P of keys 2c, 2c + 1, 2c + 8, 2c + 9, held by
            // lanes (2c, g / 2) and (2c + 1, g / 2) as their row-2c' or
            // row-2c'+1 pair
            const uint32_t he = pack2<TM>(p0, p2), ho = pack2<TM>(p1, p3);
            const int srcA = 8 * c + (g >> 1), srcB = srcA + 4;
            const uint32_t eA = __shfl_sync(0xffffffffu, he, srcA), oA = __shfl_sync(0xffffffffu, ho, srcA);
            const uint32_t eB = __shfl_sync(0xffffffffu, he, srcB), oB = __shfl_sync(0xffffffffu, ho, srcB);
            const uint32_t vA = (g & 1) ? oA : eA, vB = (g & 1) ? oB : eB;
            const uint32_t pb0 = __byte_perm(vA, vB, 0x5410), pb1 = __byte_perm(vA, vB, 0x7632);
            // A = V^T (m = head dim, k = key) of m-tile i: its row m is dim
            // 16 (m % 8) + 2i + m / 8, so that a lane's 16 dims of a V row are
            // one 16-byte chunk (g) and the two keys of an A register are
            // byte-interleaved from two rows
            const uint4 x0 = *reinterpret_cast<const uint4 *>(v8 + swz8(kw0 + 2 * c, g));
            const uint4 x1 = *reinterpret_cast<const uint4 *>(v8 + swz8(kw0 + 2 * c + 1, g));
            const uint4 y0 = *reinterpret_cast<const uint4 *>(v8 + swz8(kw0 + 2 * c + 8, g));
            const uint4 y1 = *reinterpret_cast<const uint4 *>(v8 + swz8(kw0 + 2 * c + 9, g));
            const uint32_t X0[4] = {x0.x, x0.y, x0.z, x0.w}, X1[4] = {x1.x, x1.y, x1.z, x1.w};
            const uint32_t Y0[4] = {y0.x, y0.y, y0.z, y0.w}, Y1[4] = {y1.x, y1.y, y1.z, y1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t x01 = __byte_perm(X0[i], X1[i], 0x5140), x23 = __byte_perm(X0[i], X1[i], 0x7362);
                const uint32_t y01 = __byte_perm(Y0[i], Y1[i], 0x5140), y23 = __byte_perm(Y0[i], Y1[i], 0x7362);
                const uint32_t a0[4] = {widen_e4m3x2<TM>(x01 & 0xffffu), widen_e4m3x2<TM>(x01 >> 16),
                                        widen_e4m3x2<TM>(y01 & 0xffffu), widen_e4m3x2<TM>(y01 >> 16)};
                const uint32_t a1[4] = {widen_e4m3x2<TM>(x23 & 0xffffu), widen_e4m3x2<TM>(x23 >> 16),
                                        widen_e4m3x2<TM>(y23 & 0xffffu), widen_e4m3x2<TM>(y23 >> 16)};
                mma16816<TM>(o[2 * i], a0, pb0, pb1);
                mma16816<TM>(o[2 * i + 1], a1, pb0, pb1);
            }
        } else {
            float sc[NT][4];
#pragma unroll
            for (int i = 0; i < NT; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
            if constexpr (KV8) {
                // key kw0 + 8nt + g: its 32 bytes at dims 32c .. 32c + 31 hold the
                // B fragments of all eight k-steps (see the Q fragments)
                const int g8 = lane >> 2, c8 = lane & 3;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int row = kw0 + nt * 8 + g8;
                    const uint4 u0 = *reinterpret_cast<const uint4 *>(k8 + swz8(row, 2 * c8));
                    const uint4 u1 = *reinterpret_cast<const uint4 *>(k8 + swz8(row, 2 * c8 + 1));
                    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma16816<TM>(sc[nt], qa[kk], widen_e4m3x2<TM>(w[kk] & 0xffffu), widen_e4m3x2<TM>(w[kk] >> 16));
                }
            } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
                for (int np = 0; np < NT / 2; ++np) {
                    uint32_t bf[4];
                    int key = kw0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                    ldsm_x4(bf, kb + swz(key, 2 * kk + ((lane >> 3) & 1), kDecRowBytes));
                    mma16816<TM>(sc[2 * np], qa[kk], bf[0], bf[1]);
                    mma16816<TM>(sc[2 * np + 1], qa[kk], bf[2], bf[3]);
                }
            }
            }

            const bool interior = !any_bad[kg] && j0 >= lo_max && j0 + kDecTile - 1 <= hi_min;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float x = sc[nt][e] * scale_log2;
                    if (!interior) {
                        int jj = kw0 + nt * 8 + 2 * (lane & 3) + (e & 1);
                        int j = j0 + jj;
                        bool vis = kvalid[stage * kDecTile + jj] &&
                                   (e < 2 ? (j >= lo0 && j <= pos0) : (j >= lo1 && j <= pos1));
                        if (!vis) x = -INFINITY;
                    }
                    sc[nt][e] = x;
                }
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
                mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            // the running max rises only when a tile's exceeds it by more than 8
            // (a factor 2^8; from -inf at the first key): P stays below 2^8 and
            // O is rarely rescaled
            const float mn0 = mx0 > m0 + 8.f ? mx0 : m0, mn1 = mx1 > m1 + 8.f ? mx1 : m1;
            const float base0 = mn0 == -INFINITY ? 0.f : mn0;
            const float base1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = fast_exp2(m0 - base0), al1 = fast_exp2(m1 - base1);
            float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                sc[nt][0] = fast_exp2(sc[nt][0] - base0);
                sc[nt][1] = fast_exp2(sc[nt][1] - base0);
                sc[nt][2] = fast_exp2(sc[nt][2] - base1);
                sc[nt][3] = fast_exp2(sc[nt][3] - base1);
                rs0 += sc[nt][0] + sc[nt][1];
                rs1 += sc[nt][2] + sc[nt][3];
            }
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
            m0 = mn0;
            m1 = mn1;
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    o[i][0] *= al0;
                    o[i][1] *= al0;
                    o[i][2] *= al1;
                    o[i][3] *= al1;
                }
            }
#pragma unroll
            for (int ks = 0; ks < NT / 2; ++ks) {
                uint32_t a[4];
                a[0] = pack2<TM>(sc[2 * ks][0], sc[2 * ks][1]);
                a[1] = pack2<TM>(sc[2 * ks][2], sc[2 * ks][3]);
                a[2] = pack2<TM>(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
                a[3] = pack2<TM>(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
                if constexpr (KV8) {
                    // The output dims are permuted too: column g of n-tile nt is
                    // dim 16g + nt, so the lane's 16 bytes of the keys 2c, 2c+1,
                    // 2c+8, 2c+9 feed all 16 n-tiles, the two keys of a B
                    // register interleaved byte by byte.
                    const int g8 = lane >> 2, rb = kw0 + ks * 16 + 2 * (lane & 3);
                    const uint4 x0 = *reinterpret_cast<const uint4 *>(v8 + swz8(rb, g8));
                    const uint4 x1 = *reinterpret_cast<const uint4 *>(v8 + swz8(rb + 1, g8));
                    const uint4 y0 = *reinterpret_cast<const uint4 *>(v8 + swz8(rb + 8, g8));
                    const uint4 y1 = *reinterpret_cast<const uint4 *>(v8 + swz8(rb + 9, g8));
                    const uint32_t X0[4] = {x0.x, x0.y, x0.z, x0.w}, X1[4] = {x1.x, x1.y, x1.z, x1.w};
                    const uint32_t Y0[4] = {y0.x, y0.y, y0.z, y0.w}, Y1[4] = {y1.x, y1.y, y1.z, y1.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t p01 = __byte_perm(X0[i], X1[i], 0x5140), p23 = __byte_perm(X0[i], X1[i], 0x7362);
                        const uint32_t q01 = __byte_perm(Y0[i], Y1[i], 0x5140), q23 = __byte_perm(Y0[i], Y1[i], 0x7362);
                        mma16816<TM>(o[4 * i], a, widen_e4m3x2<TM>(p01 & 0xffffu), widen_e4m3x2<TM>(q01 & 0xffffu));
                        mma16816<TM>(o[4 * i + 1], a, widen_e4m3x2<TM>(p01 >> 16), widen_e4m3x2<TM>(q01 >> 16));
                        mma16816<TM>(o[4 * i + 2], a, widen_e4m3x2<TM>(p23 & 0xffffu), widen_e4m3x2<TM>(q23 & 0xffffu));
                        mma16816<TM>(o[4 * i + 3], a, widen_e4m3x2<TM>(p23 >> 16), widen_e4m3x2<TM>(q23 >> 16));
                    }
                } else {
                    const int key = kw0 + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
                    for (int dp = 0; dp < 8; ++dp) {
                        uint32_t vf[4];
                        ldsm_x4_t(vf, vb + swz(key, 2 * dp + (lane >> 4), kDecRowBytes));
                        mma16816<TM>(o[2 * dp], a, vf[0], vf[1]);
                        mma16816<TM>(o[2 * dp + 1], a, vf[2], vf[3]);
                    }
                }
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    pdl_launch_dependents();  // the merge kernel may get ready; it waits for this grid

    // combine the key groups of this CTA through shared memory
    if constexpr (SW) {  // a row's keys are spread over the lanes of one c
#pragma unroll
        for (int o_ = 4; o_ < 32; o_ <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o_);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o_);
        }
    } else {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    }
    float *comb_o = reinterpret_cast<float *>(smem);  // [NKG][ROWS][128]
    if constexpr (SW) {
        // lane (g, c) holds rows 2c and 2c + 1 at dims 16g .. 16g + 15:
        // o[i][0 / 1] at dim 16g + 2i, o[i][2 / 3] at dim 16g + 2i + 1
        const int g = lane >> 2;
        float *w0 = &comb_o[(kg * ROWS + sr0) * kDecD + 16 * g];
        float *w1 = &comb_o[(kg * ROWS + sr1) * kDecD + 16 * g];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            *reinterpret_cast<float4 *>(w0 + 4 * q) =
                make_float4(o[2 * q][0], o[2 * q][2], o[2 * q + 1][0], o[2 * q + 1][2]);
            *reinterpret_cast<float4 *>(w1 + 4 * q) =
                make_float4(o[2 * q][1], o[2 * q][3], o[2 * q + 1][1], o[2 * q + 1][3]);
        }
        if (g == 0) {
            comb_m[kg * ROWS + sr0] = m0;
            comb_l[kg * ROWS + sr0] = l0;
            comb_m[kg * ROWS + sr1] = m1;
            comb_l[kg * ROWS + sr1] = l1;
        }
    } else if constexpr (KV8) {
        // undo the output permutation: o[nt][e] is dim 16 (2c + (e & 1)) + nt
        const int d0 = 32 * (lane & 3);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float *w0 = &comb_o[(kg * ROWS + r0) * kDecD + d0 + 4 * i];
            float *w1 = &comb_o[(kg * ROWS + r1) * kDecD + d0 + 4 * i];
            *reinterpret_cast<float4 *>(w0) = make_float4(o[4 * i][0], o[4 * i + 1][0], o[4 * i + 2][0], o[4 * i + 3][0]);
            *reinterpret_cast<float4 *>(w0 + 16) = make_float4(o[4 * i][1], o[4 * i + 1][1], o[4 * i + 2][1], o[4 * i + 3][1]);
            *reinterpret_cast<float4 *>(w1) = make_float4(o[4 * i][2], o[4 * i + 1][2], o[4 * i + 2][2], o[4 * i + 3][2]);
            *reinterpret_cast<float4 *>(w1 + 16) = make_float4(o[4 * i][3], o[4 * i + 1][3], o[4 * i + 2][3], o[4 * i + 3][3]);
        }
    } else {
#pragma unroll
        for (int nd = 0; nd < 16; ++nd) {
            int d = nd * 8 + 2 * (lane & 3);
            *reinterpret_cast<float2 *>(&comb_o[(kg * ROWS + r0) * kDecD + d]) = make_float2(o[nd][0], o[nd][1]);
            *reinterpret_cast<float2 *>(&comb_o[(kg * ROWS + r1) * kDecD + d]) = make_float2(o[nd][2], o[nd][3]);
        }
    }
    if (!SW && (lane & 3) == 0) {
        comb_m[kg * ROWS + r0] = m0;
        comb_l[kg * ROWS + r0] = l0;
        comb_m[kg * ROWS + r1] = m1;
        comb_l[kg * ROWS + r1] = l1;
    }
    __syncthreads();

    for (int idx = tid; idx < R * 32; idx += kDecThreads) {
        const int r = idx >> 5, d = (idx & 31) * 4;
        float M = -INFINITY;
#pragma unroll
        for (int g = 0; g < NKG; ++g) M = fmaxf(M, comb_m[g * ROWS + r]);
        const float Mb = M == -INFINITY ? 0.f : M;
        float lsum = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int g = 0; g < NKG; ++g) {
            float w = fast_exp2(comb_m[g * ROWS + r] - Mb);
            lsum += w * comb_l[g * ROWS + r];
            float4 x = *reinterpret_cast<const float4 *>(&comb_o[(g * ROWS + r) * kDecD + d]);
            a0 += w * x.x;
            a1 += w * x.y;
            a2 += w * x.z;
            a3 += w * x.w;
        }
        const int t = r / p.group, i = r - t * p.group, h = kvh * p.group + i;
        if (n_split == 1) {
            float sc_o, lse_v;
            if (p.sinks) {
                const float sk = p.sinks[h] * kLog2e;
                const float Mf = fmaxf(M, sk);
                const float wk = fast_exp2(M - Mf);
                const float den = lsum * wk + fast_exp2(sk - Mf);
                sc_o = bmm2 * wk / den;
                lse_v = (Mf + fast_log2(den)) * kLn2;
            } else if (lsum > 0.f) {
                sc_o = bmm2 / lsum;
                lse_v = (M + fast_log2(lsum)) * kLn2;
            } else {
                sc_o = 0.f;
                lse_v = -INFINITY;
            }
            const int64_t orow = (qrow0 + t) * p.Hqo + h;
            if (dbg_in(orow * kDecD + d, 4, p.num_tokens * p.Hqo * kDecD, p.err))
                store4(static_cast<T *>(p.out) + orow * kDecD + d, a0 * sc_o, a1 * sc_o, a2 * sc_o, a3 * sc_o);
            if (p.lse && d == 0) p.lse[orow] = lse_v;
        } else {
            const int64_t prow =
                (static_cast<int64_t>(b * p.Hkv + kvh) * p.n_split_max + s) * p.R + r;
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            if (dbg_in(prow, 1, p.ws_rows, p.err)) {
                *reinterpret_cast<float4 *>(p.ws_o + prow * kDecD + d) =
                    make_float4(a0 * inv, a1 * inv, a2 * inv, a3 * inv);
                if (d == 0) p.ws_lse[prow] = lsum > 0.f ? M + fast_log2(lsum) : -INFINITY;
            }
        }
    }
}

// One warp per output row (b*Q + t, h): weights the split partials by
// 2^lse_s, adds the sink to the denominator, applies bmm2_scale.
template <typename T>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
    pdl_wait();  // the split kernel's partials
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + warp;
    if (row >= static_cast<int64_t>(p.B) * p.Q * p.Hqo) return;
    const int h = static_cast<int>(row % p.Hqo);
    const int64_t bq = row / p.Hqo;
    const int t = static_cast<int>(bq % p.Q), b = static_cast<int>(bq / p.Q);
    int Q = p.Q;
    int64_t qrow0 = static_cast<int64_t>(b) * p.Q;
    if (p.cu_q) {  // the split kernel flagged inconsistent entries; skip them the same way
        const int c0 = p.cu_q[b], c1 = p.cu_q[b + 1];
        Q = c1 - c0;
        qrow0 = c0;
        if (c0 < 0 || Q < 0 || Q > p.Q || c1 > p.num_tokens) Q = 0;
    }
    if (t >= Q) return;
    const uint32_t L_in = p.seq_lens[b];
    const int L = L_in > static_cast<uint32_t>(p.max_seq_len) ? p.max_seq_len : static_cast<int>(L_in);
    int lo, first, n_split;
    decode_split_geometry(L, Q, p.window_left, p.chunk, lo, first, n_split);
    if (n_split <= 1) return;  // the split kernel wrote this row itself
    const int kvh = h / p.group;
    const int r = t * p.group + (h - kvh * p.group);
    const int64_t base = static_cast<int64_t>(b * p.Hkv + kvh) * p.n_split_max * p.R + r;
    float M = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
    if (!dbg_in(base, static_cast<int64_t>(n_split - 1) * p.R + 1, p.ws_rows, p.err) ||
        !dbg_in(n_split, 0, p.n_split_max, p.err))
        return;
    for (int s = 0; s < n_split; ++s) M = fmaxf(M, p.ws_lse[base + static_cast<int64_t>(s) * p.R]);
    const int d = lane * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n_split; ++s) {
            const int64_t prow = base + static_cast<int64_t>(s) * p.R;
            const float w = fast_exp2(p.ws_lse[prow] - M);
            const float4 x = *reinterpret_cast<const float4 *>(p.ws_o + prow * kDecD + d);
            den += w;
            acc.x += w * x.x;
            acc.y += w * x.y;
            acc.z += w * x.z;
            acc.w += w * x.w;
        }
        if (p.sinks) den += fast_exp2(p.sinks[h] * kLog2e - M);
    }
    const float bmm2 = p.bmm2_dev ? __ldg(p.bmm2_dev) : p.bmm2;
    const float sc = den > 0.f ? bmm2 / den : 0.f;
    const int64_t orow = (qrow0 + t) * p.Hqo + h;
    if (!dbg_in(orow * kDecD + d, 4, p.num_tokens * p.Hqo * kDecD, p.err)) return;
    store4(static_cast<T *>(p.out) + orow * kDecD + d, acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
    if (p.lse && lane == 0) p.lse[orow] = den > 0.f ? (M + fast_log2(den)) * kLn2 : -INFINITY;
}

struct DecodePlan {
    int R, MT, chunk, n_split_max;
    size_t ws_o_bytes, ws_bytes;
};

static int plan_decode(int B, int Q, int Hqo, int Hkv, int D, int max_seq_len, int page_size,
                       int window_left, DecodePlan &pl, bool kv8 = false) {
    if (B < 0 || Q < 1 || Hqo < 1 || Hkv < 1 || max_seq_len < 0 || window_left < -1)
        return PKV_ERR_INVALID_ARG;
    if (Hqo % Hkv) return PKV_ERR_INVALID_ARG;
    if (B > 65535 || Hkv > 65535) return PKV_ERR_UNSUPPORTED;
    if (D != kDecD) return PKV_ERR_UNSUPPORTED;
    if (ilog2_exact(page_size) < 0 || page_size < kDecMinPage || page_size > 256) return PKV_ERR_UNSUPPORTED;
    const int group = Hqo / Hkv;
    pl.R = group * Q;
    if (pl.R > 64) return PKV_ERR_UNSUPPORTED;
    pl.MT = pl.R <= 16 ? 1 : (pl.R <= 32 ? 2 : 4);
    const int64_t span = window_left >= 0
                             ? (static_cast<int64_t>(window_left) + Q < max_seq_len
                                    ? static_cast<int64_t>(window_left) + Q
                                    : max_seq_len)
                             : max_seq_len;
    // Larger row groups write larger partials: scale the chunk with R so the
    // partial traffic stays a few percent of the K/V bytes; then shrink it
    // while the grid would leave SMs idle.
    int chunk = 128 * pl.R;
    chunk = chunk < 1024 ? 1024 : (chunk > 4096 ? 4096 : chunk);
    // an E4M3 cache moves half the bytes per key: twice the keys per split
    // keep the per-CTA set-up and partial traffic at the same share
    if (kv8) chunk = 2 * chunk > 4096 ? 4096 : 2 * chunk;
    chunk = (chunk + kDecTile - 1) / kDecTile * kDecTile;
    // a window a little longer than the chunk (its first key need not sit on
    // a tile edge: up to 63 keys more) takes one split rather than a second,
    // nearly empty one
    const int64_t span_t = window_left >= 0 ? span + kDecTile - 1 : span;
    if (window_left >= 0 && span_t > chunk && span_t <= chunk + chunk / 4 && span_t <= kDecMaxChunk)
        chunk = static_cast<int>((span_t + kDecTile - 1) / kDecTile * kDecTile);
    const int64_t want = 2LL * num_sms();
    while (chunk > 4 * kDecTile &&
           static_cast<int64_t>(B) * Hkv * ((span + chunk - 1) / chunk) < want)
        chunk = (chunk / 2 + kDecTile - 1) / kDecTile * kDecTile;  // (tile multiples)
    pl.chunk = chunk;
    int64_t ns = span > 0 ? (span_t + chunk - 1) / chunk : 1;
    if (ns > 65535) return PKV_ERR_UNSUPPORTED;
    pl.n_split_max = static_cast<int>(ns);
    if (pl.n_split_max > 1) {
        const size_t slots = static_cast<size_t>(B) * Hkv * pl.n_split_max * pl.R;
        pl.ws_o_bytes = round_up(slots * kDecD * sizeof(float), 256);
        pl.ws_bytes = pl.ws_o_bytes + round_up(slots * sizeof(float), 256);
    } else {
        pl.ws_o_bytes = pl.ws_bytes = 0;
    }
    return PKV_OK;
}

template <typename T, int MT, int LAYOUT, bool KV8, bool SW = false>
static int launch_split(const DecodeParams &p, dim3 grid, cudaStream_t st, bool pdl) {
    constexpr int ROWS = 16 * MT, NKG = 4 / MT;
    constexpr int kDecStages = DecCfg<MT, KV8>::STAGES;
    const size_t smem = kDecStages * DecSmem<KV8>::STAGE + ROWS * kDecRowBytes +
                        kDecStages * kDecTile + 2 * NKG * ROWS * sizeof(float) + kDecMaxPages * sizeof(int);
    auto kern = decode_split_kernel<T, MT, LAYOUT, KV8, SW>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (pdl) return launch_dependent(kern, grid, dim3(kDecThreads), smem, st, p) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
    kern<<<grid, kDecThreads, smem, st>>>(p);
    return PKV_OK;
}

template <typename T, int LAYOUT, bool KV8>
static int launch_split_mt(int MT, const DecodeParams &p, dim3 grid, cudaStream_t st, bool pdl) {
    if constexpr (KV8) {
        if (p.R <= 8) return launch_split<T, 1, LAYOUT, true, true>(p, grid, st, pdl);  // swapped operands
    }
    if (MT == 1) return launch_split<T, 1, LAYOUT, KV8>(p, grid, st, pdl);
    if (MT == 2) return launch_split<T, 2, LAYOUT, KV8>(p, grid, st, pdl);
    return launch_split<T, 4, LAYOUT, KV8>(p, grid, st, pdl);
}

template <typename T>
static int run_decode(const DecodeParams &p, const DecodePlan &pl, int layout, bool kv8, bool pdl,
                      cudaStream_t st) {
    dim3 grid(pl.n_split_max, p.Hkv, p.B);
    int rc = kv8 ? (layout == PKV_HND ? launch_split_mt<T, PKV_HND, true>(pl.MT, p, grid, st, pdl)
                                      : launch_split_mt<T, PKV_NHD, true>(pl.MT, p, grid, st, pdl))
                 : (layout == PKV_HND ? launch_split_mt<T, PKV_HND, false>(pl.MT, p, grid, st, pdl)
                                      : launch_split_mt<T, PKV_NHD, false>(pl.MT, p, grid, st, pdl));
    if (rc != PKV_OK) return rc;
    int launches = 1;
    if (pl.n_split_max > 1) {
        int64_t rows = static_cast<int64_t>(p.B) * p.Q * p.Hqo;
        if (launch_dependent(decode_merge_kernel<T>, dim3(static_cast<unsigned>((rows + 3) / 4)), dim3(128), 0,
                             st, p) != cudaSuccess)
            return PKV_ERR_CUDA;
        ++launches;
    }
    note_launches(launches);
    return launch_status();
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t paged_decode_workspace_size(int32_t batch_size, int32_t q_len_per_req,
                                              int32_t num_qo_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t max_seq_len,
                                              int32_t page_size, int32_t window_left) {
    DecodePlan pl;
    if (plan_decode(batch_size, q_len_per_req, num_qo_heads, num_kv_heads, head_dim, max_seq_len,
                    page_size, window_left, pl) != PKV_OK)
        return 0;
    return pl.ws_bytes;
}

static int decode_impl(const void *query, const void *k_cache, const void *v_cache,
                            int64_t page_stride, int64_t max_num_pages, void *workspace,
                            size_t workspace_bytes, const int32_t *block_tables,
                            int32_t block_table_stride, const uint32_t *seq_lens,
                            int32_t batch_size, int32_t max_seq_len, float bmm1_scale,
                            float bmm2_scale, int32_t window_left, const float *sinks,
                            int32_t q_len_per_req, const int32_t *cum_seq_lens_q, int64_t num_tokens,
                            int32_t num_qo_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t page_size, int32_t layout, int32_t dtype,
                            void *out, float *lse, int32_t *err_word, void *stream,
                            const float *bmm1_dev = nullptr, const float *bmm2_dev = nullptr,
                            bool enable_pdl = false) {
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16 && dtype != PKV_F16_E4M3 && dtype != PKV_BF16_E4M3)
        return PKV_ERR_INVALID_ARG;
    const bool kv8 = dtype == PKV_F16_E4M3 || dtype == PKV_BF16_E4M3;  // 8-bit cache, 16-bit query/out
    const bool bf16 = dtype == PKV_BF16 || dtype == PKV_BF16_E4M3;
    DecodePlan pl;
    int rc = plan_decode(batch_size, q_len_per_req, num_qo_heads, num_kv_heads, head_dim,
                         max_seq_len, page_size, window_left, pl);
    if (rc != PKV_OK) return rc;
    if (kv8) {
        // the E4M3 plan's longer splits, whenever they fit the workspace that
        // paged_decode_workspace_size (which knows no element type) sized
        DecodePlan p8;
        if (plan_decode(batch_size, q_len_per_req, num_qo_heads, num_kv_heads, head_dim, max_seq_len,
                        page_size, window_left, p8, true) == PKV_OK &&
            p8.ws_bytes <= pl.ws_bytes)
            pl = p8;
    }
    if (page_stride < static_cast<int64_t>(num_kv_heads) * page_size * head_dim || max_num_pages < 0 ||
        static_cast<int64_t>(block_table_stride) * page_size < max_seq_len)
        return PKV_ERR_INVALID_ARG;
    if (batch_size == 0) return PKV_OK;
    if (!query || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return PKV_ERR_NULL;
    if (!aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (page_stride % (kv8 ? 16 : 8)))  // 16-byte page starts
        return PKV_ERR_INVALID_ARG;
    if (pl.ws_bytes > 0) {
        if (!workspace) return PKV_ERR_NULL;
        if (workspace_bytes < pl.ws_bytes || (reinterpret_cast<uintptr_t>(workspace) & 255))
            return PKV_ERR_WORKSPACE;
    }
    DecodeParams p;
    p.q = query;
    p.k = k_cache;
    p.v = v_cache;
    p.page_stride = page_stride;
    p.max_num_pages = max_num_pages;
    p.block_tables = block_tables;
    p.bt_stride = block_table_stride;
    p.seq_lens = seq_lens;
    p.B = batch_size;
    p.max_seq_len = max_seq_len;
    p.scale_log2 = bmm1_scale * kLog2e;
    p.bmm2 = bmm2_scale;
    p.bmm1_dev = bmm1_dev;
    p.bmm2_dev = bmm2_dev;
    p.window_left = window_left;
    p.sinks = sinks;
    p.Q = q_len_per_req;
    p.cu_q = cum_seq_lens_q;
    p.num_tokens = num_tokens;
    p.kv_extent = max_num_pages > 0 ? (max_num_pages - 1) * page_stride +
                                          static_cast<int64_t>(num_kv_heads) * page_size * head_dim
                                    : 0;
    p.ws_rows = static_cast<int64_t>(batch_size) * num_kv_heads * pl.n_split_max * pl.R;
    p.Hqo = num_qo_heads;
    p.Hkv = num_kv_heads;
    p.group = num_qo_heads / num_kv_heads;
    p.R = pl.R;
    p.page_shift = ilog2_exact(page_size);
    p.chunk = pl.chunk;
    p.n_split_max = pl.n_split_max;
    p.out = out;
    p.lse = lse;
    p.ws_o = pl.ws_bytes ? static_cast<float *>(workspace) : nullptr;
    p.ws_lse = pl.ws_bytes ? reinterpret_cast<float *>(static_cast<char *>(workspace) + pl.ws_o_bytes)
                           : nullptr;
    p.err = err_word;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return bf16 ? run_decode<__nv_bfloat16>(p, pl, layout, kv8, enable_pdl, st)
                : run_decode<__half>(p, pl, layout, kv8, enable_pdl, st);
}

extern "C" int paged_decode(const void *query, const void *k_cache, const void *v_cache,
                            int64_t page_stride, int64_t max_num_pages, void *workspace,
                            size_t workspace_bytes, const int32_t *block_tables,
                            int32_t block_table_stride, const uint32_t *seq_lens,
                            int32_t batch_size, int32_t max_seq_len, float bmm1_scale,
                            float bmm2_scale, int32_t window_left, const float *sinks,
                            int32_t q_len_per_req, int32_t num_qo_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t page_size, int32_t layout, int32_t dtype,
                            void *out, float *lse, int32_t *err_word, void *stream) {
    const CallRange nvtx_range("paged_decode");
    return decode_impl(query, k_cache, v_cache, page_stride, max_num_pages, workspace, workspace_bytes,
                       block_tables, block_table_stride, seq_lens, batch_size, max_seq_len, bmm1_scale,
                       bmm2_scale, window_left, sinks, q_len_per_req, nullptr,
                       static_cast<int64_t>(batch_size) * q_len_per_req, num_qo_heads, num_kv_heads, head_dim,
                       page_size, layout, dtype, out, lse, err_word, stream);
}

extern "C" int paged_decode_varlen(const void *query, int64_t num_tokens, const void *k_cache,
                                   const void *v_cache, int64_t page_stride, int64_t max_num_pages,
                                   void *workspace, size_t workspace_bytes, const int32_t *block_tables,
                                   int32_t block_table_stride, const uint32_t *seq_lens, int32_t batch_size,
                                   int32_t max_seq_len, float bmm1_scale, float bmm2_scale,
                                   int32_t window_left, const float *sinks, int32_t max_q_len,
                                   const int32_t *cum_seq_lens_q, int32_t num_qo_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t page_size, int32_t layout, int32_t dtype,
                                   void *out, float *lse, int32_t *err_word, void *stream) {
    const CallRange nvtx_range("paged_decode_varlen");
    if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (batch_size > 0 && num_tokens > 0 && !cum_seq_lens_q) return PKV_ERR_NULL;
    if (num_tokens == 0) return PKV_OK;
    return decode_impl(query, k_cache, v_cache, page_stride, max_num_pages, workspace, workspace_bytes,
                       block_tables, block_table_stride, seq_lens, batch_size, max_seq_len, bmm1_scale,
                       bmm2_scale, window_left, sinks, max_q_len, cum_seq_lens_q, num_tokens, num_qo_heads,
                       num_kv_heads, head_dim, page_size, layout, dtype, out, lse, err_word, stream);
}

extern "C" int paged_decode_ex(const void *query, int64_t num_tokens, const void *k_cache,
                               const void *v_cache, int64_t page_stride, int64_t max_num_pages,
                               void *workspace, size_t workspace_bytes, const int32_t *block_tables,
                               int32_t block_table_stride, const uint32_t *seq_lens, int32_t batch_size,
                               int32_t max_seq_len, float bmm1_scale, float bmm2_scale,
                               const float *bmm1_scale_dev, const float *bmm2_scale_dev, int32_t window_left,
                               const float *sinks, int32_t max_q_len, const int32_t *cum_seq_lens_q,
                               int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                               int32_t layout, int32_t dtype, int32_t enable_pdl, void *out, float *lse,
                               int32_t *err_word, void *stream) {
    const CallRange nvtx_range("paged_decode_ex");
    if (num_tokens < 0 || max_q_len < 1) return PKV_ERR_INVALID_ARG;
    if (!cum_seq_lens_q && num_tokens < static_cast<int64_t>(batch_size) * max_q_len) return PKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PKV_OK;
    return decode_impl(query, k_cache, v_cache, page_stride, max_num_pages, workspace, workspace_bytes,
                       block_tables, block_table_stride, seq_lens, batch_size, max_seq_len, bmm1_scale,
                       bmm2_scale, window_left, sinks, max_q_len, cum_seq_lens_q,
                       cum_seq_lens_q ? num_tokens : static_cast<int64_t>(batch_size) * max_q_len, num_qo_heads,
                       num_kv_heads, head_dim, page_size, layout, dtype, out, lse, err_word, stream,
                       bmm1_scale_dev, bmm2_scale_dev, enable_pdl != 0);
}

// ---- decode with a library-owned scratch array ------------------------------
//
// For callers that cannot allocate device memory where they call decode: a
// plugin running inside another runtime's execution step (that runtime owns
// the device memory and forbids allocation there), a latency-critical loop
// that cannot afford cudaMalloc's implicit device-wide synchronisation, or
// a process that reserves all device memory up front.  The split partials
// live in a fixed array in this library's own device image instead of a
// caller workspace.
#include <cudaTypedefs.h>

#include <mutex>

namespace pkv {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES);
constexpr int kNoAllocCachedContexts = 64;

// One copy per device that loads the library, held until the process exits.
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

// Unique id of the calling thread's current CUDA context (driver entry points
// fetched through the runtime: the library does not link libcuda).  False
// when no context is current yet.
static bool current_context_id(unsigned long long *id) {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_decode_scratch in the current context.  In host code
// the symbol is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress and cached per CUDA context, keyed by the context's
// unique id: after a device reset (or under another context of the same
// device) the library's module is loaded again and the array may move; the
// new context has a new id, so its address is looked up afresh.
static void *noalloc_scratch_ptr() {
    static std::mutex mu;
    static unsigned long long ids[kNoAllocCachedContexts];
    static void *ptrs[kNoAllocCachedContexts];
    static int used = 0, next = 0;
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(mu);
    if (have_id)
        for (int i = 0; i < used; ++i)
            if (ids[i] == id) return ptrs[i];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return nullptr;
    // (the lookup above made the primary context current if none was)
    if (!have_id && !current_context_id(&id)) return p;  // not cached: looked up again next call
    const int slot = used < kNoAllocCachedContexts ? used++ : (next++ % kNoAllocCachedContexts);
    ids[slot] = id;
    ptrs[slot] = p;
    return p;
}

}  // namespace pkv

extern "C" int paged_decode_noalloc(const void *query, const void *k_cache, const void *v_cache,
                                    int64_t page_stride, int64_t max_num_pages,
                                    const int32_t *block_tables, int32_t block_table_stride,
                                    const uint32_t *seq_lens, int32_t batch_size,
                                    int32_t max_seq_len, float bmm1_scale, float bmm2_scale,
                                    int32_t window_left, const float *sinks,
                                    int32_t q_len_per_req, int32_t num_qo_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                    int32_t layout, int32_t dtype, void *out, float *lse,
                                    int32_t *err_word, void *stream) {
    const CallRange nvtx_range("paged_decode_noalloc");
    DecodePlan pl;
    int rc = plan_decode(batch_size, q_len_per_req, num_qo_heads, num_kv_heads, head_dim,
                         max_seq_len, page_size, window_left, pl);
    if (rc != PKV_OK) return rc;
    if (pl.ws_bytes > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (pl.ws_bytes > 0) {
        scratch = noalloc_scratch_ptr();
        if (!scratch) return PKV_ERR_CUDA;
    }
    return paged_decode(query, k_cache, v_cache, page_stride, max_num_pages, scratch,
                        scratch ? kNoAllocScratchBytes : 0, block_tables, block_table_stride,
                        seq_lens, batch_size, max_seq_len, bmm1_scale, bmm2_scale, window_left,
                        sinks, q_len_per_req, num_qo_heads, num_kv_heads, head_dim, page_size,
                        layout, dtype, out, lse, err_word, stream);
}
