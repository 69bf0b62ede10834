// prefill.cu -- causal ragged batch prefill over a paged KV cache, with LSE.
//
// Computes what flashinfer.prefill.cudnn_batch_prefill_with_kv_cache
// documents (q, k_cache, v_cache, scale, workspace_buffer,
// max_token_per_sequence, max_sequence_kv, actual_seq_lens_q/kv,
// block_tables, causal, return_lse): queries of request b are the last
// q_b of its kv_b positions; each CTA owns 128 query rows of one qo head and
// streams the keys it can see through a cp.async ring, with an online
// softmax in registers.
#include <math.h>

#include "pkv_common.cuh"

namespace pkv {

constexpr int kPfRows = 128;   // query rows per CTA (8 warps x 16)
constexpr int kPfTile = 64;    // keys per pipeline stage
constexpr int kPfStages = 2;
constexpr int kPfThreads = 256;
constexpr int kPfDV = 128;

struct PrefillParams {
    const void *q;
    const void *k;
    const void *v;
    int64_t k_page_stride, v_page_stride, max_num_pages;
    float scale_log2;
    const int32_t *seq_lens_q;
    const int32_t *seq_lens_kv;
    const int32_t *cu_q;  // [B+1] in the workspace
    const int32_t *block_tables;
    int64_t bt_stride;
    int B, causal, Hqo, Hkv, group, page_shift, max_q, max_kv;
    void *out;
    float *lse;
    int32_t *err;
};

// cu_q = exclusive prefix sum of the query lengths (one warp, 32 at a time);
// flags requests with fewer keys than queries.
__global__ void prefill_plan_kernel(const int32_t *__restrict__ lq, const int32_t *__restrict__ lkv,
                                    int B, int max_q, int max_kv, int32_t *__restrict__ cu_q,
                                    int32_t *err) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        int b = b0 + lane;
        int v = b < B ? lq[b] : 0;
        if (b < B && (v > max_q || v < 0 || lkv[b] > max_kv)) set_err(err, PKV_DEV_ERR_LEN);
        v = min(max(v, 0), max_q);
        if (b < B && min(lkv[b], max_kv) < v) set_err(err, PKV_DEV_ERR_QLEN);
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (b < B) cu_q[b] = carry + x - v;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) cu_q[B] = carry;
}

template <typename T, int DQK, int LAYOUT>
__global__ void __launch_bounds__(kPfThreads, 1) prefill_mma_kernel(const PrefillParams p) {
    constexpr int KROW = DQK * 2, VROW = kPfDV * 2;
    constexpr int KCH = DQK / 8, VCH = kPfDV / 8;  // 16-byte chunks per row
    constexpr int KTILE = kPfTile * KROW, VTILE = kPfTile * VROW;
    constexpr int STAGE = KTILE + VTILE;
    constexpr int NT = kPfTile / 8;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *q_s = smem + kPfStages * STAGE;
    uint8_t *kvalid = q_s + kPfRows * KROW;
    __shared__ int any_bad;

    const int b = blockIdx.z, h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qb = min(max(p.seq_lens_q[b], 0), p.max_q);
    const int kvb = min(max(p.seq_lens_kv[b], 0), p.max_kv);
    const int n_qt = (qb + kPfRows - 1) / kPfRows;
    if (static_cast<int>(blockIdx.x) >= n_qt) return;
    const int qt = n_qt - 1 - blockIdx.x;  // most keys first
    const int i0 = qt * kPfRows;
    const int row_base = p.cu_q[b] + i0;
    const int kvh = h / p.group;
    const int shift = kvb - qb;  // position of query i is shift + i
    int k_hi = p.causal ? min(kvb, shift + i0 + kPfRows) : kvb;
    if (k_hi < 0) k_hi = 0;
    const int n_tiles = (k_hi + kPfTile - 1) / kPfTile;

    const T *kc = static_cast<const T *>(p.k);
    const T *vc = static_cast<const T *>(p.v);
    const int32_t *bt = p.block_tables + static_cast<int64_t>(b) * p.bt_stride;
    const int S = 1 << p.page_shift;
    if (tid == 0) any_bad = 0;
    __syncthreads();

    auto load_tile = [&](int stage, int j0) {
        uint8_t *base = smem + stage * STAGE;
        for (int idx = tid; idx < kPfTile * (KCH + VCH); idx += kPfThreads) {
            const bool is_v = idx >= kPfTile * KCH;
            const int li = is_v ? idx - kPfTile * KCH : idx;
            const int nch = is_v ? VCH : KCH;
            const int r = li / nch, c = li - r * nch;
            const int j = j0 + r;
            bool ok = j < k_hi;
            const T *src = kc;
            if (ok) {
                int page = bt[j >> p.page_shift];
                if (page < 0 || page >= p.max_num_pages) {
                    ok = false;
                    if (c == 0 && !is_v) {
                        set_err(p.err, PKV_DEV_ERR_PAGE);
                        any_bad = 1;
                    }
                } else if (is_v) {
                    src = vc + kv_row_offset<LAYOUT>(page, p.v_page_stride, kvh, j & (S - 1), p.Hkv,
                                                     S, kPfDV) + c * 8;
                } else {
                    src = kc + kv_row_offset<LAYOUT>(page, p.k_page_stride, kvh, j & (S - 1), p.Hkv,
                                                     S, DQK) + c * 8;
                }
            }
            if (!is_v && c == 0) kvalid[stage * kPfTile + r] = ok ? 1 : 0;
            uint32_t dst = smem_u32(base + (is_v ? KTILE : 0)) + swz(r, c, is_v ? VROW : KROW);
            cp_async_16(dst, src, ok);
        }
    };

    const T *qp = static_cast<const T *>(p.q);
    for (int idx = tid; idx < kPfRows * KCH; idx += kPfThreads) {
        const int r = idx / KCH, c = idx - r * KCH;
        const bool ok = i0 + r < qb;
        const T *src = ok ? qp + (static_cast<int64_t>(row_base + r) * p.Hqo + h) * DQK + c * 8 : qp;
        cp_async_16(smem_u32(q_s) + swz(r, c, KROW), src, ok);
    }
    cp_async_commit();
#pragma unroll
    for (int st = 0; st < kPfStages - 1; ++st) {
        if (st < n_tiles) load_tile(st, st * kPfTile);
        cp_async_commit();
    }
    cp_async_wait<kPfStages - 1>();
    __syncthreads();

    uint32_t qa[DQK / 16][4];
#pragma unroll
    for (int kk = 0; kk < DQK / 16; ++kk)
        ldsm_x4(qa[kk], smem_u32(q_s) + swz(16 * warp + (lane & 15), 2 * kk + (lane >> 4), KROW));

    const int ra = 16 * warp + (lane >> 2), rb = ra + 8;  // rows of this lane (tile-local)
    const int posa = shift + i0 + ra, posb = shift + i0 + rb;
    const int lim_a = p.causal ? min(posa, kvb - 1) : kvb - 1;  // last visible key
    const int lim_b = p.causal ? min(posb, kvb - 1) : kvb - 1;
    // last key visible to the warp's first / last row (warp-uniform)
    const int warp_lim_lo = p.causal ? min(shift + i0 + 16 * warp, kvb - 1) : kvb - 1;
    const int warp_lim_hi = p.causal ? min(shift + i0 + 16 * warp + 15, kvb - 1) : kvb - 1;

    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int it = 0; it < n_tiles; ++it) {
        cp_async_wait<kPfStages - 2>();
        __syncthreads();
        {
            int nxt = it + kPfStages - 1;
            if (nxt < n_tiles) load_tile(nxt % kPfStages, nxt * kPfTile);
            cp_async_commit();
        }
        const int stage = it % kPfStages;
        const int j0 = it * kPfTile;
        const uint32_t kb = smem_u32(smem + stage * STAGE);
        const uint32_t vb = kb + KTILE;
        if (j0 > warp_lim_hi) continue;  // no key of this tile is visible to this warp

        float sc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t bf[4];
                int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
                ldsm_x4(bf, kb + swz(key, 2 * kk + ((lane >> 3) & 1), KROW));
                mma16816<T>(sc[2 * np], qa[kk], bf[0], bf[1]);
                mma16816<T>(sc[2 * np + 1], qa[kk], bf[2], bf[3]);
            }
        }
        const bool interior = !any_bad && j0 + kPfTile - 1 <= warp_lim_lo;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = sc[nt][e] * p.scale_log2;
                if (!interior) {
                    int jj = nt * 8 + 2 * (lane & 3) + (e & 1);
                    int j = j0 + jj;
                    bool vis = kvalid[stage * kPfTile + jj] && j <= (e < 2 ? lim_a : lim_b);
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
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
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
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al0;
            o[i][2] *= al1;
            o[i][3] *= al1;
        }
#pragma unroll
        for (int ks = 0; ks < NT / 2; ++ks) {
            uint32_t a[4];
            a[0] = pack2<T>(sc[2 * ks][0], sc[2 * ks][1]);
            a[1] = pack2<T>(sc[2 * ks][2], sc[2 * ks][3]);
            a[2] = pack2<T>(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
            a[3] = pack2<T>(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
            const int key = ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                uint32_t vf[4];
                ldsm_x4_t(vf, vb + swz(key, 2 * dp + (lane >> 4), VROW));
                mma16816<T>(o[2 * dp], a, vf[0], vf[1]);
                mma16816<T>(o[2 * dp + 1], a, vf[2], vf[3]);
            }
        }
    }
    cp_async_wait<0>();

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
    T *outp = static_cast<T *>(p.out);
    const bool va = i0 + ra < qb, vb_ = i0 + rb < qb;
    const int64_t orow_a = static_cast<int64_t>(row_base + ra) * p.Hqo + h;
    const int64_t orow_b = static_cast<int64_t>(row_base + rb) * p.Hqo + h;
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) {
        const int d = nd * 8 + 2 * (lane & 3);
        if (va) *reinterpret_cast<uint32_t *>(outp + orow_a * kPfDV + d) = pack2<T>(o[nd][0] * inv0, o[nd][1] * inv0);
        if (vb_) *reinterpret_cast<uint32_t *>(outp + orow_b * kPfDV + d) = pack2<T>(o[nd][2] * inv1, o[nd][3] * inv1);
    }
    if ((lane & 3) == 0) {
        if (va) p.lse[orow_a] = l0 > 0.f ? (m0 + fast_log2(l0)) * kLn2 : -INFINITY;
        if (vb_) p.lse[orow_b] = l1 > 0.f ? (m1 + fast_log2(l1)) * kLn2 : -INFINITY;
    }
}

template <typename T, int DQK, int LAYOUT>
static int launch_prefill(const PrefillParams &p, dim3 grid, cudaStream_t st) {
    const size_t smem = kPfStages * (kPfTile * DQK * 2 + kPfTile * kPfDV * 2) + kPfRows * DQK * 2 +
                        kPfStages * kPfTile;
    auto kern = prefill_mma_kernel<T, DQK, LAYOUT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PKV_ERR_CUDA;
    kern<<<grid, kPfThreads, smem, st>>>(p);
    return PKV_OK;
}

template <typename T>
static int dispatch_prefill(int d_qk, int layout, const PrefillParams &p, dim3 grid, cudaStream_t st) {
    if (d_qk == 128)
        return layout == PKV_HND ? launch_prefill<T, 128, PKV_HND>(p, grid, st)
                                 : launch_prefill<T, 128, PKV_NHD>(p, grid, st);
    return layout == PKV_HND ? launch_prefill<T, 192, PKV_HND>(p, grid, st)
                             : launch_prefill<T, 192, PKV_NHD>(p, grid, st);
}

static size_t prefill_ws_bytes(int B) { return round_up(static_cast<size_t>(B + 1) * sizeof(int32_t), 256); }

}  // namespace pkv

using namespace pkv;

extern "C" size_t paged_prefill_workspace_size(int32_t batch_size, int32_t num_qo_heads,
                                               int32_t max_token_per_sequence,
                                               int32_t max_sequence_kv) {
    if (batch_size < 0 || num_qo_heads < 1 || max_token_per_sequence < 0 || max_sequence_kv < 0)
        return 0;
    return prefill_ws_bytes(batch_size);
}

extern "C" int paged_prefill(const void *q, const void *k_cache, const void *v_cache,
                             int64_t k_page_stride, int64_t v_page_stride, int64_t max_num_pages,
                             float scale, void *workspace, size_t workspace_bytes,
                             int32_t max_token_per_sequence, int32_t max_sequence_kv,
                             const int32_t *actual_seq_lens_q, const int32_t *actual_seq_lens_kv,
                             const int32_t *block_tables, int32_t block_table_stride,
                             int32_t batch_size, int32_t causal, int32_t num_qo_heads,
                             int32_t num_kv_heads, int32_t d_qk, int32_t d_vo, int32_t page_size,
                             int32_t layout, int32_t dtype, void *out, float *lse,
                             int32_t *err_word, void *stream) {
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (batch_size < 0 || num_qo_heads < 1 || num_kv_heads < 1 || max_token_per_sequence < 0 ||
        max_sequence_kv < 0 || max_num_pages < 0 || block_table_stride < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_qo_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
    if ((d_qk != 128 && d_qk != 192) || d_vo != 128) return PKV_ERR_UNSUPPORTED;
    if (ilog2_exact(page_size) < 0 || page_size > 1024) return PKV_ERR_UNSUPPORTED;
    if (batch_size > 65535 || num_qo_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if (k_page_stride < static_cast<int64_t>(num_kv_heads) * page_size * d_qk ||
        v_page_stride < static_cast<int64_t>(num_kv_heads) * page_size * d_vo ||
        static_cast<int64_t>(block_table_stride) * page_size < max_sequence_kv)
        return PKV_ERR_INVALID_ARG;
    if (batch_size == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !actual_seq_lens_q || !actual_seq_lens_kv || !block_tables ||
        !out || !lse)
        return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (k_page_stride % 8) || (v_page_stride % 8))
        return PKV_ERR_INVALID_ARG;
    if (!workspace) return PKV_ERR_NULL;
    if (workspace_bytes < prefill_ws_bytes(batch_size) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return PKV_ERR_WORKSPACE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *cu_q = static_cast<int32_t *>(workspace);
    prefill_plan_kernel<<<1, 32, 0, st>>>(actual_seq_lens_q, actual_seq_lens_kv, batch_size,
                                          max_token_per_sequence, max_sequence_kv, cu_q, err_word);
    PrefillParams p;
    p.q = q;
    p.k = k_cache;
    p.v = v_cache;
    p.k_page_stride = k_page_stride;
    p.v_page_stride = v_page_stride;
    p.max_num_pages = max_num_pages;
    p.scale_log2 = scale * kLog2e;
    p.seq_lens_q = actual_seq_lens_q;
    p.seq_lens_kv = actual_seq_lens_kv;
    p.cu_q = cu_q;
    p.block_tables = block_tables;
    p.bt_stride = block_table_stride;
    p.B = batch_size;
    p.causal = causal ? 1 : 0;
    p.Hqo = num_qo_heads;
    p.Hkv = num_kv_heads;
    p.group = num_qo_heads / num_kv_heads;
    p.page_shift = ilog2_exact(page_size);
    p.max_q = max_token_per_sequence;
    p.max_kv = max_sequence_kv;
    p.out = out;
    p.lse = lse;
    p.err = err_word;
    const int n_qt = (max_token_per_sequence + kPfRows - 1) / kPfRows;
    int launches = 1;
    if (n_qt > 0) {
        dim3 grid(n_qt, num_qo_heads, batch_size);
        int rc = dtype == PKV_BF16 ? dispatch_prefill<__nv_bfloat16>(d_qk, layout, p, grid, st)
                                   : dispatch_prefill<__half>(d_qk, layout, p, grid, st);
        if (rc != PKV_OK) return rc;
        ++launches;
    }
    note_launches(launches);
    return launch_status();
}
