// prefill.cu -- causal ragged batch prefill over a paged KV cache, with LSE.
//
// Computes what flashinfer.prefill.cudnn_batch_prefill_with_kv_cache
// documents (q, k_cache, v_cache, scale, workspace_buffer,
// max_token_per_sequence, max_sequence_kv, actual_seq_lens_q/kv,
// block_tables, causal, return_lse): the queries of request b are the last
// q_b of its kv_b positions; softmax(scale q k^T) v over the visible keys
// and the natural-log LSE of the scaled logits.
//
// A persistent CTA per SM takes work items -- 128 query rows of one qo head
// -- from a global counter (heaviest first) and walks the key tiles each can
// see; the pipelines run on across items.  Warp roles (352 threads):
//   warps 8, 10  TMA producers: Q once and the K tiles (warp 8), the V tiles
//           (warp 10), 128 keys page by page, through separate K and V rings
//           of shared-memory stages;
//   warp 9  allocates tensor memory and issues the tcgen05 MMAs from one
//           thread: S = Q K^T into one of two TMEM score buffers (so the
//           next tile's QK overlaps this tile's softmax), then per group
//           O_g += P_g V_g with P read from TMEM;
//   warps 0-7  two groups of four warps, one thread per query row each;
//           group g owns keys [64g, 64g+64) of every tile: read its S
//           columns from TMEM, mask, online softmax in base 2, write P
//           (bf16/fp16) over the consumed S columns as the A operand of its
//           PV MMA, which accumulates into the group's own O in TMEM
//           (rescaled there when the running max grows by more than 2^8).
//           At the end the two partial (O, max, sum) are merged, normalised
//           and written with the LSE.
// Every wait is bounded; a wait that gives up sets PKV_DEV_ERR_TIMEOUT, the
// other roles stop, tensor memory is freed and the CTA returns.
#include <math.h>

#include "pkv_common.cuh"
#include "sm103_ptx.cuh"

namespace pkv {

constexpr int kPfRows = 128;     // query rows per CTA
constexpr int kPfThreads = 352;  // 8 softmax warps + K-load warp + MMA warp + V-load warp
constexpr int kTmaWarp = 8, kMmaWarp = 9, kTmaVWarp = 10;
constexpr int kPfDV = 128;

// Key tiles of BN = 128; separate K and V rings (a K stage is released by
// its QK, a V stage by its PV).
template <int DQK>
struct PfCfg;
template <>
struct PfCfg<128> {
    static constexpr int SK = 3, SV = 2;
};
template <>
struct PfCfg<192> {
    static constexpr int SK = 2, SV = 2;
};
constexpr int kPfBN = 128;

struct PrefillParams {
    int64_t max_num_pages;
    int64_t total_q;
    float scale_log2;
    const int32_t *seq_lens_q;
    const int32_t *seq_lens_kv;
    const int32_t *cu_q;  // [B+1] in the workspace
    const int32_t *block_tables;
    int64_t bt_stride;
    int B, causal, Hqo, Hkv, group, page_shift, max_q, max_kv, n_qt_max;
    int *work_counter;  // in the workspace, zeroed by the plan kernel
    void *out;
    float *lse;
    int32_t *err;
};

// cu_q = exclusive prefix sum of the query lengths (one warp, 32 at a time);
// flags lengths above their maxima and requests with fewer keys than queries.
__global__ void prefill_plan_kernel(const int32_t *__restrict__ lq, const int32_t *__restrict__ lkv,
                                    int B, int max_q, int max_kv, int32_t *__restrict__ cu_q,
                                    int32_t *err, int *work_counter) {
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
    if (lane == 0) {
        cu_q[B] = carry;
        *work_counter = 0;
    }
}


// 2^x on the FMA pipe, for part of the softmax exponentials (the rest use
// the special-function unit): x = n + f with n = round(x) taken from the
// low mantissa bits of x + 1.5*2^23, f in [-1/2, 1/2]; 2^f from the degree-4
// polynomial interpolating 2^f at the Chebyshev nodes of [-1/2, 1/2]
// (coefficients from exp2_poly_fit.py beside this file, max relative error
// 3.6e-6); 2^n added to the exponent bits.  x = -inf (a masked key) gives 0.
__device__ __forceinline__ float exp2_fma(float x) {
    const float xc = fmaxf(x, -126.f);
    const float t = xc + 12582912.f;
    const float f = xc - (t - 12582912.f);
    float q = fmaf(9.666368365e-03f, f, 5.592197552e-02f);
    q = fmaf(q, f, 2.402234972e-01f);
    q = fmaf(q, f, 6.931210160e-01f);
    q = fmaf(q, f, 1.0f);
    const float r = __int_as_float(__float_as_int(q) + (__float_as_int(t) << 23));
    return x < -126.f ? 0.f : r;
}

// Share of the softmax exponentials computed by exp2_fma (one pair in
// kExpFmaEvery; 0 = none).  Measured on GB300 with the ragged-prefill
// workload: the special-function unit is not the bottleneck of this kernel,
// and moving work to the FMA pipe costs issue slots, so it is off.
constexpr int kExpFmaEvery = 0;

template <typename T>
struct IsBf16 {
    static constexpr bool value = false;
};
template <>
struct IsBf16<__nv_bfloat16> {
    static constexpr bool value = true;
};

// One query tile of one qo head of one request: the unit of work of the
// persistent kernel.  Items are numbered x-major, x = 0 being the LAST query
// tile of a request (the one that sees the most keys), so taking items in
// order hands out the heaviest tiles first.
struct PfItem {
    int b, h, i0, row_base, kvh, shift, qb, kvb, n_tiles;
};

__device__ __forceinline__ bool pf_item(const PrefillParams &p, int idx, PfItem &it) {
    const int per_x = p.Hqo * p.B;
    const int x = idx / per_x, rem = idx - x * per_x;
    it.h = rem % p.Hqo;
    it.b = rem / p.Hqo;
    it.qb = min(max(p.seq_lens_q[it.b], 0), p.max_q);
    it.kvb = min(max(p.seq_lens_kv[it.b], 0), p.max_kv);
    const int n_qt = (it.qb + kPfRows - 1) / kPfRows;
    if (x >= n_qt) return false;
    it.i0 = (n_qt - 1 - x) * kPfRows;
    it.row_base = p.cu_q[it.b] + it.i0;
    it.kvh = it.h / p.group;
    it.shift = it.kvb - it.qb;  // query i sits at position shift + i
    int k_hi = p.causal ? min(it.kvb, it.shift + it.i0 + kPfRows) : it.kvb;
    if (k_hi < 0) k_hi = 0;
    it.n_tiles = (k_hi + kPfBN - 1) / kPfBN;
    return true;
}

template <typename T, int DQK, int LAYOUT>
__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    constexpr int BN = kPfBN;
    constexpr int SK = PfCfg<DQK>::SK, SV = PfCfg<DQK>::SV;
    constexpr int QA = DQK / 64;                 // 64-column atoms of a Q / K row
    constexpr uint32_t QB = kPfRows * DQK * 2;   // bytes of the Q tile
    constexpr uint32_t KB = BN * DQK * 2;        // bytes of one K stage
    constexpr uint32_t VB = BN * kPfDV * 2;      // bytes of one V stage
    constexpr int NI = 2;                        // slots of the work-item ring
    // TMEM columns: O of group 0 and 1, then the two S buffers; P of a tile
    // (16-bit pairs, BN/2 columns) overwrites the first half of its S buffer
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t S_COL = 2 * kPfDV;
    static_assert(S_COL + 2 * BN <= TMEM_COLS, "TMEM budget");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t q_s = smem_u32(smem);
    const uint32_t k_s = q_s + QB;
    const uint32_t v_s = k_s + SK * KB;
    const uint32_t bar0 = v_s + SV * VB;
    uint8_t *v_gen = smem + QB + SK * KB;  // generic pointer to the V stages
    // barriers
    uint32_t nb = 0;
    const uint32_t b_qfull = bar0 + 8u * nb++;   // Q of the current item landed
    const uint32_t b_qempty = bar0 + 8u * nb++;  // last QK of an item done: Q buffer free
    const uint32_t b_ofree = bar0 + 8u * nb++;   // epilogue read O: accumulators free
    const uint32_t b_xchg = bar0 + 8u * nb++;    // both groups posted (max, sum)
    const uint32_t b_item_full0 = bar0 + 8u * nb; nb += NI;
    const uint32_t b_item_empty0 = bar0 + 8u * nb; nb += NI;
    const uint32_t b_kfull0 = bar0 + 8u * nb; nb += SK;
    const uint32_t b_kempty0 = bar0 + 8u * nb; nb += SK;
    const uint32_t b_vfull0 = bar0 + 8u * nb; nb += SV;
    const uint32_t b_vempty0 = bar0 + 8u * nb; nb += SV;
    const uint32_t b_sfull0 = bar0 + 8u * nb; nb += 2;
    const uint32_t b_pfull0 = bar0 + 8u * nb; nb += 4;  // [S buffer][group]
    const uint32_t b_pvdone0 = bar0 + 8u * nb; nb += 4;  // [S buffer][group]
    auto b_item_full = [&](int i) { return b_item_full0 + 8u * i; };
    auto b_item_empty = [&](int i) { return b_item_empty0 + 8u * i; };
    auto b_kfull = [&](int s) { return b_kfull0 + 8u * s; };
    auto b_kempty = [&](int s) { return b_kempty0 + 8u * s; };
    auto b_vfull = [&](int s) { return b_vfull0 + 8u * s; };
    auto b_vempty = [&](int s) { return b_vempty0 + 8u * s; };
    auto b_sfull = [&](int i) { return b_sfull0 + 8u * i; };
    // P of tile t written by group g, and PV of tile t for group g done: one
    // barrier per S buffer, so that every wait is for the newest phase that
    // can be pending.  A wait for tile t's phase finds tile t-2's complete
    // (S_t is written after PV_{t-2}) and tile t+2's impossible (QK_{t+2}
    // is issued after PV_t, which needs P_t), so parity cannot alias.
    auto b_pfull = [&](int t, int g) { return b_pfull0 + 8u * (2 * (t & 1) + g); };
    auto b_pvdone = [&](int t, int g) { return b_pvdone0 + 8u * (2 * (t & 1) + g); };
    static_assert(SV == 2, "the V tail wait relies on PV_{t-2} having waited for V_{t-2}");
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ int item_ring[NI];
    __shared__ float xchg[2][2][2][kPfRows];  // [item parity][max|sum][group][row]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total_items = p.n_qt_max * p.Hqo * p.B;

    if (tid == 0) {
        mbar_init(b_qfull, 1);
        mbar_init(b_qempty, 1);
        mbar_init(b_ofree, 256);
        mbar_init(b_xchg, 256);
        for (int i = 0; i < NI; ++i) {
            mbar_init(b_item_full(i), 1);
            mbar_init(b_item_empty(i), 2 + 256);  // MMA thread, V producer, 256 softmax threads
        }
        for (int s = 0; s < SK; ++s) {
            mbar_init(b_kfull(s), 1);
            mbar_init(b_kempty(s), 1);
        }
        for (int s = 0; s < SV; ++s) {
            mbar_init(b_vfull(s), 1);
            mbar_init(b_vempty(s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(b_sfull(i), 1);
            mbar_init(b_pfull(i, 0), 128);
            mbar_init(b_pfull(i, 1), 128);
            mbar_init(b_pvdone(i, 0), 1);
            mbar_init(b_pvdone(i, 1), 1);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&tmem_base_s), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    volatile int *abort_flag = &abort_s;
    auto give_up = [&]() {
        *abort_flag = 1;
        set_err(p.err, PKV_DEV_ERR_TIMEOUT);
    };
    // the k-th item published by the K producer (-1: no more work); every
    // consumer role takes every item, in order, and releases the ring slot
    auto take_item = [&](int k, bool &ok) -> int {
        const int slot = k % NI;
        if (!mbar_wait(b_item_full(slot), (k / NI) & 1, abort_flag)) {
            ok = false;
            return -1;
        }
        const int idx = *reinterpret_cast<volatile int *>(&item_ring[slot]);
        mbar_arrive(b_item_empty(slot));
        return idx;
    };

    if (warp == kTmaWarp || warp == kTmaVWarp) {
        // ------------------------------------------------------------ TMA producers
        // Warp 8 takes work items from the global counter, publishes them,
        // and loads Q and the K tiles; warp 10 loads the V tiles.  A K stage
        // is released by its QK and a V stage by its (later) PV, so the rings
        // advance independently.  Both warps look up a tile's page ids in one
        // coalesced load, one tile ahead; lane 0 issues the copies.
        const bool is_k = warp == kTmaWarp;
        if (lane == 0) {
            if (is_k) {
                prefetch_tmap(&tm_q);
                prefetch_tmap(&tm_k);
            } else {
                prefetch_tmap(&tm_v);
            }
        }
        const int S = 1 << p.page_shift;
        const int RB = S < BN ? S : BN;  // rows per TMA box
        const int nbox = BN / RB;       // boxes (pages or page parts) per tile, <= 16
        const int oob = static_cast<int>(p.max_num_pages);  // page coordinate past the pool: zero fill
        const int NS = is_k ? SK : SV;
        bool ok = true;
        int t_base = 0;  // tiles of earlier items (global tile counter)
        for (int k = 0; ok; ++k) {
            int idx;
            if (is_k) {
                // fetch the next valid item and publish it
                idx = -1;
                if (lane == 0) {
                    while (true) {
                        const int c = atomicAdd(p.work_counter, 1);
                        if (c >= total_items) break;
                        PfItem tmp;
                        if (pf_item(p, c, tmp)) {
                            idx = c;
                            break;
                        }
                    }
                    const int slot = k % NI;
                    if (k >= NI && !mbar_wait(b_item_empty(slot), ((k / NI) - 1) & 1, abort_flag)) {
                        give_up();
                        ok = false;
                    } else {
                        item_ring[slot] = idx;
                        mbar_arrive(b_item_full(slot));
                    }
                }
                idx = __shfl_sync(0xffffffffu, idx, 0);
                ok = __shfl_sync(0xffffffffu, ok, 0);
            } else {
                if (lane == 0) idx = take_item(k, ok);
                idx = __shfl_sync(0xffffffffu, idx, 0);
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
            if (!ok || idx < 0) break;
            PfItem it;
            pf_item(p, idx, it);
            const int32_t *bt = p.block_tables + static_cast<int64_t>(it.b) * p.bt_stride;
            // Q of this item, once the previous item's last QK is done; it is
            // loaded after the item's first K tile so that the two overlap
            auto load_q = [&]() {  // lane 0 of the K producer
                if (k >= 1 && !mbar_wait(b_qempty, (k - 1) & 1, abort_flag)) {
                    give_up();
                    ok = false;
                } else {
                    mbar_expect_tx(b_qfull, QB);
                    for (int c = 0; c < QA; ++c)
                        tma_load_3d(q_s + c * (kPfRows * 128), &tm_q, b_qfull, c * 64, it.h, it.row_base);
                }
            };
            if (is_k && lane == 0 && it.n_tiles == 0) load_q();
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            auto lookup = [&](int j) {  // lane i < nbox: page of box i of tile j
                const int key = j * BN + lane * RB;
                int page = oob;
                if (lane < nbox && key < it.kvb) {
                    page = bt[key >> p.page_shift];
                    if (page < 0 || page >= p.max_num_pages) {
                        if (is_k) set_err(p.err, PKV_DEV_ERR_PAGE);
                        page = oob;
                    }
                }
                return page;
            };
            int pg_next = it.n_tiles > 0 ? lookup(0) : oob;
            for (int j = 0; j < it.n_tiles; ++j) {
                const int t = t_base + j;
                const int pg = pg_next;
                if (j + 1 < it.n_tiles) pg_next = lookup(j + 1);
                int pages[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pages[i] = __shfl_sync(0xffffffffu, pg, i);
                if (lane == 0) {
                    const int st = t % NS, us = t / NS;
                    if (us > 0 && !mbar_wait(is_k ? b_kempty(st) : b_vempty(st), (us - 1) & 1, abort_flag)) {
                        give_up();
                        ok = false;
                    } else {
                        const uint32_t full = is_k ? b_kfull(st) : b_vfull(st);
                        mbar_expect_tx(full, is_k ? KB : VB);
                        const int j0 = j * BN;
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (i >= nbox) break;
                            const int r0 = i * RB;
                            const int slot0 = (j0 + r0) & (S - 1);
                            const int ca = LAYOUT == PKV_HND ? slot0 : it.kvh;
                            const int cb = LAYOUT == PKV_HND ? it.kvh : slot0;
                            if (is_k) {
                                for (int c = 0; c < QA; ++c)
                                    tma_load_4d(k_s + st * KB + c * (BN * 128) + r0 * 128, &tm_k, full, c * 64, ca,
                                                cb, pages[i]);
                            } else {
                                for (int c = 0; c < kPfDV / 64; ++c)
                                    tma_load_4d(v_s + st * VB + c * (BN * 128) + r0 * 128, &tm_v, full, c * 64, ca,
                                                cb, pages[i]);
                            }
                        }
                        if (is_k && j == 0) load_q();
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
            t_base += it.n_tiles;
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // Per item: QK_0, then for every tile j: QK_{j+1}, PV_{j,0}, PV_{j,1}.
        // QK_{j+1} runs on the tensor core while the softmax works on S_j.
        // tcgen05 MMAs execute in issue order, so a QK that overwrites an S
        // buffer cannot disturb the PV still reading P from it.
        if (lane == 0) {
            constexpr uint32_t idesc_qk = umma_idesc(kPfRows, BN, IsBf16<T>::value, false);
            constexpr uint32_t idesc_pv = umma_idesc(kPfRows, kPfDV, IsBf16<T>::value, true);
            const uint64_t qdesc0 = umma_sdesc_sw128(q_s, 16, 1024);
            const uint64_t kdesc0 = umma_sdesc_sw128(k_s, 16, 1024);
            const uint64_t vdesc0 = umma_sdesc_sw128(v_s, BN * 128, 1024);
            bool ok = true;
            int t_base = 0;
            int n_tiled = 0;  // items with at least one key tile so far (o_free phases)
            auto issue_qk = [&](int t) -> bool {
                const int sk = t % SK, uk = t / SK;
                if (!mbar_wait(b_kfull(sk), uk & 1, abort_flag)) return false;
                tc_fence_after();
                const uint64_t kd = kdesc0 + ((sk * KB) >> 4);
#pragma unroll
                for (int kk = 0; kk < DQK / 16; ++kk)
                    umma_ss(tmem + S_COL + (t & 1) * BN,
                            qdesc0 + (((kk >> 2) * (kPfRows * 128) + (kk & 3) * 32) >> 4),
                            kd + (((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4), idesc_qk, kk > 0 ? 1u : 0u);
                umma_commit(b_sfull(t & 1));
                umma_commit(b_kempty(sk));
                return true;
            };
            auto issue_pv = [&](int t, bool first) -> bool {
                const int sv = t % SV, uv = t / SV;
                const uint64_t vd = vdesc0 + ((sv * VB) >> 4);
                for (int hh = 0; hh < 2; ++hh) {
                    if (!mbar_wait(b_pfull(t, hh), (t >> 1) & 1, abort_flag)) return false;
                    if (hh == 0 && !mbar_wait(b_vfull(sv), uv & 1, abort_flag)) return false;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < BN / 32; ++kk)
                        umma_ts(tmem + hh * kPfDV, tmem + S_COL + (t & 1) * BN + hh * (BN / 2) + kk * 8,
                                vd + (((hh * (BN / 2) + kk * 16) * 128) >> 4), idesc_pv,
                                (!first || kk > 0) ? 1u : 0u);
                    umma_commit(b_pvdone(t, hh));
                }
                umma_commit(b_vempty(sv));
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int idx = take_item(k, ok);
                if (!ok || idx < 0) break;
                PfItem it;
                pf_item(p, idx, it);
                if (!mbar_wait(b_qfull, k & 1, abort_flag)) { ok = false; break; }
                if (it.n_tiles > 0) ok = issue_qk(t_base);
                if (ok && it.n_tiles == 1) umma_commit(b_qempty);
                for (int j = 0; ok && j < it.n_tiles; ++j) {
                    if (j + 1 < it.n_tiles) {
                        if (!issue_qk(t_base + j + 1)) { ok = false; break; }
                        if (j + 2 == it.n_tiles) umma_commit(b_qempty);  // last QK of the item issued
                    }
                    // the epilogue of the previous item with tiles must have
                    // read O before this item's first PV overwrites it
                    if (j == 0 && n_tiled >= 1 && !mbar_wait(b_ofree, (n_tiled - 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (!issue_pv(t_base + j, j == 0)) { ok = false; break; }
                }
                if (ok && it.n_tiles == 0) umma_commit(b_qempty);
                t_base += it.n_tiles;
                n_tiled += it.n_tiles > 0;
            }
            if (!ok) give_up();
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        // Two groups of four warps split every key tile by columns: group g
        // owns keys [64g, 64g+64) of each tile and keeps its own running max,
        // sum and O accumulator (TMEM columns g*128 ..), so the groups never
        // exchange anything inside the tile loop.  Warp w owns TMEM lanes /
        // query rows 32*(w%4) .. +31, one thread per (row, group).  The two
        // partial results of an item are merged in its epilogue.
        constexpr int HC = BN / 2;  // S columns per thread
        const int g = warp >> 2;
        const int r = 32 * (warp & 3) + lane;  // query row of this thread inside the tile
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
        const uint32_t o_g = g * kPfDV;  // this group's O columns
        auto wait_warp = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
        };
        bool ok = true;
        int t_base = 0;
        for (int k = 0; ok; ++k) {
            int idx = take_item(k, ok);
            ok = __all_sync(0xffffffffu, ok);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            if (!ok || idx < 0) break;
            PfItem it;
            pf_item(p, idx, it);
            const int pos = it.shift + it.i0 + r;
            const int lim = p.causal ? min(pos, it.kvb - 1) : it.kvb - 1;  // last visible key
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < it.n_tiles; ++j) {
                const int t = t_base + j;
                const int j0 = j * BN + g * HC;  // first key of this thread's columns
                const uint32_t t_s = t_lane + S_COL + (t & 1) * BN + g * HC;
                // S_t complete; by commit order so is PV_{t-2}, the last reader
                // of the P columns about to be rewritten
                if (!wait_warp(b_sfull(t & 1), (t >> 1) & 1)) { ok = false; break; }
                tc_fence_after();
                uint32_t sx[HC];
#pragma unroll
                for (int c = 0; c < HC / 32; ++c)
                    tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sx + c * 32));
                tmem_wait_ld();
                const bool full = j0 + HC - 1 <= lim;
                // row max: on the raw scores when the scale is positive (then
                // max(scale * s) = scale * max(s) and one FFMA per element
                // later does both the scaling and the shift), else scaled
                const float sc = p.scale_log2;
                const bool pos_scale = sc > 0.f;
                float m8[8] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY,
                               -INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    float v = __uint_as_float(sx[c]);
                    if (!pos_scale) v *= sc;
                    if (!full && j0 + c > lim) v = -INFINITY;
                    sx[c] = __float_as_uint(v);
                    m8[c & 7] = fmaxf(m8[c & 7], v);
                }
                float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
                if (pos_scale) mx *= sc;
                const float k_mul = pos_scale ? sc : 1.f;  // x = s * k_mul - base
                float alpha = 1.f;
                bool need = false;
                if (mx != -INFINITY) {
                    if (m_used == -INFINITY) {
                        m_used = mx;
                    } else if (mx > m_used + 8.f) {
                        alpha = fast_exp2(m_used - mx);
                        m_used = mx;
                        l *= alpha;
                        need = true;
                    }
                }
                const float base = m_used == -INFINITY ? 0.f : m_used;
                float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < HC / 2; ++e) {
                    const float x0 = fmaf(__uint_as_float(sx[2 * e]), k_mul, -base);
                    const float x1 = fmaf(__uint_as_float(sx[2 * e + 1]), k_mul, -base);
                    // pairs e with e % kExpFmaEvery == kExpFmaEvery - 1 on the
                    // FMA pipe, the rest on the special-function unit
                    const bool on_fma =
                        kExpFmaEvery > 0 && (e % (kExpFmaEvery > 0 ? kExpFmaEvery : 1)) == kExpFmaEvery - 1;
                    const float p0 = on_fma ? exp2_fma(x0) : fast_exp2(x0);
                    const float p1 = on_fma ? exp2_fma(x1) : fast_exp2(x1);
                    s4[e & 3] += p0;
                    s4[(e + 2) & 3] += p1;
                    sx[e] = pack2<T>(p0, p1);  // P column e = keys 2e, 2e+1 of this half
                }
                // P (HC keys, HC/2 columns) over the consumed first half of my S columns
                tmem_st32(t_s, *reinterpret_cast<uint32_t(*)[32]>(sx));
                l += (s4[0] + s4[1]) + (s4[2] + s4[3]);
                // rows of V past the sequence end may hold anything (even NaN):
                // zero the ones this group's PV reads so that P = 0 there
                // cannot produce 0 * NaN
                if (j0 + HC > it.kvb) {
                    const int sv = t % SV, uv = t / SV;
                    if (!wait_warp(b_vfull(sv), uv & 1)) { ok = false; break; }
                    const int zs = max(it.kvb - j * BN, g * HC), ze = (g + 1) * HC;
                    uint8_t *vbase = v_gen + sv * VB;
                    for (int q = r; q < (ze - zs) * 16; q += 128) {
                        const int row = zs + (q >> 4), chunk = q & 15;
                        *reinterpret_cast<uint4 *>(vbase + (chunk >> 3) * (BN * 128) + row * 128 + (chunk & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                // O_g *= alpha when the running max moved (rare: threshold 2^8);
                // PV_{t-1} of this group must be complete first
                if (__any_sync(0xffffffffu, need)) {
                    if (j >= 1 && !wait_warp(b_pvdone(t - 1, g), ((t - 1) >> 1) & 1)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < kPfDV / 32; ++c) {
                        uint32_t ro[32];
                        tmem_ld32(t_lane + o_g + c * 32, ro);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * alpha);
                        tmem_st32(t_lane + o_g + c * 32, ro);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(b_pfull(t, g));
            }
            if (!ok) break;
            // epilogue: wait for this group's last PV of the item (a commit
            // covers every earlier MMA too), trade (max, sum) with the other
            // group, merge the two partial O rows; group g writes output
            // columns [g*64, g*64+64) and group 0 the LSE
            const int tl = t_base + it.n_tiles - 1;
            if (it.n_tiles > 0 && !wait_warp(b_pvdone(tl, g), (tl >> 1) & 1)) { ok = false; break; }
            xchg[k & 1][0][g][r] = m_used;
            xchg[k & 1][1][g][r] = l;
            mbar_arrive(b_xchg);
            if (!wait_warp(b_xchg, k & 1)) { ok = false; break; }
            const float m0 = xchg[k & 1][0][0][r], m1 = xchg[k & 1][0][1][r];
            const float M = fmaxf(m0, m1);
            const float w0 = m0 == -INFINITY ? 0.f : fast_exp2(m0 - M);
            const float w1 = m1 == -INFINITY ? 0.f : fast_exp2(m1 - M);
            const float lt = xchg[k & 1][1][0][r] * w0 + xchg[k & 1][1][1][r] * w1;
            const bool have = it.n_tiles > 0;
            tc_fence_after();
            const int qi = it.i0 + r;
            const int64_t grow = static_cast<int64_t>(it.row_base) + r;
            const bool valid = qi < it.qb && grow < p.total_q;
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            const uint32_t ocol = g * (kPfDV / 2);
            T *orow = static_cast<T *>(p.out) + (grow * p.Hqo + it.h) * kPfDV + ocol;
#pragma unroll
            for (int c = 0; c < kPfDV / 64; ++c) {
                uint32_t ra[32], rb[32];
                if (have) {
                    tmem_ld32(t_lane + ocol + c * 32, ra);
                    tmem_ld32(t_lane + kPfDV + ocol + c * 32, rb);
                    tmem_wait_ld();
                }
                float o[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float v = 0.f;
                    if (have && w0 != 0.f) v += __uint_as_float(ra[e]) * w0;
                    if (have && w1 != 0.f) v += __uint_as_float(rb[e]) * w1;
                    o[e] = v * inv;
                }
                if (valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w = make_uint4(pack2<T>(o[q * 8 + 0], o[q * 8 + 1]), pack2<T>(o[q * 8 + 2], o[q * 8 + 3]),
                                             pack2<T>(o[q * 8 + 4], o[q * 8 + 5]), pack2<T>(o[q * 8 + 6], o[q * 8 + 7]));
                        *reinterpret_cast<uint4 *>(orow + c * 32 + q * 8) = w;
                    }
                }
            }
            if (valid && g == 0) p.lse[grow * p.Hqo + it.h] = lt > 0.f ? (M + fast_log2(lt)) * kLn2 : -INFINITY;
            // O has been read: the next item's first PV may overwrite it (items
            // without key tiles never touch O and are not counted)
            if (have) {
                tc_fence_before();
                mbar_arrive(b_ofree);
            }
            t_base += it.n_tiles;
        }
        if (!ok) give_up();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int DQK>
static size_t prefill_smem_bytes() {
    constexpr int SK = PfCfg<DQK>::SK, SV = PfCfg<DQK>::SV;
    return 1024 + kPfRows * DQK * 2 + SK * kPfBN * DQK * 2 + SV * kPfBN * kPfDV * 2 + 8 * (20 + 2 * SK + 2 * SV);
}

template <typename T, int DQK, int LAYOUT>
static int launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const PrefillParams &p, dim3 grid, cudaStream_t st) {
    const size_t smem = prefill_smem_bytes<DQK>();
    auto kern = prefill_tc_kernel<T, DQK, LAYOUT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PKV_ERR_CUDA;
    kern<<<grid, kPfThreads, smem, st>>>(tq, tk, tv, p);
    return PKV_OK;
}

template <typename T>
static int dispatch_prefill(int d_qk, int layout, const CUtensorMap &tq, const CUtensorMap &tk,
                            const CUtensorMap &tv, const PrefillParams &p, dim3 grid, cudaStream_t st) {
    if (d_qk == 128)
        return layout == PKV_HND ? launch_prefill<T, 128, PKV_HND>(tq, tk, tv, p, grid, st)
                                 : launch_prefill<T, 128, PKV_NHD>(tq, tk, tv, p, grid, st);
    return layout == PKV_HND ? launch_prefill<T, 192, PKV_HND>(tq, tk, tv, p, grid, st)
                             : launch_prefill<T, 192, PKV_NHD>(tq, tk, tv, p, grid, st);
}

// K or V cache as a 4-D tensor map whose box is one 64-element d-atom of
// `rows` consecutive slots of one (page, kv head).
static bool cache_tmap(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int layout, int d,
                       int page_size, int num_kv_heads, int64_t page_stride, int64_t num_pages,
                       int rows) {
    uint64_t dims[4], strides[3];
    uint32_t box[4];
    dims[0] = d;
    box[0] = 64;
    strides[0] = static_cast<uint64_t>(d) * 2;
    if (layout == PKV_HND) {
        dims[1] = page_size;
        dims[2] = num_kv_heads;
        strides[1] = static_cast<uint64_t>(page_size) * d * 2;
        box[1] = rows;
        box[2] = 1;
    } else {
        dims[1] = num_kv_heads;
        dims[2] = page_size;
        strides[1] = static_cast<uint64_t>(num_kv_heads) * d * 2;
        box[1] = 1;
        box[2] = rows;
    }
    dims[3] = static_cast<uint64_t>(num_pages);
    strides[2] = static_cast<uint64_t>(page_stride) * 2;
    box[3] = 1;
    return encode_tmap(m, base, dt, 4, dims, strides, box);
}

// workspace: cu_q[B+1], then the work-item counter of the persistent kernel
static size_t prefill_ws_bytes(int B) {
    return round_up(static_cast<size_t>(B + 1) * sizeof(int32_t), 256) + 256;
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t paged_prefill_workspace_size(int32_t batch_size, int32_t num_qo_heads,
                                               int32_t max_token_per_sequence,
                                               int32_t max_sequence_kv) {
    if (batch_size < 0 || num_qo_heads < 1 || max_token_per_sequence < 0 || max_sequence_kv < 0)
        return 0;
    return prefill_ws_bytes(batch_size);
}

extern "C" int paged_prefill(const void *q, int64_t total_q, const void *k_cache,
                             const void *v_cache, int64_t k_page_stride, int64_t v_page_stride,
                             int64_t max_num_pages, float scale, void *workspace,
                             size_t workspace_bytes, int32_t max_token_per_sequence,
                             int32_t max_sequence_kv, const int32_t *actual_seq_lens_q,
                             const int32_t *actual_seq_lens_kv, const int32_t *block_tables,
                             int32_t block_table_stride, int32_t batch_size, int32_t causal,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t d_qk,
                             int32_t d_vo, int32_t page_size, int32_t layout, int32_t dtype,
                             void *out, float *lse, int32_t *err_word, void *stream) {
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (batch_size < 0 || num_qo_heads < 1 || num_kv_heads < 1 || max_token_per_sequence < 0 ||
        max_sequence_kv < 0 || max_num_pages < 0 || block_table_stride < 0 || total_q < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_qo_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
    if ((d_qk != 128 && d_qk != 192) || d_vo != 128) return PKV_ERR_UNSUPPORTED;
    if (ilog2_exact(page_size) < 3 || page_size > 256) return PKV_ERR_UNSUPPORTED;
    if (batch_size > 65535 || num_qo_heads > 65535 || max_num_pages > 0x7fffffff ||
        total_q > 0x7fffffff)
        return PKV_ERR_UNSUPPORTED;
    if (k_page_stride < static_cast<int64_t>(num_kv_heads) * page_size * d_qk ||
        v_page_stride < static_cast<int64_t>(num_kv_heads) * page_size * d_vo ||
        static_cast<int64_t>(block_table_stride) * page_size < max_sequence_kv)
        return PKV_ERR_INVALID_ARG;
    if (batch_size == 0 || total_q == 0) return PKV_OK;
    // work items (query tiles x heads x requests) are counted in an int that
    // overshoots the total by one per CTA
    if (static_cast<int64_t>((max_token_per_sequence + kPfRows - 1) / kPfRows) * num_qo_heads * batch_size >
        0x7fffffff - 65536)
        return PKV_ERR_UNSUPPORTED;
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

    const CUtensorMapDataType tdt =
        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int rows = page_size < kPfBN ? page_size : kPfBN;
    CUtensorMap tq, tk, tv;
    {
        uint64_t dims[3] = {static_cast<uint64_t>(d_qk), static_cast<uint64_t>(num_qo_heads),
                            static_cast<uint64_t>(total_q)};
        uint64_t strides[2] = {static_cast<uint64_t>(d_qk) * 2,
                               static_cast<uint64_t>(num_qo_heads) * d_qk * 2};
        uint32_t box[3] = {64, 1, static_cast<uint32_t>(kPfRows)};
        if (!encode_tmap(&tq, q, tdt, 3, dims, strides, box)) return PKV_ERR_CUDA;
    }
    if (!cache_tmap(&tk, k_cache, tdt, layout, d_qk, page_size, num_kv_heads, k_page_stride,
                    max_num_pages, rows) ||
        !cache_tmap(&tv, v_cache, tdt, layout, d_vo, page_size, num_kv_heads, v_page_stride,
                    max_num_pages, rows))
        return PKV_ERR_CUDA;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *cu_q = static_cast<int32_t *>(workspace);
    int *work_counter = reinterpret_cast<int *>(static_cast<char *>(workspace) +
                                                round_up(static_cast<size_t>(batch_size + 1) * sizeof(int32_t), 256));
    prefill_plan_kernel<<<1, 32, 0, st>>>(actual_seq_lens_q, actual_seq_lens_kv, batch_size,
                                          max_token_per_sequence, max_sequence_kv, cu_q, err_word,
                                          work_counter);
    PrefillParams p;
    p.max_num_pages = max_num_pages;
    p.total_q = total_q;
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
    p.work_counter = work_counter;
    p.out = out;
    p.lse = lse;
    p.err = err_word;
    const int n_qt = (max_token_per_sequence + kPfRows - 1) / kPfRows;
    p.n_qt_max = n_qt;
    int launches = 1;
    const int64_t items = static_cast<int64_t>(n_qt) * num_qo_heads * batch_size;
    if (n_qt > 0) {
        // persistent: one CTA per SM (the shared-memory footprint allows one)
        const int64_t ctas = items < num_sms() ? items : num_sms();
        dim3 grid(static_cast<unsigned>(ctas));
        int rc = dtype == PKV_BF16 ? dispatch_prefill<__nv_bfloat16>(d_qk, layout, tq, tk, tv, p, grid, st)
                                   : dispatch_prefill<__half>(d_qk, layout, tq, tk, tv, p, grid, st);
        if (rc != PKV_OK) return rc;
        ++launches;
    }
    note_launches(launches);
    return launch_status();
}
