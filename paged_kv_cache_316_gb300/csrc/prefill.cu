// prefill.cu -- causal ragged batch prefill over a paged KV cache, with LSE.
//
// Computes what flashinfer.prefill.cudnn_batch_prefill_with_kv_cache
// documents (q, k_cache, v_cache, scale, workspace_buffer,
// max_token_per_sequence, max_sequence_kv, actual_seq_lens_q/kv,
// block_tables, causal, return_lse): the queries of request b are the last
// q_b of its kv_b positions; softmax(scale q k^T) v over the visible keys
// and the natural-log LSE of the scaled logits.
//
// A persistent CTA per SM takes work items from a global counter.  An item
// is one 128-row query tile of a request for TWO qo heads of the same kv
// head (blocks A and B; B is absent when the group size is odd and the
// heads run out), so every K/V tile brought into shared memory feeds two
// 128 x BN score tiles.  Twelve warps:
//   warps 0-7   the softmax, one thread per query row: block X = w / 4, TMEM
//           lane quarter w % 4.  Each thread reads its score row from TMEM
//           32 columns at a time, masks, takes the row max, runs the online
//           softmax in base 2 against a running max that is raised only
//           when the tile max exceeds it by more than 2^8, and writes P
//           (bf16/fp16) over the consumed S columns as the A operand of the
//           block's PV MMA, which accumulates into the block's O in TMEM; at
//           the end of the item it normalises O and writes it with the LSE;
//   warp 8      TMA producer: takes the items, loads both Q blocks and the K
//           tiles page by page through a ring of shared-memory stages;
//   warp 9      allocates tensor memory and runs the MMA issue loop (the
//           whole warp; an elect.sync leader issues the tcgen05 MMAs and
//           commits) in the order QK_A(0) QK_B(0) | PV_A(t) QK_A(t+1) PV_B(t)
//           QK_B(t+1) | ..., so that while one block's softmax runs the
//           tensor core works for the other block (ping-pong);
//   warp 10     TMA producer of the V tiles (a second ring);
//   warp 11     idle for 16-bit inputs.  With an E4M3 query and E4M3 caches
//           the QK MMAs are kind::f8f6f4 straight from the E4M3 Q and K
//           tiles, V tiles arrive as E4M3 in a byte ring and this warp widens
//           each one exactly to fp16 in the 16-bit V stage layout, so that
//           PV stays a 16-bit MMA with P in fp16.
// The softmax warps run with 200 registers and the others with 104
// (setmaxnreg).  Every wait is bounded; a wait that gives up sets
// PKV_DEV_ERR_TIMEOUT, the other roles stop, the copies in flight are
// waited for, tensor memory is freed and the CTA returns.
#include <math.h>

#include <type_traits>

#include "pkv_common.cuh"
#include "sm103_ptx.cuh"

namespace pkv {

constexpr int kPfRows = 128;     // query rows per block
constexpr int kPfDV = 128;

// Keys per tile (BN) and ring depths.  TMEM holds S of both blocks (BN
// columns each) and O of both blocks (128 columns each); shared memory holds
// both Q blocks, SK K stages and SV V stages (plus SV E4M3 V stages on the
// E4M3 path).
template <int DQK>
struct PfCfg;
template <>
struct PfCfg<128> {
    static constexpr int BN = 128, SK = 2, SV = 2;
};
template <>
struct PfCfg<192> {
    static constexpr int BN = 96, SK = 2, SV = 2;
};
template <int DQK>
struct PfRoles {
    static constexpr int kSoftmaxWarps = 8;
    static constexpr int kTmaWarp = kSoftmaxWarps, kMmaWarp = kSoftmaxWarps + 1, kTmaVWarp = kSoftmaxWarps + 2;
    // + one idle warp, so that the producer / MMA warps make a whole warpgroup
    static constexpr int kThreads = 32 * (kSoftmaxWarps + 4);
};
// Register split with one softmax thread per row (384 threads): launched at
// 168 registers a thread (65536 / 384, rounded down to a multiple of 8), the
// producer warpgroup drops to kRegsLow and the two softmax warpgroups rise to
// kRegsHigh: 128 x 104 + 256 x 200 = 64512 = 384 x 168, the launch's total.
// (A row's 128 scores and the rest of the softmax fit in 200 without spills;
// the producers spill below about 100.)
constexpr int kRegsLow = 104, kRegsHigh = 200;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= 384 * 168, "register split exceeds the launch's registers");
static int pf_bn(int d_qk) { return d_qk == 128 ? PfCfg<128>::BN : PfCfg<192>::BN; }
// Rows per TMA box: pages, or parts of pages of the largest power of two
// dividing BN, so that no box crosses a page and the boxes tile a key tile.
__host__ __device__ __forceinline__ int pf_box_rows(int page_size, int bn) {
    const int p2 = bn & -bn;
    return page_size < p2 ? page_size : p2;
}

struct PrefillParams {
    int64_t max_num_pages;
    int64_t total_q;
    float scale_log2;
    const int32_t *seq_lens_q;
    const int32_t *seq_lens_kv;
    const int32_t *cu_q;  // [B+1] in the workspace
    const int32_t *block_tables;
    int64_t bt_stride;
    const int32_t *cu_items;  // [B+1] in the workspace: U x prefix sum of query tiles
    int B, causal, Hqo, Hkv, group, page_shift, max_q, max_kv;
    int pairs;  // head pairs per kv head: (group + 1) / 2; U = Hkv * pairs items per query tile
    // contiguous K/V (no block table): [rows, Hkv, d] tensors, request b's keys
    // from row off_k[b] (K) / off_v[b] (V), by default the prefix sum cu_kv[b]
    int contiguous;
    const int32_t *cu_kv;   // [B+1] in the workspace
    // optional placement (token rows) of each request's queries, outputs and
    // keys/values; NULL = packed by the prefix sums
    const int32_t *off_q, *off_o, *off_k, *off_v;
    int *work_counter;  // in the workspace, zeroed by the plan kernel
    // device-resident dequantisation factors of E4M3 inputs (NULL: 1):
    // q_scale * k_scale multiplies the logits, v_scale the output
    const float *q_scale, *k_scale, *v_scale;
    void *out;
    float *lse;
    int32_t *err;
    unsigned long long wait_ns;  // limit of every bounded pipeline wait
    // K tiles through the 5-D map of cache_tmap5 (one copy per page part for
    // all of a row's 128-byte atoms; stages laid out [8-row group][atom][8
    // rows][128 B]) with the coordinate page * k5_ratio + kv head, or (0)
    // through the 4-D map, one copy per atom ([atom][row][128 B] stages)
    int k5, k5_ratio;
};

// cu_q / cu_kv = exclusive prefix sums of the query / kv lengths and
// cu_items = U x the exclusive prefix sum of the 128-row query tiles (one
// warp, 32 requests at a time); flags lengths above their maxima and requests with fewer keys
// than queries; zeroes the work-item counter.
__global__ void prefill_plan_kernel(const int32_t *__restrict__ lq, const int32_t *__restrict__ lkv,
                                    int B, int U, int max_q, int max_kv, int32_t *__restrict__ cu_q,
                                    int32_t *__restrict__ cu_items, int32_t *__restrict__ cu_kv,
                                    int32_t *err, int *work_counter) {
    const int lane = threadIdx.x;
    pdl_launch_dependents();  // the main kernel may start its prologue meanwhile
    int carry = 0, carry_t = 0, carry_k = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
        int b = b0 + lane;
        int v = b < B ? lq[b] : 0;
        if (b < B && (v > max_q || v < 0 || lkv[b] > max_kv)) set_err(err, PKV_DEV_ERR_LEN);
        v = min(max(v, 0), max_q);
        if (b < B && min(lkv[b], max_kv) < v) set_err(err, PKV_DEV_ERR_QLEN);
        const int nt = (v + kPfRows - 1) / kPfRows;
        const int vk = b < B ? min(max(lkv[b], 0), max_kv) : 0;
        int x = v, xt = nt, xk = vk;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, x, o);
            int yt = __shfl_up_sync(0xffffffffu, xt, o);
            int yk = __shfl_up_sync(0xffffffffu, xk, o);
            if (lane >= o) {
                x += y;
                xt += yt;
                xk += yk;
            }
        }
        if (b < B) {
            cu_q[b] = carry + x - v;
            cu_items[b] = (carry_t + xt - nt) * U;
            cu_kv[b] = carry_k + xk - vk;
        }
        carry += __shfl_sync(0xffffffffu, x, 31);
        carry_t += __shfl_sync(0xffffffffu, xt, 31);
        carry_k += __shfl_sync(0xffffffffu, xk, 31);
    }
    if (lane == 0) {
        cu_q[B] = carry;
        cu_items[B] = carry_t * U;
        cu_kv[B] = carry_k;
        *work_counter = 0;
    }
}

template <typename T>
struct IsBf16 {
    static constexpr bool value = false;
};
template <>
struct IsBf16<__nv_bfloat16> {
    static constexpr bool value = true;
};

template <typename T>
__device__ __forceinline__ float2 unpack2(uint32_t w);
template <>
__device__ __forceinline__ float2 unpack2<__nv_bfloat16>(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}
template <>
__device__ __forceinline__ float2 unpack2<__half>(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
}

// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;\n" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Wait for this thread's tensor-memory loads, with the 32 destination
// registers as operands so that no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;\n"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
                   "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]),
                   "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                   "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// One work item: query tile x (counted from the LAST tile of the request, the
// one that sees the most keys) of request b for qo heads hA and hB (hB < 0:
// block B absent).  Items are numbered request by request (so that the CTAs
// running at the same time share one request's K/V in L2), inside a request
// x-major with the (kv head, pair) units innermost, so every request hands
// out its heaviest tiles first.
struct PfItem {
    int b, hA, hB, i0, row_base, orow_base, kvh, shift, qb, kvb, n_tiles;
    int kv_k, kv_v;  // first K / V row of the request (contiguous K/V)
};

__device__ __forceinline__ void pf_item(const PrefillParams &p, const int4 itm, int bn, PfItem &it) {
    it.b = itm.x;
    it.hA = itm.y;
    it.hB = itm.z;
    it.qb = min(max(p.seq_lens_q[it.b], 0), p.max_q);
    it.kvb = min(max(p.seq_lens_kv[it.b], 0), p.max_kv);
    const int n_qt = (it.qb + kPfRows - 1) / kPfRows;
    it.i0 = (n_qt - 1 - itm.w) * kPfRows;
    it.row_base = (p.off_q ? p.off_q[it.b] : p.cu_q[it.b]) + it.i0;
    it.orow_base = (p.off_o ? p.off_o[it.b] : p.cu_q[it.b]) + it.i0;
    if (p.contiguous) {
        it.kv_k = p.off_k ? p.off_k[it.b] : p.cu_kv[it.b];
        it.kv_v = p.off_v ? p.off_v[it.b] : p.cu_kv[it.b];
    }
    it.kvh = it.hA / p.group;
    it.shift = it.kvb - it.qb;  // query i sits at position shift + i
    int k_hi = p.causal ? min(it.kvb, it.shift + it.i0 + kPfRows) : it.kvb;
    if (k_hi < 0) k_hi = 0;
    it.n_tiles = (k_hi + bn - 1) / bn;
}

// F8: the query and the caches hold E4M3 (one byte per element; d_qk 128):
// QK runs as kind::f8f6f4 MMAs straight from the E4M3 tiles, and the E4M3 V
// tiles are widened (exactly) to fp16 in shared memory by warp 11 for the
// 16-bit PV, whose P is then fp16.  T is the output type.
template <typename T, int DQK, int LAYOUT, bool F8 = false>
__global__ void __launch_bounds__(PfRoles<DQK>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    constexpr int BN = PfCfg<DQK>::BN;
    // (F8: a third V stage, so that the widening of a tile has a whole tile
    // period of slack before its PV)
    constexpr int SK = PfCfg<DQK>::SK, SV = PfCfg<DQK>::SV;
    constexpr int kTmaWarp = PfRoles<DQK>::kTmaWarp, kMmaWarp = PfRoles<DQK>::kMmaWarp,
                  kTmaVWarp = PfRoles<DQK>::kTmaVWarp;
    static_assert(!F8 || DQK == 128, "E4M3 tiles: d_qk 128");
    using TP = typename std::conditional<F8, __half, T>::type;  // element type of P (and V)
    constexpr int ES = F8 ? 1 : 2;               // bytes per Q / K element
    constexpr int QA = DQK * ES / 128;           // 128-byte atoms of a Q / K row
    constexpr uint32_t QB = kPfRows * DQK * ES;  // bytes of one Q block
    constexpr uint32_t KB = BN * DQK * ES;       // bytes of one K stage
    constexpr uint32_t VB = BN * kPfDV * 2;      // bytes of one 16-bit V stage
    constexpr uint32_t V8B = F8 ? BN * kPfDV : 0;  // bytes of one E4M3 V stage (F8)
    constexpr int KSTEPS = DQK * ES / 32;        // 32-byte K-steps of a QK MMA
    constexpr bool K5 = DQK == 192 && !F8;       // K tiles may come through the 5-D map (p.k5)
    constexpr int NI = 2;                        // slots of the work-item ring
    // TMEM columns (every region starts at a multiple of 128): S of block X
    // at X * S_STRIDE (BN columns; P of a chunk, 16-bit pairs,
    // overwrites the chunk's first columns), O of block X at O_COL + X * 128
    constexpr uint32_t TMEM_COLS = 512;
    constexpr uint32_t S_STRIDE = 128;
    constexpr uint32_t O_COL = 2 * S_STRIDE;
    static_assert(BN <= S_STRIDE, "score tile wider than its TMEM region");
    static_assert(O_COL + 2 * kPfDV <= TMEM_COLS, "TMEM budget");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t q_s = smem_u32(smem);  // block A, then block B
    const uint32_t k_s = q_s + 2 * QB;
    const uint32_t v_s = k_s + SK * KB;
    const uint32_t v8_s = v_s + SV * VB;       // E4M3 V stages (F8)
    const uint32_t bar0 = v8_s + SV * V8B;
    uint8_t *v_gen = smem + 2 * QB + SK * KB;  // generic pointer to the V stages
    const uint8_t *v8_gen = v_gen + SV * VB;   // and to the E4M3 V stages
    uint32_t nb = 0;
    const uint32_t b_qfull = bar0 + 8u * nb++;   // Q blocks of the current item landed
    const uint32_t b_qempty = bar0 + 8u * nb++;  // last QK of an item done: Q buffers free
    const uint32_t b_item_full0 = bar0 + 8u * nb; nb += NI;
    const uint32_t b_item_empty0 = bar0 + 8u * nb; nb += NI;
    const uint32_t b_kfull0 = bar0 + 8u * nb; nb += SK;
    const uint32_t b_kempty0 = bar0 + 8u * nb; nb += SK;
    const uint32_t b_vfull0 = bar0 + 8u * nb; nb += SV;
    const uint32_t b_vempty0 = bar0 + 8u * nb; nb += SV;
    const uint32_t b_sfull0 = bar0 + 8u * nb; nb += 2;  // per block: S tile written
    const uint32_t b_pfull0 = bar0 + 8u * nb; nb += 2;  // per block: P tile written
    const uint32_t b_odone0 = bar0 + 8u * nb; nb += 2;  // per block: last PV of an item done
    const uint32_t b_drain = bar0 + 8u * nb++;          // every MMA the issuer made has completed
    const uint32_t b_v8full0 = bar0 + 8u * nb; nb += F8 ? SV : 0;   // E4M3 V stage landed (F8)
    const uint32_t b_v8empty0 = bar0 + 8u * nb; nb += F8 ? SV : 0;  // E4M3 V stage widened (F8)
    auto b_item_full = [&](int i) { return b_item_full0 + 8u * i; };
    auto b_item_empty = [&](int i) { return b_item_empty0 + 8u * i; };
    auto b_kfull = [&](int s) { return b_kfull0 + 8u * s; };
    auto b_kempty = [&](int s) { return b_kempty0 + 8u * s; };
    auto b_vfull = [&](int s) { return b_vfull0 + 8u * s; };
    auto b_vempty = [&](int s) { return b_vempty0 + 8u * s; };
    auto b_sfull = [&](int x) { return b_sfull0 + 8u * x; };
    auto b_pfull = [&](int x) { return b_pfull0 + 8u * x; };
    auto b_odone = [&](int x) { return b_odone0 + 8u * x; };
    auto b_v8full = [&](int s) { return b_v8full0 + 8u * s; };
    auto b_v8empty = [&](int s) { return b_v8empty0 + 8u * s; };
    constexpr int kConvWarp = PfRoles<DQK>::kSoftmaxWarps + 3;  // (F8) the V widening warp
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ int4 item_ring[NI];  // (request, head A, head B, x); request -1: no more work

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(b_qfull, 1);
        mbar_init(b_qempty, 1);
        for (int i = 0; i < NI; ++i) {
            mbar_init(b_item_full(i), 1);
            // MMA thread, V producer, softmax threads (and the V widening warp)
            mbar_init(b_item_empty(i), 2 + 256 + (F8 ? 1 : 0));
        }
        for (int s = 0; s < SK; ++s) {
            mbar_init(b_kfull(s), 1);
            mbar_init(b_kempty(s), 1);
        }
        for (int s = 0; s < SV; ++s) {
            mbar_init(b_vfull(s), F8 ? 32 : 1);  // (F8: the widening warp's lanes)
            mbar_init(b_vempty(s), 1);
            if (F8) {
                mbar_init(b_v8full(s), 1);
                mbar_init(b_v8empty(s), 32);
            }
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(b_sfull(x), 1);
            mbar_init(b_pfull(x), 128);
            mbar_init(b_odone(x), 1);
        }
        mbar_init(b_drain, 1);
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
    pdl_wait();  // the plan kernel's prefix sums and zeroed work counter
    const uint32_t tmem = tmem_base_s;
    volatile int *abort_flag = &abort_s;
    const uint64_t wlim = p.wait_ns;
    auto give_up = [&]() {
        *abort_flag = 1;
        set_err(p.err, PKV_DEV_ERR_TIMEOUT);
    };
    // the k-th item published by the K producer (request -1: no more work);
    // every consumer role takes every item, in order, and releases the slot
    auto take_item = [&](int k, bool &ok) -> int4 {
        const int slot = k % NI;
        if (!mbar_wait(b_item_full(slot), (k / NI) & 1, abort_flag, wlim)) {
            ok = false;
            return make_int4(-1, 0, 0, 0);
        }
        const volatile int *q = reinterpret_cast<const volatile int *>(&item_ring[slot]);
        const int4 v = make_int4(q[0], q[1], q[2], q[3]);
        mbar_arrive(b_item_empty(slot));
        return v;
    };

    // Barrier phases.  Every wait below is for the newest phase that can be
    // pending, so that a parity can never match an older completed phase:
    // K/V stage s of tile t: phase t / S{K,V}; sfull/pfull of block X: the
    // block's tile count; odone of block X: the block's count of items with
    // tiles; qfull/qempty: the item count.  S_X(t+1) is written by a QK
    // issued after PV_X(t), which needs P_X(t), so no block can run two
    // phases ahead of its partner.

    if (warp >= PfRoles<DQK>::kSoftmaxWarps) {
        // warps 8-11 (one warpgroup): the producers, the MMA issuer and an idle
        // warp give registers to the softmax warpgroups
        reg_dealloc<kRegsLow>();
        if (warp == kTmaWarp || warp == kTmaVWarp) {
            // ------------------------------------------------------------ TMA producers
            // Warp 8 takes items from the global counter, publishes them, loads
            // the Q blocks and the K tiles; warp 10 loads the V tiles.  A K stage
            // is released by the last QK that reads it and a V stage by the last
            // PV.  Each warp looks up a tile's page ids in one coalesced load,
            // one tile ahead; an elect.sync leader issues the copies.
            const bool is_k = warp == kTmaWarp;
            const bool leader = elect_one();
            const int leader_lane = __ffs(__ballot_sync(0xffffffffu, leader)) - 1;
            if (leader) {
                if (is_k) {
                    prefetch_tmap(&tm_q);
                    prefetch_tmap(&tm_k);
                } else {
                    prefetch_tmap(&tm_v);
                }
            }
            const int S = 1 << p.page_shift;
            // rows per TMA box: a page or part of one; a whole tile for contiguous K/V
            const int RB = p.contiguous ? BN : pf_box_rows(S, BN);
            const int nbox = BN / RB;       // boxes (pages or page parts) per tile, <= 16
            const int oob = static_cast<int>(p.max_num_pages);  // page coordinate past the pool: zero fill
            const int NS = is_k ? SK : SV;
            const int U = p.Hkv * p.pairs;
            // the V producer's ring: the 16-bit V stages, or (F8) the E4M3
            // stages the widening warp reads
            auto v_full = [&](int st) { return F8 ? b_v8full(st) : b_vfull(st); };
            auto v_empty = [&](int st) { return F8 ? b_v8empty(st) : b_vempty(st); };
            bool ok = true;
            int t_base = 0;  // tiles of earlier items (global tile counter)
            int t_next = 0;  // (leader) tiles [0, t_next) have their copies issued
            int q_loads = 0; // (leader) Q blocks of items [0, q_loads) issued
            const int total_items = is_k ? p.cu_items[p.B] : 0;
            int b_scan = 0;  // request of this CTA's previous item: items come in increasing order
            for (int k = 0; ok; ++k) {
                int4 itm = make_int4(-1, 0, 0, 0);
                if (is_k) {
                    // take the next item from the counter, find its request with a
                    // warp-wide forward scan of cu_items, and publish it
                    int c = 0;
                    if (leader) c = atomicAdd(p.work_counter, 1);
                    c = __shfl_sync(0xffffffffu, c, leader_lane);
                    if (c < total_items) {
                        while (true) {  // ends: cu_items[B] = total > c
                            const int bi = b_scan + lane;
                            const int v = bi <= p.B ? p.cu_items[bi] : 0x7fffffff;
                            const unsigned m = __ballot_sync(0xffffffffu, v > c);
                            if (m) {
                                b_scan += __ffs(m) - 2;  // cu_items[b_scan] <= c always
                                break;
                            }
                            b_scan += 32;
                        }
                        const int rem = c - p.cu_items[b_scan];
                        const int u = rem % U, kvh = u / p.pairs;
                        const int hA = kvh * p.group + 2 * (u % p.pairs);
                        const int hB = hA + 1 < (kvh + 1) * p.group ? hA + 1 : -1;
                        itm = make_int4(b_scan, hA, hB, rem / U);
                    }
                    if (leader) {
                        const int slot = k % NI;
                        if (k >= NI && !mbar_wait(b_item_empty(slot), ((k / NI) - 1) & 1, abort_flag, wlim)) {
                            give_up();
                            ok = false;
                        } else {
                            item_ring[slot] = itm;
                            mbar_arrive(b_item_full(slot));
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, leader_lane);
                } else {
                    if (leader) itm = take_item(k, ok);
                    itm.x = __shfl_sync(0xffffffffu, itm.x, leader_lane);
                    itm.y = __shfl_sync(0xffffffffu, itm.y, leader_lane);
                    itm.z = __shfl_sync(0xffffffffu, itm.z, leader_lane);
                    itm.w = __shfl_sync(0xffffffffu, itm.w, leader_lane);
                    ok = __shfl_sync(0xffffffffu, ok, leader_lane);
                }
                if (!ok || itm.x < 0) break;
                PfItem it;
                pf_item(p, itm, BN, it);
                const int32_t *bt = p.block_tables + static_cast<int64_t>(it.b) * p.bt_stride;
                // Q blocks of this item, once the previous item's last QK is done;
                // loaded after the item's first K tile so that the two overlap
                auto load_q = [&]() {  // the K producer's leader
                    if (k >= 1 && !mbar_wait(b_qempty, (k - 1) & 1, abort_flag, wlim)) {
                        give_up();
                        ok = false;
                    } else {
                        mbar_expect_tx(b_qfull, 2 * QB);
                        if (kDebugBounds && it.qb > 0) dbg_in(it.row_base, 1, p.total_q, p.err);
                        // both blocks' Q in one copy (heads hA and hA + 1; when block B
                        // is absent the second head's rows land in its unused buffer)
                        tma_load_4d(q_s, &tm_q, b_qfull, 0, it.row_base, 0, it.hA);
                        q_loads = k + 1;
                    }
                };
                // the item's Q blocks into L2 now: their load waits for the
                // previous item's last QK, and from HBM (128 rows 8 KB apart per
                // head and atom) it would take several thousand cycles
                if (is_k && leader && it.n_tiles > 0) tma_prefetch_l2_4d(&tm_q, 0, it.row_base, 0, it.hA);
                if (is_k && leader && it.n_tiles == 0) load_q();
                ok = __shfl_sync(0xffffffffu, ok, leader_lane);
                if (!ok) break;
                auto lookup = [&](int j) {  // lane i < nbox: page of box i of tile j
                    const int key = j * BN + lane * RB;
                    int page = oob;
                    if (p.contiguous) return 0;  // one page: the whole tensor
                    if (lane < nbox && key < it.kvb &&
                        dbg_in(key >> p.page_shift, 1, (p.max_kv + S - 1) >> p.page_shift, p.err)) {
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
                    if (leader) {
                        const int st = t % NS, us = t / NS;
                        if (us > 0 && !mbar_wait(is_k ? b_kempty(st) : v_empty(st), (us - 1) & 1, abort_flag, wlim)) {
                            give_up();
                            ok = false;
                        } else {
                            const uint32_t full = is_k ? b_kfull(st) : v_full(st);
                            mbar_expect_tx(full, is_k ? KB : (F8 ? V8B : VB));
                            const int j0 = j * BN;
    #pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                if (i >= nbox) break;
                                const int r0 = i * RB;
                                const int slot0 = p.contiguous ? (is_k ? it.kv_k : it.kv_v) + j0 + r0
                                                               : (j0 + r0) & (S - 1);
                                const int ca = LAYOUT == PKV_HND ? slot0 : it.kvh;
                                const int cb = LAYOUT == PKV_HND ? it.kvh : slot0;
                                // (debug build) a box starts on a pool page or on the
                                // zero-fill page and stays inside its page; the tensor
                                // map bounds every copy in hardware, so the copy is
                                // issued regardless and the barrier's byte count holds
                                if (kDebugBounds && !p.contiguous) {
                                    dbg_in(pages[i], 1, p.max_num_pages + 1, p.err);
                                    dbg_in(slot0, RB, S, p.err);
                                }
                                if (is_k && K5 && p.k5) {  // every atom of the page part in one copy
                                    tma_load_5d(k_s + st * KB + r0 * (QA * 128), &tm_k, full, 0, 0, 0, slot0 >> 3,
                                                pages[i] * p.k5_ratio + it.kvh);
                                } else if (is_k) {
                                    for (int c = 0; c < QA; ++c)
                                        tma_load_4d(k_s + st * KB + c * (BN * 128) + r0 * 128, &tm_k, full,
                                                    c * (128 / ES), ca, cb, pages[i]);
                                } else if (F8) {  // one 128-byte atom: a whole E4M3 row
                                    tma_load_4d(v8_s + st * V8B + r0 * 128, &tm_v, full, 0, ca, cb, pages[i]);
                                } else {
                                    for (int c = 0; c < kPfDV / 64; ++c)
                                        tma_load_4d(v_s + st * VB + c * (BN * 128) + r0 * 128, &tm_v, full, c * 64, ca,
                                                    cb, pages[i]);
                                }
                            }
                            t_next = t + 1;
                            if (is_k && j == 0) load_q();
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, leader_lane);
                    if (!ok) break;
                }
                t_base += it.n_tiles;
            }
            // Before the CTA exits -- after the last item, or after a wait gave
            // up with copies in flight -- wait for every copy this warp issued to
            // land: the last phase issued on each stage (the earlier ones of a
            // stage completed before it was reused) and the last Q blocks.
            if (leader) {
                for (int t = t_next > NS ? t_next - NS : 0; t < t_next; ++t)
                    if (!mbar_wait_drain(is_k ? b_kfull(t % NS) : v_full(t % NS), (t / NS) & 1))
                        set_err(p.err, PKV_DEV_ERR_TIMEOUT);
                if (is_k && q_loads > 0 && !mbar_wait_drain(b_qfull, (q_loads - 1) & 1))
                    set_err(p.err, PKV_DEV_ERR_TIMEOUT);
            }
            __syncwarp();
        } else if (warp == kMmaWarp) {
            // ------------------------------------------------------------ MMA issuer
            // Per item of n tiles: QK_A(0) QK_B(0), then for every tile t:
            // PV_A(t) QK_A(t+1) PV_B(t) QK_B(t+1).  tcgen05 MMAs execute in issue
            // order, so QK_X(t+1), which overwrites S_X, cannot disturb PV_X(t)
            // reading P_X from it, and a completed S_X(t+1) implies that PV_X(t)
            // is complete (the softmax relies on both).
            // The whole warp runs the loop (warp-uniform descriptor arithmetic);
            // one elected lane issues every MMA and commit, so that each commit
            // tracks all the MMAs before it.
            {
                const bool leader = elect_one();
                auto mwait = [&](uint32_t bar, uint32_t parity) {
                    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, wlim));
                };
                auto commit = [&](uint32_t bar) {
                    if (leader) umma_commit(bar);
                };
                // (F8: kind::f8f6f4 with E4M3 A and B, whose format code is 0)
                constexpr uint32_t idesc_qk = umma_idesc(kPfRows, BN, !F8 && IsBf16<T>::value, false);
                constexpr uint32_t idesc_pv = umma_idesc(kPfRows, kPfDV, IsBf16<TP>::value, true);
                const uint64_t qdesc0 = umma_sdesc_sw128(q_s, 16, 1024);
                const bool k5 = K5 && p.k5;
                const uint64_t kdesc0 = umma_sdesc_sw128(k_s, 16, k5 ? QA * 1024 : 1024);
                const uint32_t k_atom = k5 ? 1024u : static_cast<uint32_t>(BN * 128);
                const uint64_t vdesc0 = umma_sdesc_sw128(v_s, BN * 128, 1024);
                bool ok = true;
                int t_base = 0;   // K/V tiles of earlier items
                int tb_base = 0;  // tiles of block B in earlier items
                auto wait_k = [&](int t) {
                    if (!mwait(b_kfull(t % SK), (t / SK) & 1)) return false;
                    tc_fence_after();
                    return true;
                };
                auto qk = [&](int x, int t) {  // S_X = Q_X K(t)^T
                    const uint64_t kd = kdesc0 + (((t % SK) * KB) >> 4);
                    const uint64_t qd = qdesc0 + ((x * QB) >> 4);
    #pragma unroll
                    for (int kk = 0; kk < KSTEPS; ++kk) {  // 32-byte steps, four per 128-byte atom
                        const uint64_t qa = qd + (((kk >> 2) * (kPfRows * 128) + (kk & 3) * 32) >> 4);
                        const uint64_t ka = kd + (((kk >> 2) * k_atom + (kk & 3) * 32) >> 4);
                        if (!leader) continue;
                        if constexpr (F8)
                            umma_ss_f8(tmem + x * S_STRIDE, qa, ka, idesc_qk, kk > 0 ? 1u : 0u);
                        else
                            umma_ss(tmem + x * S_STRIDE, qa, ka, idesc_qk, kk > 0 ? 1u : 0u);
                    }
                    commit(b_sfull(x));
                };
                // P column of keys 16kk .. 16kk+15: the softmax writes chunk c
                // (keys 32c .. 32c + 31) as 16-bit pairs at the chunk's first
                // column
                auto pcol = [](int kk) { return 32 * (kk / 2) + 8 * (kk % 2); };
                auto pv = [&](int x, int t, bool first) {  // O_X (+)= P_X V(t)
                    const uint64_t vd = vdesc0 + (((t % SV) * VB) >> 4);
    #pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        if (leader)
                            umma_ts(tmem + O_COL + x * kPfDV, tmem + x * S_STRIDE + pcol(kk), vd + ((kk * 16 * 128) >> 4),
                                    idesc_pv, (!first || kk > 0) ? 1u : 0u);
                };
                for (int k = 0; ok; ++k) {
                    int4 itm = make_int4(-1, 0, 0, 0);
                    if (lane == 0) itm = take_item(k, ok);
                    itm.x = __shfl_sync(0xffffffffu, itm.x, 0);
                    itm.y = __shfl_sync(0xffffffffu, itm.y, 0);
                    itm.z = __shfl_sync(0xffffffffu, itm.z, 0);
                    itm.w = __shfl_sync(0xffffffffu, itm.w, 0);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok || itm.x < 0) break;
                    PfItem it;
                    pf_item(p, itm, BN, it);
                    const bool hasB = it.hB >= 0;
                    const int n = it.n_tiles;
                    if (!mwait(b_qfull, k & 1)) { ok = false; break; }
                    if (n == 0) {
                        commit(b_qempty);
                        continue;
                    }
                    if (!wait_k(t_base)) { ok = false; break; }
                    qk(0, t_base);
                    if (hasB) qk(1, t_base);
                    commit(b_kempty(t_base % SK));
                    if (n == 1) commit(b_qempty);
                    for (int j = 0; j < n; ++j) {
                        const int t = t_base + j, tb = tb_base + j;
                        const bool more = j + 1 < n;
                        // block A: PV_A(t), then QK_A(t+1).  V(t) and K(t+1) arrive
                        // long before P_A(t): wait for them first, so that once P_A
                        // is there the MMAs go out back to back
                        if (!mwait(b_vfull(t % SV), (t / SV) & 1)) { ok = false; break; }
                        if (more && !mwait(b_kfull((t + 1) % SK), ((t + 1) / SK) & 1)) {
                            ok = false;
                            break;
                        }
                        if (!mwait(b_pfull(0), t & 1)) { ok = false; break; }
                        tc_fence_after();
                        pv(0, t, j == 0);
                        if (!more) commit(b_odone(0));
                        if (more) {
                            qk(0, t + 1);
                            if (!hasB) {
                                commit(b_kempty((t + 1) % SK));
                                if (j + 2 == n) commit(b_qempty);
                            }
                        }
                        // block B: PV_B(t), then QK_B(t+1)
                        if (hasB) {
                            if (!mwait(b_pfull(1), tb & 1)) { ok = false; break; }
                            tc_fence_after();
                            pv(1, t, j == 0);
                            if (!more) commit(b_odone(1));
                            if (more) {
                                qk(1, t + 1);
                                commit(b_kempty((t + 1) % SK));
                                if (j + 2 == n) commit(b_qempty);
                            }
                        }
                        commit(b_vempty(t % SV));
                    }
                    t_base += n;
                    if (hasB) tb_base += n;
                }
                if (!ok && leader) give_up();
                // every MMA issued (also those of an abandoned item) completes
                // before tensor memory is freed
                commit(b_drain);
                if (leader && !mbar_wait_drain(b_drain, 0)) set_err(p.err, PKV_DEV_ERR_TIMEOUT);
            }
            __syncwarp();
        } else if (F8 && warp == kConvWarp) {
            // ------------------------------------------------------------ V widening (F8)
            // Every E4M3 V stage is widened, exactly, into the matching fp16
            // stage in the layout the TMA gives a 16-bit tile (two 64-dim
            // atoms, 128-byte swizzle), once PV has released that stage; then
            // each lane makes its writes visible to the tensor core and arrives.
            bool ok = true;
            int t_base = 0;
            for (int k = 0; ok; ++k) {
                int4 itm = make_int4(-1, 0, 0, 0);
                if (lane == 0) itm = take_item(k, ok);
                itm.x = __shfl_sync(0xffffffffu, itm.x, 0);
                itm.y = __shfl_sync(0xffffffffu, itm.y, 0);
                itm.z = __shfl_sync(0xffffffffu, itm.z, 0);
                itm.w = __shfl_sync(0xffffffffu, itm.w, 0);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok || itm.x < 0) break;
                PfItem it;
                pf_item(p, itm, BN, it);
                for (int j = 0; j < it.n_tiles; ++j) {
                    const int t = t_base + j, st = t % SV, us = t / SV;
                    bool w = mbar_wait(b_v8full(st), us & 1, abort_flag, wlim);
                    if (us > 0) w = w && mbar_wait(b_vempty(st), (us - 1) & 1, abort_flag, wlim);
                    if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                    const uint8_t *__restrict__ src = v8_gen + st * V8B;
                    uint8_t *__restrict__ dst = v_gen + st * VB;
                    // 16-byte chunk q: row q / 8, dims 16c .. 16c + 15 (c = q % 8);
                    // four chunks per lane loaded before any is widened and stored
                    constexpr int kBatch = 4;
#pragma unroll 1
                    for (int q0 = lane; q0 < BN * 8; q0 += 32 * kBatch) {
                        uint4 raw[kBatch];
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int q = q0 + 32 * u, row = q >> 3, c = q & 7;
                            raw[u] = *reinterpret_cast<const uint4 *>(src + row * 128 + ((c ^ (row & 7)) << 4));
                        }
#pragma unroll
                        for (int u = 0; u < kBatch; ++u) {
                            const int q = q0 + 32 * u, row = q >> 3, c = q & 7;
                            const uint32_t x[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
                            uint32_t h[8];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                h[2 * i] = widen_e4m3x2<__half>(x[i] & 0xffffu);
                                h[2 * i + 1] = widen_e4m3x2<__half>(x[i] >> 16);
                            }
                            // dims 16c .. 16c + 7 and 16c + 8 .. 16c + 15: 16-byte
                            // chunks 2(c % 4) and 2(c % 4) + 1 of 64-dim atom c / 4
                            uint8_t *d0 = dst + (c >> 2) * (BN * 128) + row * 128;
                            const int ch = 2 * (c & 3);
                            *reinterpret_cast<uint4 *>(d0 + ((ch ^ (row & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
                            *reinterpret_cast<uint4 *>(d0 + (((ch + 1) ^ (row & 7)) << 4)) =
                                make_uint4(h[4], h[5], h[6], h[7]);
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(b_vfull(st));
                    mbar_arrive(b_v8empty(st));
                }
                t_base += it.n_tiles;
            }
            if (!ok) give_up();
            __syncwarp();
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        // One thread per query row, one warpgroup per block: warp w serves
        // block X = w / 4, TMEM lane quarter w % 4.  The row's scores are held
        // in registers (the softmax warpgroups' larger register budget); per
        // tile the thread takes their max, keeps a running max m in base 2
        // that rises only when a tile's max exceeds it by more than 8 (a
        // factor 2^8; P then stays below 2^8; the row sum and O are rescaled
        // then), and writes P, 16-bit pairs, over the first half of each
        // consumed 32-column chunk of S: the A operand of the block's PV MMA.
        reg_alloc<kRegsHigh>();
        constexpr int NCH = BN / 32;  // 32-column chunks of a row
        static_assert(BN % 32 == 0, "score tile in 32-column chunks");
        const int X = warp >> 2, qd = warp & 3;
        const int r = 32 * qd + lane;  // query row inside the tile
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * qd) << 16);
        const uint32_t s_addr = t_lane + X * S_STRIDE;
        const uint32_t o_addr = t_lane + O_COL + X * kPfDV;
        const float sc = p.scale_log2 * (p.q_scale ? __ldg(p.q_scale) : 1.f) * (p.k_scale ? __ldg(p.k_scale) : 1.f);
        const bool pos_scale = sc > 0.f;  // max on raw scores, one FFMA scales and shifts
        const float k_mul = pos_scale ? sc : 1.f;
        const float2 kk2 = make_float2(k_mul, k_mul);
        auto wait_warp = [&](uint32_t bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, wlim));
        };
        // scores of chunk i of the tile at key offset j0: scaled if the scale
        // is not positive, masked past the row's last key
        auto scale_mask = [&](int i, int j0, bool warp_full, int lim, uint32_t(&ra)[32]) {
            if (!pos_scale) {
#pragma unroll
                for (int c = 0; c < 32; ++c) ra[c] = __float_as_uint(__uint_as_float(ra[c]) * sc);
            }
            if (!warp_full) {
                const int lr = lim - (j0 + 32 * i);  // last visible column of the chunk
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c > lr) ra[c] = __float_as_uint(-INFINITY);
            }
        };
        auto chunk_max = [&](const uint32_t(&ra)[32]) {
            float m3[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float a = fmax3(__uint_as_float(ra[8 * q]), __uint_as_float(ra[8 * q + 1]),
                                      __uint_as_float(ra[8 * q + 2]));
                const float b = fmax3(__uint_as_float(ra[8 * q + 3]), __uint_as_float(ra[8 * q + 4]),
                                      __uint_as_float(ra[8 * q + 5]));
                m3[q] = fmax3(a, b, fmaxf(__uint_as_float(ra[8 * q + 6]), __uint_as_float(ra[8 * q + 7])));
            }
            return fmax3(fmaxf(m3[0], m3[1]), m3[2], m3[3]);
        };
        // P of a 32-key chunk, 2^(s k - base): 16-bit pairs into pw, sums
        // into la / lb
        auto exp_chunk = [&](const uint32_t(&ra)[32], float base, float2 &la, float2 &lb, uint32_t(&pw)[16]) {
            const float2 nb2 = make_float2(-base, -base);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float2 x =
                    __ffma2_rn(make_float2(__uint_as_float(ra[2 * e]), __uint_as_float(ra[2 * e + 1])), kk2, nb2);
                const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                if (e & 1)
                    lb = __fadd2_rn(lb, make_float2(p0, p1));
                else
                    la = __fadd2_rn(la, make_float2(p0, p1));
                pw[e] = pack2<TP>(p0, p1);  // P column: keys 2e, 2e+1 of the chunk
            }
        };
        bool ok = true;
        int t_base = 0;    // K/V tiles of earlier items
        int tx_base = 0;   // tiles of this block in earlier items
        int nx_items = 0;  // items with tiles processed by this block
        for (int k = 0; ok; ++k) {
            const int4 itm = take_item(k, ok);  // every thread reads the same slot
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || itm.x < 0) break;
            PfItem it;
            pf_item(p, itm, BN, it);
            const int n = it.n_tiles;
            const int h = X == 0 ? it.hA : it.hB;
            if (h < 0) {  // block B absent in this item
                t_base += n;
                continue;
            }
            const int pos = it.shift + it.i0 + r;
            const int lim = p.causal ? min(pos, it.kvb - 1) : it.kvb - 1;  // last visible key
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n; ++j) {
                const int t = t_base + j, tx = tx_base + j;
                const int j0 = j * BN;
                // S_X(t) complete, and with it PV_X(t-1)
                if (!wait_warp(b_sfull(X), tx & 1)) { ok = false; break; }
                tc_fence_after();
                const bool warp_full = __all_sync(0xffffffffu, j0 + BN - 1 <= lim);
                uint32_t rs[NCH][32];
#pragma unroll
                for (int i = 0; i < NCH; ++i) tmem_ld32(s_addr + 32 * i, rs[i]);
#pragma unroll
                for (int i = 0; i < NCH; ++i) tmem_wait_ld_regs(rs[i]);  // (the first waits for all)
                float mh = -INFINITY;
#pragma unroll
                for (int i = 0; i < NCH; ++i) {
                    scale_mask(i, j0, warp_full, lim, rs[i]);
                    mh = fmaxf(mh, chunk_max(rs[i]));
                }
                const float mt = pos_scale ? mh * sc : mh;
                float alpha = 1.f;
                if (mt > m_used + 8.f) {  // (first tile: from -inf)
                    alpha = fast_exp2(m_used - mt);
                    m_used = mt;
                    l *= alpha;
                }
                float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
                const float base = m_used == -INFINITY ? 0.f : m_used;
#pragma unroll
                for (int i = 0; i < NCH; ++i) {
                    uint32_t pw[16];
                    exp_chunk(rs[i], base, la, lb, pw);
                    tmem_st16(s_addr + 32 * i, pw);
                }
                l += (la.x + la.y) + (lb.x + lb.y);
                // rows of V past the sequence end may hold anything (even NaN):
                // block A zeroes them before its PV (block B's PV comes later in
                // issue order), so that P = 0 there cannot produce 0 * NaN
                if (X == 0 && j0 + BN > it.kvb) {
                    const int sv = t % SV, uv = t / SV;
                    if (!wait_warp(b_vfull(sv), uv & 1)) { ok = false; break; }
                    const int zs = max(it.kvb - j0, 0);
                    uint8_t *vbase = v_gen + sv * VB;
                    for (int q = r; q < (BN - zs) * 16; q += 128) {
                        const int row = zs + (q >> 4), chunk = q & 15;
                        *reinterpret_cast<uint4 *>(vbase + (chunk >> 3) * (BN * 128) + row * 128 + (chunk & 7) * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                // O_X *= alpha when the running max moved; PV_X(t-1) is
                // complete (S_X(t) is), and at the item's first tile O is
                // about to be overwritten anyway
                if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c = 0; c < kPfDV / 32; ++c) {
                        uint32_t ro[32];
                        tmem_ld32(o_addr + c * 32, ro);
                        tmem_wait_ld_regs(ro);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ro[e] = __float_as_uint(__uint_as_float(ro[e]) * alpha);
                        tmem_st32(o_addr + c * 32, ro);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(b_pfull(X));
            }
            if (!ok) break;
            // epilogue: after the block's last PV of the item, normalise O and
            // write it with the LSE
            const bool have = n > 0;
            if (have && !wait_warp(b_odone(X), nx_items & 1)) { ok = false; break; }
            tc_fence_after();
            const int qi = it.i0 + r;
            const int64_t grow = static_cast<int64_t>(it.orow_base) + r;
            const bool valid = qi < it.qb && grow >= 0 && grow < p.total_q;
            if (kDebugBounds && qi < it.qb) dbg_in(grow, 1, p.total_q, p.err);
            const float inv = l > 0.f ? (p.v_scale ? __ldg(p.v_scale) : 1.f) / l : 0.f;
            T *orow = static_cast<T *>(p.out) + (grow * p.Hqo + h) * kPfDV;
#pragma unroll
            for (int c = 0; c < kPfDV / 32; ++c) {
                uint32_t ro[32];
                if (have) {
                    tmem_ld32(o_addr + c * 32, ro);
                    tmem_wait_ld_regs(ro);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ro[e] = 0u;
                }
                if (valid) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        auto o = [&](int e) { return __uint_as_float(ro[q * 8 + e]) * inv; };
                        uint4 w = make_uint4(pack2<T>(o(0), o(1)), pack2<T>(o(2), o(3)), pack2<T>(o(4), o(5)),
                                             pack2<T>(o(6), o(7)));
                        *reinterpret_cast<uint4 *>(orow + c * 32 + q * 8) = w;
                    }
                }
            }
            if (valid) p.lse[grow * p.Hqo + h] = l > 0.f ? (m_used + fast_log2(l)) * kLn2 : -INFINITY;
            tc_fence_before();  // O read before the next item's first PV_X overwrites it
            t_base += n;
            tx_base += n;
            nx_items += have;
        }
        if (!ok) give_up();
        // (a tile abandoned after its P stores: they complete before the
        // allocation is freed; the whole warp gets here together)
        tmem_wait_st();
        tmem_wait_ld();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int DQK, bool F8>
static size_t prefill_smem_bytes() {
    constexpr int BN = PfCfg<DQK>::BN, SK = PfCfg<DQK>::SK, SV = PfCfg<DQK>::SV, ES = F8 ? 1 : 2;
    return 1024 + 2 * kPfRows * DQK * ES + SK * BN * DQK * ES + SV * BN * kPfDV * 2 + (F8 ? SV * BN * kPfDV : 0) +
           8 * (13 + 2 * SK + 2 * SV + (F8 ? 2 * SV : 0));
}

template <typename T, int DQK, int LAYOUT, bool F8 = false>
static int launch_prefill(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          const PrefillParams &p, dim3 grid, cudaStream_t st) {
    const size_t smem = prefill_smem_bytes<DQK, F8>();
    auto kern = prefill_tc_kernel<T, DQK, LAYOUT, F8>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PKV_ERR_CUDA;
    {
        // the register split draws on the registers the CTA is launched with:
        // refuse to launch if the compiled kernel was given fewer (the
        // softmax warps' setmaxnreg.inc would wait for registers forever)
        static int ok = -1;
        if (ok < 0) {
            cudaFuncAttributes fa;
            if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return PKV_ERR_CUDA;
            ok = fa.numRegs * PfRoles<DQK>::kThreads >= 128 * kRegsLow + 256 * kRegsHigh ? 1 : 0;
        }
        if (!ok) return PKV_ERR_UNSUPPORTED;
    }
    // launched as the plan kernel's dependent: the prologue (barriers, tensor
    // memory, descriptor prefetch) overlaps the plan kernel
    if (launch_dependent(kern, grid, dim3(PfRoles<DQK>::kThreads), smem, st, tq, tk, tv, p) != cudaSuccess)
        return PKV_ERR_CUDA;
    return PKV_OK;
}

// ---- E4M3 (FP8) inputs --------------------------------------------------------
// The tensor-core path multiplies 16-bit operands.  E4M3 query rows and cache
// rows are widened into the workspace first -- exactly: every E4M3 value is a
// bf16 and an fp16 value -- the caches packed request by request as
// contiguous [rows, Hkv, d] tensors (request b at rows cu_kv[b] ..); the
// scale tensors are applied inside the main kernel.
struct WidenKvParams {
    const uint8_t *src[2];  // K, V caches, one byte per element
    int64_t page_stride[2];
    int d[2];
    void *dst[2];           // widened K, V: [rows, Hkv, d] of the 16-bit type
    int64_t max_num_pages;
    const int32_t *block_tables;
    int64_t bt_stride;
    const int32_t *seq_lens_kv;
    const int32_t *cu_kv;   // from the plan kernel
    int max_kv, Hkv, page_shift;
    int32_t *err;
};
constexpr int kWidenTok = 32;  // keys per CTA of the cache widening

// CTA (key block, request, K or V): every 16-byte source chunk of its keys
// becomes 32 bytes of the packed 16-bit tensor.  A page id outside the pool
// flags PKV_DEV_ERR_PAGE and its rows widen to zeros, as the 16-bit path's
// zero-filled rows.
template <typename T, int LAYOUT>
__global__ void __launch_bounds__(256) prefill_widen_kv_kernel(const WidenKvParams w) {
    pdl_wait();  // cu_kv
    pdl_launch_dependents();
    const int b = blockIdx.y, z = blockIdx.z;
    const int kvb = min(max(w.seq_lens_kv[b], 0), w.max_kv);
    const int j0 = blockIdx.x * kWidenTok;
    if (j0 >= kvb) return;
    const int d = w.d[z], CH = d / 16;
    const int S = 1 << w.page_shift;
    const int64_t row0 = w.cu_kv[b];
    const int n = min(kWidenTok, kvb - j0) * w.Hkv * CH;
    const int32_t *bt = w.block_tables + b * w.bt_stride;
    T *dst = static_cast<T *>(w.dst[z]);
    for (int idx = threadIdx.x; idx < n; idx += blockDim.x) {
        const int c = idx % CH, rest = idx / CH;
        const int h = rest % w.Hkv, j = j0 + rest / w.Hkv;
        const int page = bt[j >> w.page_shift];
        uint4 raw = make_uint4(0u, 0u, 0u, 0u);
        if (page < 0 || page >= w.max_num_pages) {
            if (z == 0 && h == 0 && c == 0) set_err(w.err, PKV_DEV_ERR_PAGE);
        } else {
            raw = *reinterpret_cast<const uint4 *>(
                w.src[z] + kv_row_offset<LAYOUT>(page, w.page_stride[z], h, j & (S - 1), w.Hkv, S, d) + c * 16);
        }
        const uint32_t x[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = widen_e4m3x2<T>(x[i] & 0xffffu);
            o[2 * i + 1] = widen_e4m3x2<T>(x[i] >> 16);
        }
        uint4 *out = reinterpret_cast<uint4 *>(dst + ((row0 + j) * w.Hkv + h) * d + c * 16);
        out[0] = make_uint4(o[0], o[1], o[2], o[3]);
        out[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// n16 chunks of 16 E4M3 values (the query rows) -> 16-bit, in order.
template <typename T>
__global__ void __launch_bounds__(256) widen_rows_kernel(const uint8_t *__restrict__ src, T *__restrict__ dst,
                                                         int64_t n16) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 raw = reinterpret_cast<const uint4 *>(src)[i];
        const uint32_t x[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            o[2 * k] = widen_e4m3x2<T>(x[k] & 0xffffu);
            o[2 * k + 1] = widen_e4m3x2<T>(x[k] >> 16);
        }
        uint4 *out = reinterpret_cast<uint4 *>(dst) + 2 * i;
        out[0] = make_uint4(o[0], o[1], o[2], o[3]);
        out[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// What an E4M3 call adds to the 16-bit path.
struct PrefillFp8 {
    const float *q_scale = nullptr, *k_scale = nullptr, *v_scale = nullptr;
    bool direct = false;             // E4M3 query and caches read as they are (kind::f8f6f4 QK)
    const uint8_t *q_src = nullptr;  // E4M3 query rows, widened into the call's `q` first
    bool kv8 = false;                // widen the paged caches after the plan kernel
    WidenKvParams widen{};           // (cu_kv and err filled in by prefill_impl)
    int layout = PKV_HND;            // of the E4M3 caches
};

template <typename T>
static int dispatch_prefill(int d_qk, int layout, const CUtensorMap &tq, const CUtensorMap &tk,
                            const CUtensorMap &tv, const PrefillParams &p, dim3 grid, cudaStream_t st,
                            bool f8_direct) {
    if (f8_direct)  // (d_qk 128)
        return layout == PKV_HND ? launch_prefill<T, 128, PKV_HND, true>(tq, tk, tv, p, grid, st)
                                 : launch_prefill<T, 128, PKV_NHD, true>(tq, tk, tv, p, grid, st);
    if (d_qk == 128)
        return layout == PKV_HND ? launch_prefill<T, 128, PKV_HND>(tq, tk, tv, p, grid, st)
                                 : launch_prefill<T, 128, PKV_NHD>(tq, tk, tv, p, grid, st);
    return layout == PKV_HND ? launch_prefill<T, 192, PKV_HND>(tq, tk, tv, p, grid, st)
                             : launch_prefill<T, 192, PKV_NHD>(tq, tk, tv, p, grid, st);
}

// K or V cache as a 4-D tensor map whose box is one 128-byte d-atom (64
// 16-bit or 128 one-byte elements, es bytes each) of `rows` consecutive
// slots of one (page, kv head).
static bool cache_tmap(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int layout, int d,
                       int page_size, int num_kv_heads, int64_t page_stride, int64_t num_pages,
                       int rows, int es = 2) {
    uint64_t dims[4], strides[3];
    uint32_t box[4];
    dims[0] = d;
    box[0] = 128 / es;
    strides[0] = static_cast<uint64_t>(d) * es;
    if (layout == PKV_HND) {
        dims[1] = page_size;
        dims[2] = num_kv_heads;
        strides[1] = static_cast<uint64_t>(page_size) * d * es;
        box[1] = rows;
        box[2] = 1;
    } else {
        dims[1] = num_kv_heads;
        dims[2] = page_size;
        strides[1] = static_cast<uint64_t>(num_kv_heads) * d * es;
        box[1] = 1;
        box[2] = rows;
    }
    dims[3] = static_cast<uint64_t>(num_pages);
    strides[2] = static_cast<uint64_t>(page_stride) * es;
    box[3] = 1;
    return encode_tmap(m, base, dt, 4, dims, strides, box);
}

// A paged cache as a 5-D map whose box holds every 128-byte atom of `rows`
// slots of one page: dims (64 elements, 8 slots, d / 64 atoms, page_size / 8
// slot groups, u = page * ratio + kv head), so one copy fills
// [group][atom][8 rows][128 B] of shared memory -- a 128-byte-swizzled
// K-major layout with 8-row groups QA * 1024 bytes apart.  The atom
// dimension's stride (128 B) is below the slot dimension's; the driver
// accepts the map.  Possible when the page stride is a multiple of
// page_size * d (HND) or d (NHD) elements, so that (page, head) is one index
// u, and u fits an int32 coordinate.  Used for d_qk 192 (three atoms, one
// copy instead of three): at d_qk 128 the two-atom box measured slower.
static bool cache_tmap5_ok(int layout, int d, int S, int hkv, int64_t P, int64_t pages, int rows, int &ratio) {
    if (d != 192 || S % 8 || rows % 8) return false;
    const int64_t unit = layout == PKV_HND ? static_cast<int64_t>(S) * d : d;
    if (P % unit) return false;
    const int64_t r = P / unit;
    if ((pages + 1) * r + hkv >= (1LL << 31)) return false;
    ratio = static_cast<int>(r);
    return true;
}
static bool cache_tmap5(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int layout, int d, int S, int hkv,
                        int ratio, int64_t pages, int rows) {
    uint64_t dims[5] = {64, 8, static_cast<uint64_t>(d / 64), static_cast<uint64_t>(S / 8),
                        static_cast<uint64_t>(pages > 0 ? pages * ratio : 1)};
    uint64_t strides[4];
    if (layout == PKV_HND) {
        strides[0] = static_cast<uint64_t>(d) * 2;
        strides[1] = 128;
        strides[2] = 8ull * d * 2;
        strides[3] = static_cast<uint64_t>(S) * d * 2;
    } else {
        strides[0] = static_cast<uint64_t>(hkv) * d * 2;
        strides[1] = 128;
        strides[2] = 8ull * hkv * d * 2;
        strides[3] = static_cast<uint64_t>(d) * 2;
    }
    uint32_t box[5] = {64, 8, static_cast<uint32_t>(d / 64), static_cast<uint32_t>(rows / 8), 1};
    return encode_tmap(m, base, dt, 5, dims, strides, box);
}

// Contiguous K or V ([rows, num_kv_heads, d], row stride in elements) as the
// NHD map of a single page holding every row; a box is one 64-element d-atom
// of `box_rows` consecutive rows of one kv head.
static bool contiguous_tmap(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int d, int num_kv_heads,
                            int64_t row_stride, int64_t rows, int box_rows) {
    uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(num_kv_heads),
                        static_cast<uint64_t>(rows > 0 ? rows : 1), 1};
    uint64_t strides[3] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(row_stride) * 2,
                           static_cast<uint64_t>(row_stride) * 2 * (rows > 0 ? rows : 1)};
    uint32_t box[4] = {64, 1, static_cast<uint32_t>(box_rows), 1};
    return encode_tmap(m, base, dt, 4, dims, strides, box);
}

// workspace: cu_q[B+1], cu_items[B+1], cu_kv[B+1], then the work-item
// counter of the persistent kernel
static size_t prefill_ws_bytes(int B) {
    return 3 * round_up(static_cast<size_t>(B + 1) * sizeof(int32_t), 256) + 256;
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

static int prefill_impl(const void *q, int64_t total_q, const void *k_cache,
                             const void *v_cache, int64_t k_page_stride, int64_t v_page_stride,
                             int64_t max_num_pages, float scale, void *workspace,
                             size_t workspace_bytes, int32_t max_token_per_sequence,
                             int32_t max_sequence_kv, const int32_t *actual_seq_lens_q,
                             const int32_t *actual_seq_lens_kv, const int32_t *block_tables,
                             int32_t block_table_stride, int32_t batch_size, int32_t causal,
                             int32_t num_qo_heads, int32_t num_kv_heads, int32_t d_qk,
                             int32_t d_vo, int32_t page_size, int32_t layout, int32_t dtype,
                             void *out, float *lse, int32_t *err_word, void *stream,
                             const int32_t *off_q, const int32_t *off_o, const int32_t *off_k,
                             const int32_t *off_v, PrefillFp8 *f8 = nullptr) {
    // no block table: contiguous K/V of max_num_pages rows, page strides are row strides
    const bool contiguous = block_tables == nullptr;
    if (contiguous) {
        if (layout != PKV_NHD) return PKV_ERR_INVALID_ARG;  // [rows, heads, d] is token-major
        page_size = 1;
        block_table_stride = max_sequence_kv;
    }
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (dtype != PKV_F16 && dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    if (batch_size < 0 || num_qo_heads < 1 || num_kv_heads < 1 || max_token_per_sequence < 0 ||
        max_sequence_kv < 0 || max_num_pages < 0 || block_table_stride < 0 || total_q < 0)
        return PKV_ERR_INVALID_ARG;
    if (num_qo_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
    if ((d_qk != 128 && d_qk != 192) || d_vo != 128) return PKV_ERR_UNSUPPORTED;
    if (!contiguous && (ilog2_exact(page_size) < 3 || page_size > 256)) return PKV_ERR_UNSUPPORTED;
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
    if (!q || !k_cache || !v_cache || !actual_seq_lens_q || !actual_seq_lens_kv || !out || !lse)
        return PKV_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (k_page_stride % 8) || (v_page_stride % 8))
        return PKV_ERR_INVALID_ARG;
    if (!workspace) return PKV_ERR_NULL;
    if (workspace_bytes < prefill_ws_bytes(batch_size) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255))
        return PKV_ERR_WORKSPACE;

    // (the E4M3 query and caches read as they are: one-byte elements)
    const bool f8d = f8 && f8->direct;
    const int es = f8d ? 1 : 2;
    const CUtensorMapDataType tdt = f8d ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                        : (dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    const int bn = pf_bn(d_qk);
    const int rows = pf_box_rows(page_size, bn);
    CUtensorMap tq, tk, tv;
    int k5 = 0, k5_ratio = 0;
    {
        // (128-byte atom elements, token rows, atoms, qo heads): one box is the
        // two heads' Q blocks, [head][atom][row][128 B]
        uint64_t dims[4] = {static_cast<uint64_t>(128 / es), static_cast<uint64_t>(total_q > 0 ? total_q : 1),
                            static_cast<uint64_t>(d_qk * es / 128), static_cast<uint64_t>(num_qo_heads)};
        uint64_t strides[3] = {static_cast<uint64_t>(num_qo_heads) * d_qk * es, 128,
                               static_cast<uint64_t>(d_qk) * es};
        uint32_t box[4] = {static_cast<uint32_t>(128 / es), static_cast<uint32_t>(kPfRows),
                           static_cast<uint32_t>(d_qk * es / 128), 2};
        if (!encode_tmap(&tq, q, tdt, 4, dims, strides, box)) return PKV_ERR_CUDA;
    }
    if (f8d) {
        if (contiguous || !cache_tmap(&tk, k_cache, tdt, layout, d_qk, page_size, num_kv_heads, k_page_stride,
                                      max_num_pages, rows, 1) ||
            !cache_tmap(&tv, v_cache, tdt, layout, d_vo, page_size, num_kv_heads, v_page_stride, max_num_pages,
                        rows, 1))
            return PKV_ERR_CUDA;
    } else if (contiguous) {
        if (!contiguous_tmap(&tk, k_cache, tdt, d_qk, num_kv_heads, k_page_stride, max_num_pages, bn) ||
            !contiguous_tmap(&tv, v_cache, tdt, d_vo, num_kv_heads, v_page_stride, max_num_pages, bn))
            return PKV_ERR_CUDA;
    } else {
        k5 = cache_tmap5_ok(layout, d_qk, page_size, num_kv_heads, k_page_stride, max_num_pages, rows, k5_ratio) ? 1
                                                                                                                   : 0;
        if (!(k5 ? cache_tmap5(&tk, k_cache, tdt, layout, d_qk, page_size, num_kv_heads, k5_ratio, max_num_pages, rows)
                 : cache_tmap(&tk, k_cache, tdt, layout, d_qk, page_size, num_kv_heads, k_page_stride, max_num_pages,
                              rows)) ||
            !cache_tmap(&tv, v_cache, tdt, layout, d_vo, page_size, num_kv_heads, v_page_stride, max_num_pages, rows))
            return PKV_ERR_CUDA;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int launches = 0;
    if (f8 && f8->q_src) {  // E4M3 query rows -> the 16-bit rows `q` points at
        const int64_t n16 = total_q * num_qo_heads * d_qk / 16;
        const int64_t cap = 8LL * num_sms();
        const unsigned blocks = static_cast<unsigned>((n16 + 255) / 256 < cap ? (n16 + 255) / 256 : cap);
        if (dtype == PKV_BF16)
            widen_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, st>>>(
                f8->q_src, static_cast<__nv_bfloat16 *>(const_cast<void *>(q)), n16);
        else
            widen_rows_kernel<__half><<<blocks, 256, 0, st>>>(f8->q_src, static_cast<__half *>(const_cast<void *>(q)),
                                                              n16);
        ++launches;
    }
    const size_t cu_bytes = round_up(static_cast<size_t>(batch_size + 1) * sizeof(int32_t), 256);
    int32_t *cu_q = static_cast<int32_t *>(workspace);
    int32_t *cu_items = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + cu_bytes);
    int32_t *cu_kv = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + 2 * cu_bytes);
    int *work_counter = reinterpret_cast<int *>(static_cast<char *>(workspace) + 3 * cu_bytes);
    const int pairs = (num_qo_heads / num_kv_heads + 1) / 2;  // head pairs per kv head
    prefill_plan_kernel<<<1, 32, 0, st>>>(actual_seq_lens_q, actual_seq_lens_kv, batch_size, num_kv_heads * pairs,
                                          max_token_per_sequence, max_sequence_kv, cu_q, cu_items, cu_kv, err_word,
                                          work_counter);
    ++launches;
    if (f8 && f8->kv8) {
        // widen the E4M3 caches (needs cu_kv); the main kernel then reads them
        // as contiguous K/V
        f8->widen.cu_kv = cu_kv;
        f8->widen.err = err_word;
        const dim3 wgrid(static_cast<unsigned>((max_sequence_kv + kWidenTok - 1) / kWidenTok),
                         static_cast<unsigned>(batch_size), 2);
        if (max_sequence_kv > 0) {
            auto wk = dtype == PKV_BF16
                          ? (f8->layout == PKV_HND ? prefill_widen_kv_kernel<__nv_bfloat16, PKV_HND>
                                                   : prefill_widen_kv_kernel<__nv_bfloat16, PKV_NHD>)
                          : (f8->layout == PKV_HND ? prefill_widen_kv_kernel<__half, PKV_HND>
                                                   : prefill_widen_kv_kernel<__half, PKV_NHD>);
            if (launch_dependent(wk, wgrid, dim3(256), 0, st, f8->widen) != cudaSuccess) return PKV_ERR_CUDA;
            ++launches;
        }
    }
    PrefillParams p;
    p.max_num_pages = max_num_pages;
    p.total_q = total_q;
    p.scale_log2 = scale * kLog2e;
    p.seq_lens_q = actual_seq_lens_q;
    p.seq_lens_kv = actual_seq_lens_kv;
    p.cu_q = cu_q;
    p.cu_items = cu_items;
    p.block_tables = block_tables;
    p.bt_stride = block_table_stride;
    p.B = batch_size;
    p.causal = causal ? 1 : 0;
    p.Hqo = num_qo_heads;
    p.Hkv = num_kv_heads;
    p.group = num_qo_heads / num_kv_heads;
    p.pairs = pairs;
    p.contiguous = contiguous ? 1 : 0;
    p.cu_kv = cu_kv;
    p.off_q = off_q;
    p.off_o = off_o;
    p.off_k = off_k;
    p.off_v = off_v;
    p.page_shift = ilog2_exact(page_size);
    p.max_q = max_token_per_sequence;
    p.max_kv = max_sequence_kv;
    p.work_counter = work_counter;
    p.q_scale = f8 ? f8->q_scale : nullptr;
    p.k_scale = f8 ? f8->k_scale : nullptr;
    p.v_scale = f8 ? f8->v_scale : nullptr;
    p.out = out;
    p.lse = lse;
    p.err = err_word;
    p.wait_ns = wait_limit_ns();
    p.k5 = k5;
    p.k5_ratio = k5_ratio;
    const int n_qt = (max_token_per_sequence + kPfRows - 1) / kPfRows;
    const int64_t items = static_cast<int64_t>(n_qt) * num_kv_heads * pairs * batch_size;
    if (n_qt > 0) {
        // persistent: one CTA per SM (the shared-memory footprint allows one)
        const int64_t ctas = items < num_sms() ? items : num_sms();
        dim3 grid(static_cast<unsigned>(ctas));
        int rc = dtype == PKV_BF16 ? dispatch_prefill<__nv_bfloat16>(d_qk, layout, tq, tk, tv, p, grid, st, f8d)
                                   : dispatch_prefill<__half>(d_qk, layout, tq, tk, tv, p, grid, st, f8d);
        if (rc != PKV_OK) return rc;
        ++launches;
    }
    note_launches(launches);
    return launch_status();
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
    const CallRange nvtx_range("paged_prefill");
    return prefill_impl(q, total_q, k_cache, v_cache, k_page_stride, v_page_stride, max_num_pages, scale,
                        workspace, workspace_bytes, max_token_per_sequence, max_sequence_kv, actual_seq_lens_q,
                        actual_seq_lens_kv, block_tables, block_table_stride, batch_size, causal, num_qo_heads,
                        num_kv_heads, d_qk, d_vo, page_size, layout, dtype, out, lse, err_word, stream, nullptr,
                        nullptr, nullptr, nullptr);
}

extern "C" int paged_prefill_ex(const void *q, int64_t total_q, const void *k_cache,
                                const void *v_cache, int64_t k_page_stride, int64_t v_page_stride,
                                int64_t max_num_pages, float scale, void *workspace,
                                size_t workspace_bytes, int32_t max_token_per_sequence,
                                int32_t max_sequence_kv, const int32_t *actual_seq_lens_q,
                                const int32_t *actual_seq_lens_kv, const int32_t *block_tables,
                                int32_t block_table_stride, int32_t batch_size, int32_t causal,
                                int32_t num_qo_heads, int32_t num_kv_heads, int32_t d_qk,
                                int32_t d_vo, int32_t page_size, int32_t layout, int32_t dtype,
                                void *out, float *lse, const int32_t *batch_offsets_q,
                                const int32_t *batch_offsets_o, const int32_t *batch_offsets_k,
                                const int32_t *batch_offsets_v, int32_t *err_word, void *stream) {
    const CallRange nvtx_range("paged_prefill_ex");
    if (block_tables && (batch_offsets_k || batch_offsets_v)) return PKV_ERR_INVALID_ARG;  // pages place K/V
    return prefill_impl(q, total_q, k_cache, v_cache, k_page_stride, v_page_stride, max_num_pages, scale,
                        workspace, workspace_bytes, max_token_per_sequence, max_sequence_kv, actual_seq_lens_q,
                        actual_seq_lens_kv, block_tables, block_table_stride, batch_size, causal, num_qo_heads,
                        num_kv_heads, d_qk, d_vo, page_size, layout, dtype, out, lse, err_word, stream,
                        batch_offsets_q, batch_offsets_o, batch_offsets_k, batch_offsets_v);
}

// ---- E4M3 (FP8) query and/or caches ----------------------------------------------

// Workspace of paged_prefill_fp8: the 16-bit path's, then the widened query
// rows (E4M3 query) and the widened, packed K and V (E4M3 caches; room for
// batch_size * max_sequence_kv keys, the most the lengths allow).
// An E4M3 query with E4M3 caches at d_qk = d_vo = 128 is read as it is (the
// kind::f8f6f4 kernel): nothing is widened into the workspace.
static bool prefill_fp8_direct(bool q8, bool kv8, int d_qk, int d_vo) { return q8 && kv8 && d_qk == 128 && d_vo == 128; }

static size_t prefill_fp8_ws_bytes(int B, int Hqo, int Hkv, int max_kv, int64_t total_q, int d_qk, int d_vo,
                                   bool q8, bool kv8, size_t *q_off, size_t *k_off, size_t *v_off) {
    size_t off = prefill_ws_bytes(B);
    if (prefill_fp8_direct(q8, kv8, d_qk, d_vo)) {
        *q_off = *k_off = *v_off = off;
        return off;
    }
    *q_off = off;
    if (q8) off += round_up(static_cast<size_t>(total_q) * Hqo * d_qk * 2, 256);
    *k_off = off;
    const size_t rows = static_cast<size_t>(B) * max_kv;
    if (kv8) off += round_up(rows * Hkv * d_qk * 2, 256);
    *v_off = off;
    if (kv8) off += round_up(rows * Hkv * d_vo * 2, 256);
    return off;
}

extern "C" size_t paged_prefill_fp8_workspace_size(int32_t batch_size, int32_t num_qo_heads, int32_t num_kv_heads,
                                                   int32_t max_token_per_sequence, int32_t max_sequence_kv,
                                                   int64_t total_q, int32_t d_qk, int32_t d_vo, int32_t q_dtype,
                                                   int32_t kv_dtype) {
    if (batch_size < 0 || num_qo_heads < 1 || num_kv_heads < 1 || max_token_per_sequence < 0 ||
        max_sequence_kv < 0 || total_q < 0 || d_qk < 1 || d_vo < 1)
        return 0;
    size_t a, b, c;
    return prefill_fp8_ws_bytes(batch_size, num_qo_heads, num_kv_heads, max_sequence_kv, total_q, d_qk, d_vo,
                                q_dtype == PKV_E4M3, kv_dtype == PKV_E4M3, &a, &b, &c);
}

extern "C" int paged_prefill_fp8(const void *q, int64_t total_q, const void *k_cache, const void *v_cache,
                                 int64_t k_page_stride, int64_t v_page_stride, int64_t max_num_pages, float scale,
                                 const float *q_scale, const float *k_scale, const float *v_scale, void *workspace,
                                 size_t workspace_bytes, int32_t max_token_per_sequence, int32_t max_sequence_kv,
                                 const int32_t *actual_seq_lens_q, const int32_t *actual_seq_lens_kv,
                                 const int32_t *block_tables, int32_t block_table_stride, int32_t batch_size,
                                 int32_t causal, int32_t num_qo_heads, int32_t num_kv_heads, int32_t d_qk,
                                 int32_t d_vo, int32_t page_size, int32_t layout, int32_t q_dtype,
                                 int32_t kv_dtype, int32_t out_dtype, void *out, float *lse, int32_t *err_word,
                                 void *stream) {
    const CallRange nvtx_range("paged_prefill_fp8");
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16) return PKV_ERR_INVALID_ARG;
    const bool q8 = q_dtype == PKV_E4M3, kv8 = kv_dtype == PKV_E4M3;
    if ((!q8 && q_dtype != out_dtype) || (!kv8 && kv_dtype != out_dtype)) return PKV_ERR_INVALID_ARG;
    if (!block_tables) return PKV_ERR_INVALID_ARG;  // paged caches
    if (batch_size < 0 || num_qo_heads < 1 || num_kv_heads < 1 || max_token_per_sequence < 0 ||
        max_sequence_kv < 0 || max_num_pages < 0 || block_table_stride < 0 || total_q < 0)
        return PKV_ERR_INVALID_ARG;
    if (layout != PKV_NHD && layout != PKV_HND) return PKV_ERR_INVALID_ARG;
    if (num_qo_heads % num_kv_heads) return PKV_ERR_INVALID_ARG;
    if ((d_qk != 128 && d_qk != 192) || d_vo != 128) return PKV_ERR_UNSUPPORTED;
    if (ilog2_exact(page_size) < 3 || page_size > 256) return PKV_ERR_UNSUPPORTED;
    if (batch_size > 65535 || static_cast<int64_t>(batch_size) * max_sequence_kv > 0x7fffffff)
        return PKV_ERR_UNSUPPORTED;
    if (k_page_stride < static_cast<int64_t>(num_kv_heads) * page_size * d_qk ||
        v_page_stride < static_cast<int64_t>(num_kv_heads) * page_size * d_vo ||
        static_cast<int64_t>(block_table_stride) * page_size < max_sequence_kv)
        return PKV_ERR_INVALID_ARG;
    if (batch_size == 0 || total_q == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !actual_seq_lens_q || !actual_seq_lens_kv || !out || !lse)
        return PKV_ERR_NULL;
    // 16-byte page starts and rows (an E4M3 element is one byte)
    if (kv8 && (!aligned16(k_cache) || !aligned16(v_cache) || (k_page_stride % 16) || (v_page_stride % 16)))
        return PKV_ERR_INVALID_ARG;
    if (q8 && !aligned16(q)) return PKV_ERR_INVALID_ARG;
    size_t q_off, k_off, v_off;
    const size_t need = prefill_fp8_ws_bytes(batch_size, num_qo_heads, num_kv_heads, max_sequence_kv, total_q,
                                             d_qk, d_vo, q8, kv8, &q_off, &k_off, &v_off);
    if (!workspace) return PKV_ERR_NULL;
    if (workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255)) return PKV_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    PrefillFp8 f8;
    f8.q_scale = q_scale;
    f8.k_scale = k_scale;
    f8.v_scale = v_scale;
    if (prefill_fp8_direct(q8, kv8, d_qk, d_vo)) {
        f8.direct = true;
        return prefill_impl(q, total_q, k_cache, v_cache, k_page_stride, v_page_stride, max_num_pages, scale,
                            workspace, workspace_bytes, max_token_per_sequence, max_sequence_kv, actual_seq_lens_q,
                            actual_seq_lens_kv, block_tables, block_table_stride, batch_size, causal, num_qo_heads,
                            num_kv_heads, d_qk, d_vo, page_size, layout, out_dtype, out, lse, err_word, stream,
                            nullptr, nullptr, nullptr, nullptr, &f8);
    }
    const void *qq = q;
    if (q8) {
        f8.q_src = static_cast<const uint8_t *>(q);
        qq = ws + q_off;
    }
    if (!kv8)
        return prefill_impl(qq, total_q, k_cache, v_cache, k_page_stride, v_page_stride, max_num_pages, scale,
                            workspace, workspace_bytes, max_token_per_sequence, max_sequence_kv,
                            actual_seq_lens_q, actual_seq_lens_kv, block_tables, block_table_stride, batch_size,
                            causal, num_qo_heads, num_kv_heads, d_qk, d_vo, page_size, layout, out_dtype, out, lse,
                            err_word, stream, nullptr, nullptr, nullptr, nullptr, &f8);
    f8.kv8 = true;
    f8.layout = layout;
    WidenKvParams &w = f8.widen;
    w.src[0] = static_cast<const uint8_t *>(k_cache);
    w.src[1] = static_cast<const uint8_t *>(v_cache);
    w.page_stride[0] = k_page_stride;
    w.page_stride[1] = v_page_stride;
    w.d[0] = d_qk;
    w.d[1] = d_vo;
    w.dst[0] = ws + k_off;
    w.dst[1] = ws + v_off;
    w.max_num_pages = max_num_pages;
    w.block_tables = block_tables;
    w.bt_stride = block_table_stride;
    w.seq_lens_kv = actual_seq_lens_kv;
    w.max_kv = max_sequence_kv;
    w.Hkv = num_kv_heads;
    w.page_shift = ilog2_exact(page_size);
    // the main kernel reads the widened caches as contiguous K/V: [rows, Hkv, d]
    const int64_t rows = static_cast<int64_t>(batch_size) * max_sequence_kv;
    return prefill_impl(qq, total_q, ws + k_off, ws + v_off, static_cast<int64_t>(num_kv_heads) * d_qk,
                        static_cast<int64_t>(num_kv_heads) * d_vo, rows, scale, workspace, workspace_bytes,
                        max_token_per_sequence, max_sequence_kv, actual_seq_lens_q, actual_seq_lens_kv, nullptr, 0,
                        batch_size, causal, num_qo_heads, num_kv_heads, d_qk, d_vo, 1, PKV_NHD, out_dtype, out, lse,
                        err_word, stream, nullptr, nullptr, nullptr, nullptr, &f8);
}
