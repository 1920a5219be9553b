// fmha_bwd_d256_sm103.cuh -- attention backward for head size 256 on sm_103a.
//
// The same operation as the D <= 128 backward (the Pallas page's
// `_attention_bwd`: delta = rowsum(O * dO) from the given O, a dQ pass over the
// KV tiles of each query tile and a dK/dV pass over the query tiles of each KV
// tile, dQ and dK scaled), for D = 256, which the page's benchmark sweeps beside
// 64 and 128.
//
// At D = 256 one 128-row gradient accumulator takes 256 tensor-memory columns:
// dK and dV of one key tile would fill all 512 and leave none for S^T and dP^T,
// and K, V (64 KB each) with one stage of Q and dO (128 KB) would not fit in
// shared memory either.  So the work runs as three launches of one kernel, each
// with a single accumulator (`Role`):
//   dV   rows = 128 keys:    S^T = K Q^T;  P^T = 2^(S^T scale log2e - lse2);
//                            dV += P^T dO                                2 products
//   dK   rows = 128 keys:    S^T = K Q^T,  dP^T = V dO^T;
//                            dS^T = P^T (dP^T - delta);  dK += dS^T Q    3 products
//   dQ   rows = 128 queries: S = Q K^T,  dP = dO V^T;
//                            dS = P (dP - delta);  dQ += dS K            3 products
// S and dP are recomputed by each launch that needs them: 8 products of
// 128 x 128 x 256 per (query tile, key tile) pair against the 5 of the gradient.
//
// The rows' own operands (K; K and V; Q and dO) stay in shared memory for a work
// item (64 KB each, four 64-column swizzled chunks).  The other side streams in
// halves of 128 rows x 128 columns (32 KB) through a ring, in the order the MMAs
// read them, each half read by one product and released by its commit:
//   3-product roles:  X1_0, X2_0, then per step n: X1_{n+1}, Y_n, X2_{n+1}
//   dV:               X1_0, X1_1, then per step n: Y_n, X1_{n+2}
// (X1 = the streamed operand of S, X2 = that of dP, Y = the accumulator's B
// operand; each as its two halves of the head dimension).  The producer and the
// MMA warp both walk this one sequence (`entry_of`), so they cannot disagree.
//
// Tensor memory: S at columns 0-127; dP (or, for dV, a second S buffer) at
// 128-255; the accumulator at 256-511.  dS is packed over dP and P (dV) over its
// S buffer, each group of elementwise warps over the start of its own columns,
// as in the D <= 128 kernels.
//
// Warps (352 threads): eight elementwise warps (TMEM lane quarter x column half),
// the MMA warp, the TMA warp (then the release warp of the abort path) and a ring
// watcher.  The elementwise warps hand over to the MMA warp through hardware named
// barriers.  In the dK and dQ launches so does the watcher, for each ring half, so
// within an item the MMA warp polls no mbarrier (such a poll would first wait for
// its queued MMAs to drain) and each half's products start as soon as it lands;
// in the dV launch (deeper ring, usually full ahead) the MMA warp polls both
// halves of a product once, which measured faster there, and the watcher idles.
// Every mbarrier wait is bounded.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "fmha_bwd_sm103.cuh"

namespace attn {
namespace bwd256 {

using bwd::BwdParams;
using bwd::kBarReadyThreads;
using bwd::kCols;
using bwd::kComputeWarps;
using bwd::kLoadWarp;
using bwd::kMmaWarp;
constexpr int kWatchWarp = kLoadWarp + 1;
constexpr int kThreads = 32 * (kWatchWarp + 1);  // 352

enum Role : int { kRoleDV = 0, kRoleDK = 1, kRoleDQ = 2 };

constexpr int kD = 256;
constexpr int kChunk = kHalfBytes;  // 128 rows x 64 columns: 16 KB
constexpr int kTile = 4 * kChunk;   // 128 rows x 256 columns: 64 KB
constexpr int kHalf = 2 * kChunk;   // 128 rows x 128 columns: 32 KB, one ring slot
constexpr int kMaxSlots = 5;

// Named barriers (elementwise warps arrive, the MMA warp syncs).  3-product
// roles: S read out (2) and dS stored (3).  dV: P stored, alternating 2 and 3 by
// step parity -- the elementwise warps may store P_{n+1} before the MMA warp has
// synced for P_n (S_{n+1} is issued before that sync), so consecutive steps must
// not share a barrier; step n+2 needs S_{n+2}, issued only after the sync for n.
constexpr uint32_t kBarSRead = 2, kBarDsReady = 3, kBarP0 = 2;
// Ring hand-off: the watcher warp polls each slot's "landed" mbarrier and arrives
// on that slot's named barrier (kBarRing0 + slot), where the MMA warp syncs before
// the half's MMAs: an mbarrier poll by the MMA warp itself would first wait for its
// queued MMAs to drain.  Fill f + kSlots reuses slot f's barrier only after the MMA
// warp consumed fill f (its commit frees the slot for the refill), so generations
// never mix.
constexpr uint32_t kBarRing0 = 4, kBarRingThreads = 64;

enum : int {
    B_A1FULL = 0,                  // the item's first resident tile landed
    B_A1EMPTY,                     // its last S completed: the tile may be replaced
    B_A2FULL,
    B_A2EMPTY,                     // its last dP completed
    B_FULL,                        // [slot]
    B_EMPTY = B_FULL + kMaxSlots,  // [slot]
    B_SFULL = B_EMPTY + kMaxSlots, // [S buffer]
    B_DPFULL = B_SFULL + 2,
    B_ACCDONE,                     // the item's last accumulator product completed
    B_ITEMFULL,                    // [2] next work item published
    B_ITEMEMPTY = B_ITEMFULL + 2,  // [2] read by the MMA warp and the 8 elementwise warps
    B_MMADONE = B_ITEMEMPTY + 2,   // teardown
    B_COUNT
};

template <int kRole>
struct Geo {
    static constexpr bool kThree = kRole != kRoleDV;   // S, dP and the accumulator
    static constexpr bool kWatch = kThree;             // ring hand-off through the watcher warp
    static constexpr int kResident = kThree ? 2 : 1;   // resident 64 KB tiles
    static constexpr int kSlots = kThree ? 3 : 5;      // ring slots of 32 KB
    static constexpr int kRes0 = 0;
    static constexpr int kRes1 = kTile;
    static constexpr int kRing = kResident * kTile;
    static constexpr int kBar = kRing + kSlots * kHalf;
    static constexpr int kTmemSlot = kBar + B_COUNT * 8;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kItems = kAbort + 4;    // [2] published work items
    static constexpr int kMmaExit = kItems + 8;  // set once the MMA warp left its loop
    static constexpr int kFills = kMmaExit + 4;  // ring fills the producer issued in all
    static constexpr int kProdDone = kFills + 4; // set once kFills is final
    static constexpr int kSmemBytes = kProdDone + 4 + 1024;
    static_assert(kSlots <= kMaxSlots, "barrier area");
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
    static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemAcc = 256;
};

// Work item: dQ -- (b, query head h, query tile `tile`), steps = its visible KV
// tiles; dK / dV -- (b, key/value head h, KV tile `tile`), steps = (query head of
// the group, query tile t0 + i) pairs that see a key of the tile.  The numbering
// is the D <= 128 kernels' (blocks of a few heads, longest items first).
struct Item {
    int b, h, tile, steps, t0, tiles_per_head;
};

template <int kRole>
__host__ __device__ __forceinline__ int n_items_of(const BwdParams& p) {
    return kRole == kRoleDQ ? p.B * p.Hq * p.n_q_tiles : p.B * p.Hkv * p.n_kv_tiles;
}

template <int kRole>
__host__ __device__ __forceinline__ Item item_of(const BwdParams& p, int u) {
    Item it{};
    if constexpr (kRole == kRoleDQ) {
        bwd::dq_item(p, u, it.b, it.h, it.tile);
        it.steps = bwd::kv_tiles_for_rows(p, it.tile * kBM);
    } else {
        bwd::dkdv_item(p, u, it.b, it.h, it.tile);
        const int r0 = bwd::first_row_for_kv_tile(p, it.tile);
        it.t0 = r0 >= p.Sq ? p.n_q_tiles : r0 / kBM;  // no query row sees the tile: no steps
        it.tiles_per_head = p.n_q_tiles - it.t0;
        it.steps = (p.Hq / p.Hkv) * it.tiles_per_head;
    }
    return it;
}

// Streamed operand kinds
enum : int { kX1 = 0, kX2 = 1, kY = 2 };

template <int kRole>
__host__ __device__ constexpr int products_per_step() {
    return kRole == kRoleDV ? 2 : 3;
}

// Entry e (0 <= e < products_per_step * N) of the product sequence of an item
// with N >= 1 steps: which streamed operand, of which step.
template <int kRole>
__host__ __device__ __forceinline__ void entry_of(int e, int N, int& kind, int& step) {
    if constexpr (kRole != kRoleDV) {
        if (e < 2) {  // X1_0, X2_0
            kind = e;
            step = 0;
            return;
        }
        const int r = e - 2, q = r / 3, m = r - 3 * q;
        if (q < N - 1) {  // X1_{q+1}, Y_q, X2_{q+1}
            kind = m == 0 ? kX1 : (m == 1 ? kY : kX2);
            step = m == 1 ? q : q + 1;
        } else {  // the last step's Y
            kind = kY;
            step = N - 1;
        }
    } else {
        const int lead = N < 2 ? N : 2;  // X1_0 and X1_1
        if (e < lead) {
            kind = kX1;
            step = e;
            return;
        }
        const int r = e - lead, pairs = N > 2 ? N - 2 : 0;
        if (r < 2 * pairs) {  // Y_n, X1_{n+2}
            kind = (r & 1) ? kX1 : kY;
            step = (r >> 1) + ((r & 1) ? 2 : 0);
        } else {  // the last two steps' Y
            kind = kY;
            step = pairs + (r - 2 * pairs);
        }
    }
}

// 128 x 128 x 128 half of an S-type product: d (+)= A[:, 128 h .. +128) X_h^T,
// A resident (four chunks, K-major), X_h one ring slot (two chunks, K-major).
__device__ __forceinline__ void mma_s_half(uint32_t d, uint64_t a_desc, uint64_t ring_kdesc, int slot, int h,
                                           uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t aoff = static_cast<uint64_t>(((2 * h + (kk >> 2)) * kChunk + (kk & 3) * 32) >> 4);
        const uint64_t xoff = static_cast<uint64_t>((slot * kHalf + (kk >> 2) * kChunk + (kk & 3) * 32) >> 4);
        mma_bf16_ss(d, a_desc + aoff, ring_kdesc + xoff, idesc, (h > 0 || kk > 0) ? 1u : 0u);
    }
}

template <int kRole, bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_bwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const BwdParams p) {
    using G = Geo<kRole>;
    constexpr bool kThree = G::kThree;
    constexpr int kP = products_per_step<kRole>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::kAbort);
    volatile int* item_slot = reinterpret_cast<volatile int*>(smem + G::kItems);
    volatile int* mma_exit = reinterpret_cast<volatile int*>(smem + G::kMmaExit);
    volatile int* fills_total = reinterpret_cast<volatile int*>(smem + G::kFills);
    volatile int* prod_done = reinterpret_cast<volatile int*>(smem + G::kProdDone);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + G::kBar + 8 * i; };
    const int n_items = n_items_of<kRole>(p);
    const int group = p.Hq / p.Hkv;
    const unsigned int limit = p.poll_limit;
    int* const counter = p.work + (kRole == kRoleDV ? 0 : (kRole == kRoleDQ ? 1 : 2));

    if (warp == kLoadWarp && lane == 0) {
        mbar_init(bar(B_A1FULL), 1);
        mbar_init(bar(B_A1EMPTY), 1);
        mbar_init(bar(B_A2FULL), 1);
        mbar_init(bar(B_A2EMPTY), 1);
        for (int s = 0; s < G::kSlots; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 1);
        }
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_SFULL + 1), 1);
        mbar_init(bar(B_DPFULL), 1);
        mbar_init(bar(B_ACCDONE), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_ITEMFULL + i), 1);
            mbar_init(bar(B_ITEMEMPTY + i), 1 + kComputeWarps);
        }
        mbar_init(bar(B_MMADONE), 1);
        *abort_flag = 0;
        *mma_exit = 0;
        *fills_total = 0;
        *prod_done = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == kLoadWarp) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            const uint64_t pol_fix = l2_policy_evict_first();
            const uint64_t pol_stream = l2_policy_evict_last();
            int f = 0, w = 0;        // ring fills issued, items with work loaded
            int a1 = 0, a2 = 0;      // resident fills issued (for the drain)
            // a 4-chunk resident tile or one 2-chunk half of a streamed tile
            auto load = [&](uint32_t dst, const CUtensorMap* m, int col0, int nchunks, int h, int row0, int b,
                            uint32_t full, uint64_t pol) {
                for (int c = 0; c < nchunks; ++c) tma_load_4d(dst + c * kChunk, m, col0 + 64 * c, h, row0, b, full, pol);
            };
            for (int j = 0;; ++j) {
                const int slot = j & 1;
                if (j >= 2 && !wait_bounded(bar(B_ITEMEMPTY + slot), ((j >> 1) - 1) & 1, abort_flag, limit)) break;
                int u = *abort_flag ? -1 : atomicAdd(counter, 1);
                if (u >= n_items) u = -1;
                item_slot[slot] = u;
                mbar_arrive(bar(B_ITEMFULL + slot));
                if (u < 0) break;
                const Item it = item_of<kRole>(p, u);
                if (it.steps == 0) continue;
                const int hkv = kRole == kRoleDQ ? it.h / group : it.h;
                // resident tiles, each once the previous item no longer reads its own
                if (w > 0 && !wait_bounded(bar(B_A1EMPTY), (w - 1) & 1, abort_flag, limit)) break;
                mbar_arrive_expect_tx(bar(B_A1FULL), kTile);
                if constexpr (kRole == kRoleDQ)
                    load(sbase + G::kRes0, &tm_q, 0, 4, it.h, it.tile * kBM, it.b, bar(B_A1FULL), pol_fix);
                else
                    load(sbase + G::kRes0, &tm_k, 0, 4, hkv, it.tile * kBN, it.b, bar(B_A1FULL), pol_fix);
                ++a1;
                if constexpr (kThree) {
                    if (w > 0 && !wait_bounded(bar(B_A2EMPTY), (w - 1) & 1, abort_flag, limit)) break;
                    mbar_arrive_expect_tx(bar(B_A2FULL), kTile);
                    if constexpr (kRole == kRoleDQ)
                        load(sbase + G::kRes1, &tm_do, 0, 4, it.h, it.tile * kBM, it.b, bar(B_A2FULL), pol_fix);
                    else
                        load(sbase + G::kRes1, &tm_v, 0, 4, hkv, it.tile * kBN, it.b, bar(B_A2FULL), pol_fix);
                    ++a2;
                }
                ++w;
                // the streamed halves, in the MMA warp's order
                bool ok = true;
                const int entries = kP * it.steps;
                for (int e = 0; ok && e < entries; ++e) {
                    int kind, step;
                    entry_of<kRole>(e, it.steps, kind, step);
                    const CUtensorMap* m;
                    int h, row0;
                    if constexpr (kRole == kRoleDQ) {  // K (S and dQ) or V (dP) of KV tile `step`
                        m = kind == kX2 ? &tm_v : &tm_k;
                        h = hkv;
                        row0 = step * kBN;
                    } else {  // Q (S and dK) or dO (dP and dV) of (query head, query tile) `step`
                        const bool is_do = kRole == kRoleDV ? kind == kY : kind == kX2;
                        m = is_do ? &tm_do : &tm_q;
                        h = it.h * group + step / it.tiles_per_head;
                        row0 = (it.t0 + step % it.tiles_per_head) * kBM;
                    }
                    for (int hh = 0; hh < 2; ++hh, ++f) {
                        const int s = f % G::kSlots, use = f / G::kSlots;
                        if (use > 0 && !wait_bounded(bar(B_EMPTY + s), (use - 1) & 1, abort_flag, limit)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(bar(B_FULL + s), kHalf);
                        load(sbase + G::kRing + s * kHalf, m, 128 * hh, 2, h, row0, it.b, bar(B_FULL + s), pol_stream);
                    }
                }
                if (!ok) break;
            }
            *fills_total = f;  // the watcher stops after this many fills
            __threadfence_block();
            *prod_done = 1;
            // drain: every copy issued has landed before the CTA may exit
            if (a1 > 0) drain_bounded(bar(B_A1FULL), (a1 - 1) & 1, limit);
            if (a2 > 0) drain_bounded(bar(B_A2FULL), (a2 - 1) & 1, limit);
            for (int s = 0; s < G::kSlots; ++s) {
                const int fills = f > s ? (f - 1 - s) / G::kSlots + 1 : 0;
                if (fills) drain_bounded(bar(B_FULL + s), (fills - 1) & 1, limit);
            }
        }
        __syncwarp();
        // release warp of the abort path: the elementwise warps' and the watcher's
        // arrivals (see bwd::release_named_barriers).  It starts only after the loop
        // above has stopped re-arming slots and drained every fill it issued, so an
        // MMA warp it frees from a ring hand-off reads landed data and frees slots
        // that are never refilled.
        const unsigned long long cap = 64ull * limit;
        unsigned long long i = 0;
        for (; i < cap && !*mma_exit; ++i) {
            if (*abort_flag) {
                for (int id = 0; id < 2; ++id)
                    for (int k = 0; k < kComputeWarps; ++k) named_bar_arrive(2 + id, kBarReadyThreads);
                if constexpr (G::kWatch)
                    for (int s = 0; s < G::kSlots; ++s) named_bar_arrive(kBarRing0 + s, kBarRingThreads);
            } else {
                nanosleep_ns(1024);
            }
        }
        if (i == cap) atomicOr(&g_attn_status, kStatusTimeout);
    } else if (warp == kWatchWarp) {
        // =========================== ring watcher ===========================
        // Fill f landed -> arrive on its slot's named barrier.  Stops once the
        // producer has finished and every fill it issued was handed over.
        for (int f = 0; G::kWatch; ++f) {
            const int s = f % G::kSlots;
            bool landed = false;
            unsigned int i = 0;
            for (; i < limit; ++i) {
                if (mbar_try_wait(bar(B_FULL + s), (f / G::kSlots) & 1)) {
                    landed = true;
                    break;
                }
                if ((i & 15u) == 15u && (*abort_flag || (*prod_done && f >= *fills_total))) break;
            }
            if (!__all_sync(0xffffffffu, landed)) {
                if (i == limit) {
                    *abort_flag = 1;
                    atomicOr(&g_attn_status, kStatusTimeout);
                }
                break;
            }
            named_bar_arrive(kBarRing0 + s, kBarRingThreads);
        }
    } else if (warp == kMmaWarp) {
        // =========================== MMA issuer =============================
        constexpr uint32_t idesc_s = idesc_f16kind_f32(kBM, kBN, false, kF16);  // S, dP (or transposed)
        constexpr uint32_t idesc_acc = idesc_f16kind_f32(kBM, 128, true, kF16);  // one half of the accumulator
        const uint64_t a1_desc = sdesc_sw128(sbase + G::kRes0, 16, 1024);
        const uint64_t a2_desc = sdesc_sw128(sbase + G::kRes1, 16, 1024);
        const uint64_t ring_k = sdesc_sw128(sbase + G::kRing, 16, 1024);
        const uint64_t ring_mn = sdesc_sw128(sbase + G::kRing, kChunk, 1024);
        const uint32_t tAcc = tmem_base + G::kTmemAcc;
        bool ok = true;
        int f = 0, g = 0, w = 0;  // ring fills consumed, steps (over all items), items with work
        int s_issued = 0;         // S products issued (3-product roles: the S read-out sync count)
        // Half hh of the product whose first fill is f has landed.  With the watcher:
        // its hand-off, per half.  Without (dV, whose deeper ring is usually full
        // ahead): one poll of both halves' barriers before the first half, measured
        // faster there than the watcher.
        auto half_ready = [&](int hh) -> bool {
            if constexpr (G::kWatch) {
                named_bar_sync(kBarRing0 + static_cast<uint32_t>((f + hh) % G::kSlots), kBarRingThreads);
            } else {
                if (hh == 0)
                    for (int k = 0; k < 2; ++k)
                        if (!wait_bounded(bar(B_FULL + (f + k) % G::kSlots), ((f + k) / G::kSlots) & 1, abort_flag,
                                          limit))
                            return false;
            }
            tc_fence_after();
            return true;
        };
        for (int j = 0; ok; ++j) {
            const int slot = j & 1;
            if (!wait_bounded(bar(B_ITEMFULL + slot), (j >> 1) & 1, abort_flag, limit)) break;
            const int u = item_slot[slot];
            __syncwarp();
            if (elect_one()) mbar_arrive(bar(B_ITEMEMPTY + slot));
            __syncwarp();
            if (u < 0) break;
            const Item it = item_of<kRole>(p, u);
            const int N = it.steps;
            if (N == 0) continue;
            const int entries = kP * N;
            for (int e = 0; e < entries; ++e) {
                int kind, step;
                entry_of<kRole>(e, N, kind, step);
                const int gs = g + step;
                if (kind == kX1) {
                    // S_step = A1 X1^T into its buffer
                    if (kThree && s_issued > 0) named_bar_sync(kBarSRead, kBarReadyThreads);  // previous S read out
                    if (step == 0 && !wait_bounded(bar(B_A1FULL), w & 1, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t d = tmem_base + (kThree ? G::kTmemS : 128u * static_cast<uint32_t>(gs & 1));
                    for (int hh = 0; hh < 2; ++hh) {
                        if (!half_ready(hh)) {
                            ok = false;
                            break;
                        }
                        if (elect_one()) {
                            mma_s_half(d, a1_desc, ring_k, (f + hh) % G::kSlots, hh, idesc_s);
                            mma_commit(bar(B_EMPTY + (f + hh) % G::kSlots));
                            if (hh == 1) {
                                mma_commit(bar(B_SFULL + (kThree ? 0 : (gs & 1))));
                                if (step == N - 1) mma_commit(bar(B_A1EMPTY));  // the item's last S
                            }
                        }
                        __syncwarp();
                    }
                    ++s_issued;
                } else if (kind == kX2) {
                    // dP_step = A2 X2^T (3-product roles only)
                    if (step == 0 && !wait_bounded(bar(B_A2FULL), w & 1, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    for (int hh = 0; hh < 2; ++hh) {
                        if (!half_ready(hh)) {
                            ok = false;
                            break;
                        }
                        if (elect_one()) {
                            mma_s_half(tmem_base + G::kTmemDP, a2_desc, ring_k, (f + hh) % G::kSlots, hh, idesc_s);
                            mma_commit(bar(B_EMPTY + (f + hh) % G::kSlots));
                            if (hh == 1) {
                                mma_commit(bar(B_DPFULL));
                                if (step == N - 1) mma_commit(bar(B_A2EMPTY));  // the item's last dP
                            }
                        }
                        __syncwarp();
                    }
                } else {
                    // acc[:, 128 h .. +128) (+)= E_step Y_h, E = dS (over dP) or P (over its S buffer)
                    if constexpr (kThree)
                        named_bar_sync(kBarDsReady, kBarReadyThreads);
                    else
                        named_bar_sync(kBarP0 + static_cast<uint32_t>(gs & 1), kBarReadyThreads);
                    tc_fence_after();
                    const uint32_t tE = tmem_base + (kThree ? G::kTmemDP : 128u * static_cast<uint32_t>(gs & 1));
                    for (int hh = 0; hh < 2; ++hh) {
                        if (!half_ready(hh)) {
                            ok = false;
                            break;
                        }
                        if (elect_one()) {
                            bwd::mma_tmem_mn(tAcc + 128 * hh, tE,
                                             ring_mn + static_cast<uint64_t>((((f + hh) % G::kSlots) * kHalf) >> 4),
                                             idesc_acc, step > 0);
                            mma_commit(bar(B_EMPTY + (f + hh) % G::kSlots));
                            if (hh == 1 && step == N - 1) mma_commit(bar(B_ACCDONE));
                        }
                        __syncwarp();
                    }
                }
                if (!ok) break;
                f += 2;
            }
            if (!ok) break;
            g += N;
            ++w;
        }
        // 3-product roles: the last S read-out is the one signal not yet met
        if (kThree && ok && s_issued > 0) named_bar_sync(kBarSRead, kBarReadyThreads);
        *mma_exit = 1;  // the release loop may stop
        if (elect_one()) {
            mma_commit(bar(B_MMADONE));
            drain_bounded(bar(B_MMADONE), 0, limit);
        }
        __syncwarp();
    } else {
        // =========================== elementwise warps ======================
        const int quarter = warp % 4, grp = warp / 4;
        const int r = quarter * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int g = 0, w = 0;
        for (int j = 0; ok; ++j) {
            const int slot = j & 1;
            const bool got_item = wait_bounded(bar(B_ITEMFULL + slot), (j >> 1) & 1, abort_flag, limit);
            if (!__all_sync(0xffffffffu, got_item)) break;
            const int u = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_ITEMEMPTY + slot));
            if (u < 0) break;
            const Item it = item_of<kRole>(p, u);
            const int N = it.steps;
            const int row = it.tile * kBM + r;  // query row (dQ) or key (dK, dV) of this thread
            // dQ: this row's lse2, delta and last visible key (keys past Skv are masked too)
            float neg_l2 = 0.f, dlt = 0.f;
            int lim = 0;
            if constexpr (kRole == kRoleDQ) {
                const size_t vo = (static_cast<size_t>(it.b) * p.Hq + it.h) * p.sq_pad + row;  // row < sq_pad
                neg_l2 = -p.lse2[vo];
                dlt = p.delta[vo];
                const long long lim_ll =
                    p.causal ? min((long long)row + p.diag, (long long)p.Skv - 1) : (long long)p.Skv - 1;
                lim = static_cast<int>(lim_ll < -1 ? -1 : lim_ll);
            }
            for (int n = 0; n < N; ++n) {
                const int gs = g + n;
                const uint32_t sbuf = kThree ? G::kTmemS : 128u * static_cast<uint32_t>(gs & 1);
                const uint32_t tS = tmem_base + lane_off + sbuf + kCols * grp;
                // dK / dV: the columns are query rows of (query head hq, tile t)
                const float* l2v = nullptr;
                const float* dlv = nullptr;
                int cmin = -1;  // first visible column of this group (dK / dV, causal)
                if constexpr (kRole != kRoleDQ) {
                    const int hq = it.h * group + n / it.tiles_per_head;
                    const int t = it.t0 + n % it.tiles_per_head;
                    const size_t vo = (static_cast<size_t>(it.b) * p.Hq + hq) * p.sq_pad +
                                      static_cast<size_t>(t) * kBM + kCols * grp;
                    l2v = p.lse2 + vo;
                    dlv = p.delta + vo;
                    if (p.causal) cmin = row - p.diag - (t * kBM + kCols * grp);
                }
                float lv[kCols];
                if constexpr (kRole != kRoleDQ) {
#pragma unroll
                    for (int c = 0; c < kCols; c += 4) {
                        const float4 x4 = *reinterpret_cast<const float4*>(l2v + c);
                        lv[c] = x4.x;
                        lv[c + 1] = x4.y;
                        lv[c + 2] = x4.z;
                        lv[c + 3] = x4.w;
                    }
                }
                const bool got = wait_bounded(bar(B_SFULL + (kThree ? 0 : (gs & 1))), kThree ? (gs & 1) : ((gs >> 1) & 1),
                                              abort_flag, limit);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t x[kCols];
                bwd::tmem_ld_cols<kCols>(tS, x);
                if constexpr (kThree) {
                    tc_fence_before();
                    named_bar_arrive(kBarSRead, kBarReadyThreads);  // S may now be overwritten
                }
                float pv[kCols];
#pragma unroll
                for (int c = 0; c < kCols; c += 2) {
                    if constexpr (kRole == kRoleDQ)
                        ffma2_bc(pv[c], pv[c + 1], __uint_as_float(x[c]), __uint_as_float(x[c + 1]), sl2, neg_l2);
                    else
                        bwd::ffma2_b(pv[c], pv[c + 1], __uint_as_float(x[c]), __uint_as_float(x[c + 1]), sl2, -lv[c],
                                     -lv[c + 1]);
                    pv[c] = ex2_approx(pv[c]);
                    pv[c + 1] = ex2_approx(pv[c + 1]);
                }
                if constexpr (kRole == kRoleDQ) {
                    const int nvis = lim - (n * kBN + kCols * grp) + 1;  // visible columns of this group
                    if (nvis < kCols) {
#pragma unroll
                        for (int c = 0; c < kCols; ++c)
                            if (c >= nvis) pv[c] = 0.f;
                    }
                } else {
                    if (cmin > 0) {
#pragma unroll
                        for (int c = 0; c < kCols; ++c)
                            if (c < cmin) pv[c] = 0.f;
                    }
                }
                if constexpr (!kThree) {
                    // dV: P^T packed over this group's own S columns
                    uint32_t pk[kCols / 2];
#pragma unroll
                    for (int c = 0; c < kCols / 2; ++c) pk[c] = pack_x2<kF16>(pv[2 * c], pv[2 * c + 1]);
                    bwd::tmem_st_packed<kCols>(tS, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    named_bar_arrive(kBarP0 + static_cast<uint32_t>(gs & 1), kBarReadyThreads);
                } else {
                    // dK: this group's delta, 32 columns at a time, each loaded one piece
                    // ahead (the first before the wait) so its latency is hidden
                    float dv[32];
                    auto load_delta = [&](int c0) {
#pragma unroll
                        for (int c = 0; c < 32; c += 4) {
                            if constexpr (kRole == kRoleDK) {
                                const float4 d4 = *reinterpret_cast<const float4*>(dlv + c0 + c);
                                dv[c] = d4.x;
                                dv[c + 1] = d4.y;
                                dv[c + 2] = d4.z;
                                dv[c + 3] = d4.w;
                            } else {
                                dv[c] = dv[c + 1] = dv[c + 2] = dv[c + 3] = dlt;
                            }
                        }
                    };
                    load_delta(0);
                    const bool got2 = wait_bounded(bar(B_DPFULL), gs & 1, abort_flag, limit);
                    if (!__all_sync(0xffffffffu, got2)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t tDP = tmem_base + lane_off + G::kTmemDP + kCols * grp;
                    // dS = P (dP - delta), 32 columns at a time; packed over this group's own dP columns
#pragma unroll
                    for (int hc = 0; hc < kCols; hc += 32) {
                        uint32_t y[32];
                        tmem_ld32(tDP + hc, y);
                        tmem_wait_ld_regs(y);
                        uint32_t pk[16];
#pragma unroll
                        for (int c = 0; c < 32; c += 2) {
                            float d0, d1;
                            bwd::fsubmul2(d0, d1, pv[hc + c], pv[hc + c + 1], __uint_as_float(y[c]),
                                          __uint_as_float(y[c + 1]), dv[c], dv[c + 1]);
                            pk[c / 2] = pack_x2<kF16>(d0, d1);
                        }
                        if (hc + 32 < kCols) load_delta(hc + 32);
                        tmem_st16(tDP + hc / 2, pk);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    named_bar_arrive(kBarDsReady, kBarReadyThreads);
                }
            }
            if (!ok) break;
            // epilogue: this row's accumulator columns [128 grp, 128 grp + 128), times the
            // scale for dQ and dK; read out before this thread's next hand-off arrival,
            // which gates the next item's first accumulator product
            const bool have = N > 0;
            if (have) {
                const bool got = wait_bounded(bar(B_ACCDONE), w & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got)) break;
                tc_fence_after();
            }
            uint16_t* out;
            bool write;
            size_t off;
            if constexpr (kRole == kRoleDQ) {
                write = row < p.Sq;
                off = ((static_cast<size_t>(it.b) * p.Sq + (write ? row : 0)) * p.Hq + it.h) * kD;
                out = p.dq;
            } else {
                write = row < p.Skv;
                off = ((static_cast<size_t>(it.b) * p.Skv + (write ? row : 0)) * p.Hkv + it.h) * kD;
                out = kRole == kRoleDK ? p.dk : p.dv;
            }
            const float mul = kRole == kRoleDV ? 1.f : p.scale;
#pragma unroll
            for (int c = 0; c < 2; ++c)
                bwd::store_acc_part<kF16, 128>(tmem_base + lane_off + G::kTmemAcc + 128 * grp + 64 * c, have, mul,
                                               out + off + 128 * grp + 64 * c, write);
            if (have) {
                g += N;
                ++w;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace bwd256
}  // namespace attn
