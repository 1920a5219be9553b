// fmha_bwd_sm103.cuh -- attention backward for sm_103a (GB300).
//
// Given Q, K, V, the forward output O, its LSE and the output gradient dO, the
// three kernels below produce dQ, dK and dV: the Pallas page's
// `_attention_bwd` (delta = rowsum(O * dO); a dQ kernel that walks the KV
// tiles of one query tile; a dK/dV kernel that walks the query tiles of one KV
// tile), rebuilt on tcgen05 with tensor-memory accumulators.
//
//   prep    delta_i = sum_d dO[i,d] O[i,d] and lse2_i = lse_i * log2(e) of every
//           query row into a padded workspace (+inf / 0 on padding and on rows
//           that see no key, so their weights vanish without a mask).
//   dK/dV   one CTA per (batch, key/value head, 128-key tile).  For every query
//           head of the group and every 128-row query tile that sees a key of
//           the tile:
//             S^T  = K Q^T            (tensor memory, 128 keys x 128 rows)
//             dP^T = V dO^T
//             P^T  = 2^(S^T scale log2e - lse2)       (bf16, over S^T)
//             dS^T = P^T (dP^T - delta)               (bf16, over dP^T)
//             dV  += P^T dO,   dK += dS^T Q           (A operands from tensor memory)
//           The group's query heads accumulate into the same dK/dV, which is
//           the page's sum of per-head dK/dV over each group, done in place.
//   dQ      one CTA per (batch, query head, 128-row tile), over its visible KV tiles:
//             S = Q K^T,  dP = dO V^T,  dS = P (dP - delta)   (bf16, over dP)
//             dQ += dS K
//   dQ and dK carry the softmax scale (applied to the fp32 accumulators).
//
// Warp roles (320 threads): warps 0-7 elementwise work (warp w owns TMEM lane
// quarter w % 4 and one half of the 128 columns: w / 4), warp 8 issues the MMAs
// (one elected lane), warp 9 drives the TMA copies and then serves as the release
// warp of the abort path.  The elementwise warps hand P and dS to the MMA warp
// through hardware named barriers (they arrive, it syncs), as in the forward
// kernel: an mbarrier poll by the MMA-issuing warp would first wait for its
// queued MMAs to drain.  The operand that stays
// fixed for the CTA (K and V, or Q and dO) is loaded once; the other pair
// streams through a two-stage ring.  Every mbarrier wait is bounded as in the
// forward kernel (timeout status, CTA abort flag, drained copies, freed TMEM).
#pragma once
#include <cstdint>
#include <cuda.h>

#include "fmha_fwd_sm103.cuh"

namespace attn {
namespace bwd {

// The release loop of the abort path, run by a whole warp (the forward kernel's
// release warp does the same inline).  An MMA warp that waits on a hardware named
// barrier cannot time out, so until that warp reports (through mma_exit) that it
// left its loop, this loop sleeps; once the abort flag is up it arrives on the
// named barriers first_id .. first_id + n_ids - 1, arrivals_per_round times each
// per round (the other parties' share of nthreads), so a waiting MMA warp moves on
// and meets the abort at its next bounded mbarrier wait.  Surplus arrivals only
// complete generations nobody waits for.
__device__ __forceinline__ void release_named_barriers(volatile int* mma_exit, volatile int* abort_flag,
                                                       uint32_t first_id, int n_ids, uint32_t nthreads,
                                                       int arrivals_per_round, unsigned int limit) {
    const unsigned long long cap = 64ull * limit;
    unsigned long long i = 0;
    for (; i < cap && !*mma_exit; ++i) {
        if (*abort_flag) {
            for (int b = 0; b < n_ids; ++b)
                for (int k = 0; k < arrivals_per_round; ++k) named_bar_arrive(first_id + b, nthreads);
        } else {
            nanosleep_ns(1024);
        }
    }
    if (i == cap) atomicOr(&g_attn_status, kStatusTimeout);
}

// The elementwise warps split each 128-column tile into kGroups groups of
// kCols columns: warp w owns TMEM lane quarter w % 4 and column group w / 4.
constexpr int kGroups = 2;
constexpr int kCols = 128 / kGroups;
constexpr int kComputeWarps = 4 * kGroups;
constexpr int kMmaWarp = kComputeWarps;
constexpr int kLoadWarp = kComputeWarps + 1;
constexpr int kThreads = 32 * (kComputeWarps + 2);
constexpr int kStages = 2;
constexpr int kVecBytes = kBM * 4;  // lse2 or delta of one 128-row tile
// named barriers (elementwise warps arrive, the MMA warp syncs): P (or S read out)
// and dS in tensor memory
constexpr uint32_t kBarPReady = 2, kBarDsReady = 3;
constexpr uint32_t kBarReadyThreads = 32 * kComputeWarps + 32;

// Barriers of the dK/dV kernel.
enum : int {
    BAR_KFULL = 0,                 // the item's K tile landed
    BAR_KEMPTY,                    // its last S^T completed: K may be replaced
    BAR_VFULL,
    BAR_VEMPTY,                    // its last dP^T completed: V may be replaced
    BAR_FULL,                      // [stage] Q, dO and their lse2 / delta
    BAR_EMPTY = BAR_FULL + kStages,
    BAR_SFULL = BAR_EMPTY + kStages,
    BAR_DPFULL,
    BAR_ACCDONE,                   // the item's last dK completed
    BAR_ITEMFULL,                  // [2] next work item published
    BAR_ITEMEMPTY = BAR_ITEMFULL + 2,  // [2] read by the MMA warp and the 8 elementwise warps
    BAR_MMADONE = BAR_ITEMEMPTY + 2,   // teardown
    BAR_COUNT
};

// Shared memory: two fixed tiles, two rings of kStages tiles, and (dK/dV) the
// per-stage lse2 / delta vectors.  1024-byte aligned base.
template <int kD>
struct BwdGeo {
    static_assert(kD == 64 || kD == 128, "head size 64 or 128");
    static constexpr int kHalves = kD / 64;
    static constexpr int kTileBytes = kBM * kD * 2;
    static constexpr int kFix0 = 0;
    static constexpr int kFix1 = kTileBytes;
    static constexpr int kRing0 = 2 * kTileBytes;
    static constexpr int kRing1 = kRing0 + kStages * kTileBytes;
    static constexpr int kVec = kRing1 + kStages * kTileBytes;  // [stage] {lse2[128], delta[128]}
    static constexpr int kBar = kVec + kStages * 2 * kVecBytes;
    static constexpr int kTmemSlot = kBar + BAR_COUNT * 8;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kItems = kAbort + 4;          // [2] published work items
    static constexpr int kMmaExit = kItems + 8;        // set once the MMA warp left its loop
    static constexpr int kSmemBytes = kMmaExit + 4 + 1024;
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
    // tensor-memory columns
    static constexpr uint32_t kTmemS = 0;
    static constexpr uint32_t kTmemDP = 128;
    static constexpr uint32_t kTmemAcc0 = 256;        // dV (dK/dV kernel) or dQ
    static constexpr uint32_t kTmemAcc1 = 256 + kD;   // dK
};

struct BwdParams {
    int B, Sq, Skv, Hq, Hkv, D;
    int causal;                 // 0: none; 1: bottom-right; 2: top-left
    int diag;                   // key j visible from row i iff j <= i + diag (when causal)
    int sq_pad;                 // rows per (b, h) in the workspace vectors (multiple of 128)
    float scale;                // softmax scale
    float scale_log2;           // scale * log2(e)
    float* lse2;                // [B, Hq, sq_pad]
    float* delta;               // [B, Hq, sq_pad]
    uint16_t* dq;               // [B, Sq, Hq, D]
    uint16_t* dk;               // [B, Skv, Hkv, D]
    uint16_t* dv;               // [B, Skv, Hkv, D]
    int* work;                  // work-item counters (zeroed by prep): dK/dV or dV ([0]), dQ ([1]), dK ([2])
    int n_q_tiles, n_kv_tiles;
    unsigned int poll_limit;
};

// 1-d bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// packed fp32x2: (d0, d1) = (a0 * b + c0, a1 * b + c1)
__device__ __forceinline__ void ffma2_b(float& d0, float& d1, float a0, float a1, float b, float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %4};\n\t"
        "mov.b64 rc, {%5, %6};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
}

// packed fp32x2: (d0, d1) = (p0 * (x0 - y0), p1 * (x1 - y1))
__device__ __forceinline__ void fsubmul2(float& d0, float& d1, float p0, float p1, float x0, float x1, float y0,
                                         float y1) {
    asm("{\n\t.reg .b64 rp, rx, ry, rd;\n\t"
        "mov.b64 rp, {%2, %3};\n\t"
        "mov.b64 rx, {%4, %5};\n\t"
        "mov.b64 ry, {%6, %7};\n\t"
        "sub.rn.f32x2 rd, rx, ry;\n\t"
        "mul.rn.f32x2 rd, rd, rp;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(p0), "f"(p1), "f"(x0), "f"(x1), "f"(y0), "f"(y1));
}

template <bool kF16>
__device__ __forceinline__ float widen16(uint16_t x) {
    if constexpr (kF16) {
        float f;
        asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(x));
        return f;
    } else {
        return __uint_as_float(static_cast<uint32_t>(x) << 16);
    }
}

// First query row that sees a key of KV tile n (causal), clamped at 0.
__host__ __device__ __forceinline__ int first_row_for_kv_tile(const BwdParams& p, int n) {
    if (!p.causal) return 0;
    const long long r = (long long)n * kBN - p.diag;
    return r < 0 ? 0 : (r > p.Sq ? p.Sq : static_cast<int>(r));
}

// Number of KV tiles the query tile starting at row0 visits.
__host__ __device__ __forceinline__ int kv_tiles_for_rows(const BwdParams& p, int row0) {
    if (row0 >= p.Sq) return 0;
    if (!p.causal) return p.n_kv_tiles;
    const int last_row = row0 + kBM - 1 < p.Sq - 1 ? row0 + kBM - 1 : p.Sq - 1;
    const long long last_key = (long long)last_row + p.diag;
    if (last_key < 0) return 0;
    const long long n = last_key / kBN + 1;
    return n < p.n_kv_tiles ? static_cast<int>(n) : p.n_kv_tiles;
}

// ---------------------------------------------------------------- prep
// delta and lse2 of every padded row.  Grid: (rows of a batch entry / block,
// batch).  Within a batch entry rows are taken in memory order (i, h), so a
// warp's loads of O and dO are contiguous: each lane loads 16 bytes of each,
// kD / 8 lanes cover a row, and a warp handles kPrepIters groups of
// 32 / (kD / 8) rows with all loads issued before the reductions.
constexpr int kPrepIters = 2;
template <int kD>
__host__ __device__ constexpr int prep_rows_per_warp() {
    return (32 / (kD / 8)) * kPrepIters;
}

template <bool kF16, int kD>
__global__ void __launch_bounds__(256)
    bwd_prep_kernel(const uint16_t* __restrict__ o, const uint16_t* __restrict__ dO, const float* __restrict__ lse,
                    const BwdParams p) {
    constexpr int kL = kD / 8;          // lanes per row
    constexpr int kR = 32 / kL;         // rows per load instruction
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const int b = static_cast<int>(blockIdx.y);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)  // the work queues
        p.work[0] = p.work[1] = p.work[2] = 0;
    const int per_batch = p.sq_pad * p.Hq;  // rows (i, h) of one batch entry, in memory order
    const int row0 = (static_cast<int>(blockIdx.x) * 8 + static_cast<int>(threadIdx.x) / 32) * (kR * kPrepIters);
    uint4 ov[kPrepIters], dv[kPrepIters];
    int ii[kPrepIters], hh[kPrepIters];
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
        const int r = row0 + it * kR + lane / kL;
        ii[it] = r < per_batch ? r / p.Hq : p.sq_pad;
        hh[it] = r - (r / p.Hq) * p.Hq;
        ov[it] = dv[it] = make_uint4(0u, 0u, 0u, 0u);
        if (ii[it] < p.Sq) {
            const size_t off = ((static_cast<size_t>(b) * p.Sq + ii[it]) * p.Hq + hh[it]) * kD + 8 * (lane % kL);
            ov[it] = *reinterpret_cast<const uint4*>(o + off);
            dv[it] = *reinterpret_cast<const uint4*>(dO + off);
        }
    }
#pragma unroll
    for (int it = 0; it < kPrepIters; ++it) {
        const uint32_t a[4] = {ov[it].x, ov[it].y, ov[it].z, ov[it].w};
        const uint32_t c[4] = {dv[it].x, dv[it].y, dv[it].z, dv[it].w};
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc += widen16<kF16>(static_cast<uint16_t>(a[e] & 0xFFFF)) * widen16<kF16>(static_cast<uint16_t>(c[e] & 0xFFFF));
            acc += widen16<kF16>(static_cast<uint16_t>(a[e] >> 16)) * widen16<kF16>(static_cast<uint16_t>(c[e] >> 16));
        }
#pragma unroll
        for (int sft = kL / 2; sft > 0; sft >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sft);
        const int i = ii[it], h = hh[it];
        if (lane % kL == 0 && i < p.sq_pad) {
            const size_t w = (static_cast<size_t>(b) * p.Hq + h) * p.sq_pad + i;
            float l2 = INFINITY, dl = 0.f;
            if (i < p.Sq) {
                const float l = lse[(static_cast<size_t>(b) * p.Hq + h) * p.Sq + i];
                l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
                dl = acc;
            }
            p.lse2[w] = l2;
            p.delta[w] = dl;
        }
    }
}

// ---------------------------------------------------------------- shared helpers
struct Roles {
    uint8_t* smem;
    uint32_t sbase;
    int warp, lane;
};

// K-major x K-major product over the head dimension: D[128 x 128] = A[128 x kD] B[128 x kD]^T
template <int kD>
__device__ __forceinline__ void mma_kmajor(uint32_t d, uint64_t a0, uint64_t b0, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
        mma_bf16_ss(d, a0 + off, b0 + off, idesc, kk > 0 ? 1u : 0u);
    }
}

// A from tensor memory (128 lanes x 128 packed 16-bit elements) times an MN-major
// 128 x kD shared-memory tile: D[128 x kD] (+)= A B.  The packed A is stored as
// kGroups pieces of kCols elements (kCols / 2 columns each) at columns
// a_tmem + kCols * g: each group of elementwise warps packs its piece over the
// start of its own fp32 columns, so no group overwrites columns another is
// still reading.
__device__ __forceinline__ void mma_tmem_mn(uint32_t d, uint32_t a_tmem, uint64_t b0, uint32_t idesc,
                                            bool accumulate) {
    constexpr int kStepsPerGroup = kCols / 16;
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)
        mma_bf16_ts(d, a_tmem + (kk / kStepsPerGroup) * kCols + (kk % kStepsPerGroup) * 8,
                    b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// kN consecutive fp32 columns of this thread's lane (kN = 16, 32 or 64)
template <int kN>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[kN]) {
    if constexpr (kN == 64) {
        tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
        tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
        tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    } else if constexpr (kN == 32) {
        tmem_ld32(taddr, r);
        tmem_wait_ld_regs(r);
    } else {
        tmem_ld16(taddr, r);
        tmem_wait_ld_regs16(r);
    }
}

// kN / 2 packed columns (kN = 32 or 64) from registers to tensor memory
template <int kN>
__device__ __forceinline__ void tmem_st_packed(uint32_t taddr, const uint32_t (&pk)[kN / 2]) {
#pragma unroll
    for (int c = 0; c < kN / 2; c += 16) tmem_st16(taddr + c, *reinterpret_cast<const uint32_t(*)[16]>(&pk[c]));
}

// 64 consecutive fp32 columns of this thread's lane (two x32 loads)
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
    tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
    tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
}

// kN accumulator columns of this thread's lane from taddr on, times `mul`, to
// kN 16-bit elements at dst (16-byte aligned); kN = kD / kGroups.
template <bool kF16, int kD>
__device__ __forceinline__ void store_acc_part(uint32_t taddr, bool have, float mul, uint16_t* dst, bool write) {
    constexpr int kN = kD / kGroups;  // 16, 32 or 64
    uint32_t a[kN];
    if (have) {
        tmem_ld_cols<kN>(taddr, a);
    } else {
#pragma unroll
        for (int e = 0; e < kN; ++e) a[e] = 0u;
    }
    if (!write) return;
#pragma unroll
    for (int q = 0; q < kN / 8; ++q) {
        float f[8];
#pragma unroll
        for (int e = 0; e < 8; e += 2)
            fmul2_b(f[e], f[e + 1], __uint_as_float(a[8 * q + e]), __uint_as_float(a[8 * q + e + 1]), mul);
        reinterpret_cast<uint4*>(dst)[q] = make_uint4(pack_x2<kF16>(f[0], f[1]), pack_x2<kF16>(f[2], f[3]),
                                                      pack_x2<kF16>(f[4], f[5]), pack_x2<kF16>(f[6], f[7]));
    }
}

// ---------------------------------------------------------------- dK / dV
// Work item u = one (b, hkv, 128-key tile).  Items are numbered in blocks of
// kItemHeads heads: within a block by KV tile (the tiles near the start of the
// keys, which see the most query rows under a causal mask, first), then by
// head.  So the longest items come first within each block, and the CTAs in
// flight work on a few heads at a time, whose Q and dO stay in L2.
constexpr int kItemHeads = 4;

__host__ __device__ __forceinline__ void dkdv_item(const BwdParams& p, int u, int& b, int& hkv, int& n) {
    const int nbh = p.B * p.Hkv;
    const int per_block = kItemHeads * p.n_kv_tiles;
    const int blk = u / per_block;
    const int within = u - blk * per_block;
    const int heads = nbh - blk * kItemHeads < kItemHeads ? nbh - blk * kItemHeads : kItemHeads;
    n = within / heads;
    const int bh = blk * kItemHeads + (within - n * heads);
    b = bh / p.Hkv;
    hkv = bh % p.Hkv;
}

// Persistent: at most one CTA per SM; the TMA warp takes items from a global
// counter (the prep kernel zeroes it) and publishes each through a two-slot
// ring in shared memory.  The Q/dO ring and the per-step barriers run on across
// items; K of the next item is loaded as soon as the current item's last S^T
// has read its K, V as soon as its last dP^T has read its V, and the next
// item's first dV / dK (which start the accumulators afresh) come only after
// the elementwise warps have read the current accumulators out.
template <bool kF16, int kD>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const BwdParams p) {
    using G = BwdGeo<kD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::kAbort);
    volatile int* item_slot = reinterpret_cast<volatile int*>(smem + G::kItems);
    volatile int* mma_exit = reinterpret_cast<volatile int*>(smem + G::kMmaExit);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + G::kBar + 8 * i; };
    const int n_items = p.B * p.Hkv * p.n_kv_tiles;
    const int group = p.Hq / p.Hkv;
    const unsigned int limit = p.poll_limit;
    // the item's first query tile and number of (head, query tile) steps
    auto steps_of = [&](int n, int& t0, int& tiles_per_head) {
        const int r0 = first_row_for_kv_tile(p, n);
        t0 = r0 >= p.Sq ? p.n_q_tiles : r0 / kBM;  // no query row sees the tile: no steps
        tiles_per_head = p.n_q_tiles - t0;
        return group * tiles_per_head;
    };

    if (warp == kLoadWarp && lane == 0) {
        mbar_init(bar(BAR_KFULL), 1);
        mbar_init(bar(BAR_KEMPTY), 1);
        mbar_init(bar(BAR_VFULL), 1);
        mbar_init(bar(BAR_VEMPTY), 1);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(BAR_FULL + s), 1);
            mbar_init(bar(BAR_EMPTY + s), 1);
        }
        mbar_init(bar(BAR_SFULL), 1);
        mbar_init(bar(BAR_DPFULL), 1);
        mbar_init(bar(BAR_ACCDONE), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(BAR_ITEMFULL + i), 1);
            mbar_init(bar(BAR_ITEMEMPTY + i), 1 + kComputeWarps);
        }
        mbar_init(bar(BAR_MMADONE), 1);
        *abort_flag = 0;
        *mma_exit = 0;
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
            int g = 0, w = 0;        // ring fills issued, items with work loaded
            int kfix = 0, vfix = 0;  // K and V fills issued (for the drain)
            for (int j = 0;; ++j) {
                // take the next item and publish it
                const int slot = j & 1;
                if (j >= 2 && !wait_bounded(bar(BAR_ITEMEMPTY + slot), ((j >> 1) - 1) & 1, abort_flag, limit)) break;
                int u = *abort_flag ? -1 : atomicAdd(p.work, 1);
                if (u >= n_items) u = -1;
                item_slot[slot] = u;
                mbar_arrive(bar(BAR_ITEMFULL + slot));
                if (u < 0) break;
                int b, hkv, n, t0, tiles_per_head;
                dkdv_item(p, u, b, hkv, n);
                const int steps = steps_of(n, t0, tiles_per_head);
                if (steps == 0) continue;
                // K, then V of this item, each once the previous item no longer reads it
                if (w > 0 && !wait_bounded(bar(BAR_KEMPTY), (w - 1) & 1, abort_flag, limit)) break;
                mbar_arrive_expect_tx(bar(BAR_KFULL), G::kTileBytes);
                for (int h = 0; h < G::kHalves; ++h)
                    tma_load_4d(sbase + G::kFix0 + h * kHalfBytes, &tm_k, h * 64, hkv, n * kBN, b, bar(BAR_KFULL),
                                pol_fix);
                ++kfix;
                if (w > 0 && !wait_bounded(bar(BAR_VEMPTY), (w - 1) & 1, abort_flag, limit)) break;
                mbar_arrive_expect_tx(bar(BAR_VFULL), G::kTileBytes);
                for (int h = 0; h < G::kHalves; ++h)
                    tma_load_4d(sbase + G::kFix1 + h * kHalfBytes, &tm_v, h * 64, hkv, n * kBN, b, bar(BAR_VFULL),
                                pol_fix);
                ++vfix;
                ++w;
                bool ok = true;
                for (int st = 0; st < steps; ++st, ++g) {
                    const int s = g % kStages, use = g / kStages;
                    if (use > 0 && !wait_bounded(bar(BAR_EMPTY + s), (use - 1) & 1, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    const int hq = hkv * group + st / tiles_per_head;
                    const int t = t0 + st % tiles_per_head;
                    mbar_arrive_expect_tx(bar(BAR_FULL + s), 2 * G::kTileBytes + 2 * kVecBytes);
                    for (int h = 0; h < G::kHalves; ++h) {
                        tma_load_4d(sbase + G::kRing0 + s * G::kTileBytes + h * kHalfBytes, &tm_q, h * 64, hq,
                                    t * kBM, b, bar(BAR_FULL + s), pol_stream);
                        tma_load_4d(sbase + G::kRing1 + s * G::kTileBytes + h * kHalfBytes, &tm_do, h * 64, hq,
                                    t * kBM, b, bar(BAR_FULL + s), pol_stream);
                    }
                    const size_t vo = (static_cast<size_t>(b) * p.Hq + hq) * p.sq_pad + static_cast<size_t>(t) * kBM;
                    bulk_load(sbase + G::kVec + s * 2 * kVecBytes, p.lse2 + vo, kVecBytes, bar(BAR_FULL + s));
                    bulk_load(sbase + G::kVec + s * 2 * kVecBytes + kVecBytes, p.delta + vo, kVecBytes,
                              bar(BAR_FULL + s));
                }
                if (!ok) break;
            }
            // drain: every copy issued has landed before the CTA may exit
            if (kfix > 0) drain_bounded(bar(BAR_KFULL), (kfix - 1) & 1, limit);
            if (vfix > 0) drain_bounded(bar(BAR_VFULL), (vfix - 1) & 1, limit);
            for (int s = 0; s < kStages; ++s) {
                const int fills = g > s ? (g - 1 - s) / kStages + 1 : 0;
                if (fills) drain_bounded(bar(BAR_FULL + s), (fills - 1) & 1, limit);
            }
        }
        __syncwarp();
        // release warp of the abort path: the elementwise warps' arrivals
        release_named_barriers(mma_exit, abort_flag, kBarPReady, 2, kBarReadyThreads, kComputeWarps, limit);
    } else if (warp == kMmaWarp) {
        // =========================== MMA issuer =============================
        constexpr uint32_t idesc_s = idesc_f16kind_f32(kBN, kBM, false, kF16);  // S^T, dP^T
        constexpr uint32_t idesc_acc = idesc_f16kind_f32(kBN, kD, true, kF16);  // dV, dK
        const uint64_t k_desc = sdesc_sw128(sbase + G::kFix0, 16, 1024);
        const uint64_t v_desc = sdesc_sw128(sbase + G::kFix1, 16, 1024);
        const uint64_t q_k0 = sdesc_sw128(sbase + G::kRing0, 16, 1024);
        const uint64_t do_k0 = sdesc_sw128(sbase + G::kRing1, 16, 1024);
        const uint64_t q_mn0 = sdesc_sw128(sbase + G::kRing0, kHalfBytes, 1024);
        const uint64_t do_mn0 = sdesc_sw128(sbase + G::kRing1, kHalfBytes, 1024);
        const uint32_t tS = tmem_base + G::kTmemS, tDP = tmem_base + G::kTmemDP;
        const uint32_t tDV = tmem_base + G::kTmemAcc0, tDK = tmem_base + G::kTmemAcc1;
        // Per item, issue order S^T_0, dP^T_0, then per step t:
        //   dV_t, S^T_{t+1}, dK_t, dP^T_{t+1}
        // so each elementwise phase (P^T_t before dV_t, dS^T_t before dK_t) is
        // covered by two products.  S^T_{t+1} overwrites P^T_t after dV_t has read
        // it and dP^T_{t+1} overwrites dS^T_t after dK_t (one thread's tcgen05
        // MMAs execute in issue order).  g counts steps over all items.
        auto stage_off = [](int gs) { return static_cast<uint64_t>(((gs % kStages) * G::kTileBytes) >> 4); };
        auto issue_s = [&](int gs) -> bool {  // S^T of global step gs; its stage must have landed
            if (!wait_bounded(bar(BAR_FULL + gs % kStages), (gs / kStages) & 1, abort_flag, limit)) return false;
            tc_fence_after();
            if (elect_one()) {
                mma_kmajor<kD>(tS, k_desc, q_k0 + stage_off(gs), idesc_s);
                mma_commit(bar(BAR_SFULL));
            }
            __syncwarp();
            return true;
        };
        auto issue_dp = [&](int gs) {
            if (elect_one()) {
                mma_kmajor<kD>(tDP, v_desc, do_k0 + stage_off(gs), idesc_s);
                mma_commit(bar(BAR_DPFULL));
            }
            __syncwarp();
        };
        auto commit_to = [&](int which) {
            if (elect_one()) mma_commit(bar(which));
            __syncwarp();
        };
        bool ok = true;
        int g = 0, w = 0;
        for (int j = 0; ok; ++j) {
            const int slot = j & 1;
            if (!wait_bounded(bar(BAR_ITEMFULL + slot), (j >> 1) & 1, abort_flag, limit)) break;
            const int u = item_slot[slot];
            __syncwarp();
            if (elect_one()) mbar_arrive(bar(BAR_ITEMEMPTY + slot));
            __syncwarp();
            if (u < 0) break;
            int b, hkv, n, t0, tiles_per_head;
            dkdv_item(p, u, b, hkv, n);
            const int steps = steps_of(n, t0, tiles_per_head);
            if (steps == 0) continue;
            ok = wait_bounded(bar(BAR_KFULL), w & 1, abort_flag, limit) && issue_s(g);
            if (!ok) break;
            if (steps == 1) commit_to(BAR_KEMPTY);  // the item's only S^T is issued
            ok = wait_bounded(bar(BAR_VFULL), w & 1, abort_flag, limit);
            if (!ok) break;
            tc_fence_after();
            issue_dp(g);
            if (steps == 1) commit_to(BAR_VEMPTY);
            for (int st = 0; ok && st < steps; ++st) {
                const int gs = g + st;
                named_bar_sync(kBarPReady, kBarReadyThreads);  // P^T_st in tensor memory
                tc_fence_after();
                if (elect_one()) mma_tmem_mn(tDV, tS, do_mn0 + stage_off(gs), idesc_acc, st > 0);
                __syncwarp();
                if (st + 1 < steps) {
                    if (!issue_s(gs + 1)) {
                        ok = false;
                        break;
                    }
                    if (st + 2 == steps) commit_to(BAR_KEMPTY);  // the item's last S^T is issued
                }
                named_bar_sync(kBarDsReady, kBarReadyThreads);  // dS^T_st in tensor memory
                tc_fence_after();
                if (elect_one()) {
                    mma_tmem_mn(tDK, tDP, q_mn0 + stage_off(gs), idesc_acc, st > 0);
                    mma_commit(bar(BAR_EMPTY + gs % kStages));
                    if (st == steps - 1) mma_commit(bar(BAR_ACCDONE));
                }
                __syncwarp();
                if (st + 1 < steps) {
                    issue_dp(gs + 1);
                    if (st + 2 == steps) commit_to(BAR_VEMPTY);  // the item's last dP^T is issued
                }
            }
            g += steps;
            ++w;
        }
        *mma_exit = 1;  // the release loop may stop
        if (elect_one()) {
            mma_commit(bar(BAR_MMADONE));
            drain_bounded(bar(BAR_MMADONE), 0, limit);
        }
        __syncwarp();
    } else {
        // =========================== elementwise warps ======================
        const int quarter = warp % 4, grp = warp / 4;
        const int jr = quarter * 32 + lane;  // key within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + G::kTmemS + kCols * grp;
        const uint32_t tP = tmem_base + lane_off + G::kTmemS + kCols * grp;  // packed over own fp32 columns
        const uint32_t tDP = tmem_base + lane_off + G::kTmemDP + kCols * grp;
        const uint32_t tDS = tmem_base + lane_off + G::kTmemDP + kCols * grp;  // packed over own fp32 columns
        const float sl2 = p.scale_log2;
        bool ok = true;
        int g = 0, w = 0;
        for (int j = 0; ok; ++j) {
            const int slot = j & 1;
            const bool got_item = wait_bounded(bar(BAR_ITEMFULL + slot), (j >> 1) & 1, abort_flag, limit);
            if (!__all_sync(0xffffffffu, got_item)) break;
            const int u = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(BAR_ITEMEMPTY + slot));
            if (u < 0) break;
            int b, hkv, n, t0, tiles_per_head;
            dkdv_item(p, u, b, hkv, n);
            const int steps = steps_of(n, t0, tiles_per_head);
            const int key = n * kBN + jr;
            for (int st = 0; st < steps; ++st) {
                const int gs = g + st;
                const int s = gs % kStages, use = gs / kStages;
                const int t = t0 + st % tiles_per_head;
                // the stage's lse2 / delta have landed (visible to this thread), and S^T is in TMEM
                const bool got = wait_bounded(bar(BAR_FULL + s), use & 1, abort_flag, limit) &&
                                 wait_bounded(bar(BAR_SFULL), gs & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float* l2 = reinterpret_cast<const float*>(smem + G::kVec + s * 2 * kVecBytes) + kCols * grp;
                const float* dl = l2 + kBM;
                uint32_t x[kCols];
                tmem_ld_cols<kCols>(tS, x);
                // row i = t*128 + 64*half + c sees this key iff key <= i + diag
                const int row0 = t * kBM + kCols * grp;
                const int cmin = p.causal ? key - p.diag - row0 : -1;  // first visible column
                float pv[kCols];
#pragma unroll
                for (int c = 0; c < kCols; c += 2) {
                    ffma2_b(pv[c], pv[c + 1], __uint_as_float(x[c]), __uint_as_float(x[c + 1]), sl2, -l2[c],
                            -l2[c + 1]);
                    pv[c] = ex2_approx(pv[c]);
                    pv[c + 1] = ex2_approx(pv[c + 1]);
                }
                if (cmin > 0) {
#pragma unroll
                    for (int c = 0; c < kCols; ++c)
                        if (c < cmin) pv[c] = 0.f;
                }
                {
                    uint32_t pk[kCols / 2];
#pragma unroll
                    for (int c = 0; c < kCols / 2; ++c) pk[c] = pack_x2<kF16>(pv[2 * c], pv[2 * c + 1]);
                    tmem_st_packed<kCols>(tP, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                named_bar_arrive(kBarPReady, kBarReadyThreads);
                const bool got2 = wait_bounded(bar(BAR_DPFULL), gs & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got2)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_ld_cols<kCols>(tDP, x);
                {
                    uint32_t pk[kCols / 2];
#pragma unroll
                    for (int c = 0; c < kCols; c += 2) {
                        float d0, d1;
                        fsubmul2(d0, d1, pv[c], pv[c + 1], __uint_as_float(x[c]), __uint_as_float(x[c + 1]), dl[c],
                                 dl[c + 1]);
                        pk[c / 2] = pack_x2<kF16>(d0, d1);
                    }
                    tmem_st_packed<kCols>(tDS, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                named_bar_arrive(kBarDsReady, kBarReadyThreads);
            }
            if (!ok) break;
            // epilogue: dV and scale * dK of this key, columns [grp kD/kGroups, (grp+1) kD/kGroups).
            // The accumulators are read out (tcgen05.ld completed) before this
            // thread's next arrival on the P barrier, which gates the next item's
            // first dV and dK.
            bool have = steps > 0;
            if (have) {
                const bool got = wait_bounded(bar(BAR_ACCDONE), w & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got)) break;
                tc_fence_after();
            }
            const bool write = key < p.Skv;
            const size_t off =
                ((static_cast<size_t>(b) * p.Skv + (write ? key : 0)) * p.Hkv + hkv) * kD + grp * (kD / kGroups);
            store_acc_part<kF16, kD>(tmem_base + lane_off + G::kTmemAcc0 + grp * (kD / kGroups), have, 1.f, p.dv + off,
                                     write);
            store_acc_part<kF16, kD>(tmem_base + lane_off + G::kTmemAcc1 + grp * (kD / kGroups), have, p.scale,
                                     p.dk + off, write);
            if (have) {
                g += steps;
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

// ---------------------------------------------------------------- dQ
// Shared memory of the dQ kernel: Q and dO fixed, then separate rings for K
// (three stages: read by S_n and, at the end of the step, by dQ_n) and V (two
// stages: read only by dP_n, so a V stage frees early).
template <int kD>
struct DqGeo {
    static_assert(kD == 64 || kD == 128, "head size 64 or 128");
    static constexpr int kHalves = kD / 64;
    static constexpr int kTileBytes = kBM * kD * 2;
    static constexpr int kKStages = 3, kVStages = 2;
    static constexpr int kFix0 = 0;                                  // Q
    static constexpr int kFix1 = kTileBytes;                         // dO
    static constexpr int kKRing = 2 * kTileBytes;
    static constexpr int kVRing = kKRing + kKStages * kTileBytes;
    static constexpr int kBar = kVRing + kVStages * kTileBytes;
    static constexpr int kTmemSlot = kBar + 24 * 8;
    static constexpr int kAbort = kTmemSlot + 4;
    static constexpr int kItems = kAbort + 4;          // [2] published work items
    static constexpr int kMmaExit = kItems + 8;        // set once the MMA warp left its loop
    static constexpr int kSmemBytes = kMmaExit + 4 + 1024;
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
    static constexpr uint32_t kTmemS = 0, kTmemDP = 128, kTmemDQ = 256;
};

enum : int {
    DQB_QFULL = 0,        // the item's Q landed
    DQB_QEMPTY,           // its last S completed: Q may be replaced
    DQB_DOFULL,
    DQB_DOEMPTY,          // its last dP completed: dO may be replaced
    DQB_KFULL,            // [K stage]
    DQB_KEMPTY = DQB_KFULL + 3,
    DQB_VFULL = DQB_KEMPTY + 3,   // [V stage]
    DQB_VEMPTY = DQB_VFULL + 2,
    DQB_SFULL = DQB_VEMPTY + 2,
    DQB_DPFULL,
    DQB_ACCDONE,          // the item's last dQ product completed
    DQB_ITEMFULL,         // [2]
    DQB_ITEMEMPTY = DQB_ITEMFULL + 2,  // [2]
    DQB_MMADONE = DQB_ITEMEMPTY + 2,
    DQB_COUNT
};
static_assert(DQB_COUNT <= 24, "barrier area");
// Work item u = one (b, hq, 128-row query tile), numbered in blocks of
// kItemHeads query heads: within a block by row tile (under a causal mask the
// last tiles visit the most KV tiles and go first), then by head, so the CTAs
// in flight stream the K/V of a few heads (of one GQA group) out of L2.
__host__ __device__ __forceinline__ void dq_item(const BwdParams& p, int u, int& b, int& hq, int& t) {
    const int nbh = p.B * p.Hq;
    const int per_block = kItemHeads * p.n_q_tiles;
    const int blk = u / per_block;
    const int within = u - blk * per_block;
    const int heads = nbh - blk * kItemHeads < kItemHeads ? nbh - blk * kItemHeads : kItemHeads;
    const int tr = within / heads;
    const int bh = blk * kItemHeads + (within - tr * heads);
    t = p.causal ? p.n_q_tiles - 1 - tr : tr;
    b = bh / p.Hq;
    hq = bh % p.Hq;
}

// Persistent, like the dK/dV kernel: items from the second queue, Q and dO of
// the next item loaded as soon as the current item's last S / dP has read
// them, K/V rings and per-step barriers running on across items; the next
// item's first dQ product (which starts the accumulator afresh) waits for the
// elementwise warps' next dS, issued after they read the accumulator out.
template <bool kF16, int kD>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdParams p) {
    using G = DqGeo<kD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::kAbort);
    volatile int* item_slot = reinterpret_cast<volatile int*>(smem + G::kItems);
    volatile int* mma_exit = reinterpret_cast<volatile int*>(smem + G::kMmaExit);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + G::kBar + 8 * i; };
    const int n_items = p.B * p.Hq * p.n_q_tiles;
    const unsigned int limit = p.poll_limit;

    if (warp == kLoadWarp && lane == 0) {
        mbar_init(bar(DQB_QFULL), 1);
        mbar_init(bar(DQB_QEMPTY), 1);
        mbar_init(bar(DQB_DOFULL), 1);
        mbar_init(bar(DQB_DOEMPTY), 1);
        for (int s = 0; s < G::kKStages; ++s) {
            mbar_init(bar(DQB_KFULL + s), 1);
            mbar_init(bar(DQB_KEMPTY + s), 1);
        }
        for (int s = 0; s < G::kVStages; ++s) {
            mbar_init(bar(DQB_VFULL + s), 1);
            mbar_init(bar(DQB_VEMPTY + s), 1);
        }
        mbar_init(bar(DQB_SFULL), 1);
        mbar_init(bar(DQB_DPFULL), 1);
        mbar_init(bar(DQB_ACCDONE), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(DQB_ITEMFULL + i), 1);
            mbar_init(bar(DQB_ITEMEMPTY + i), 1 + kComputeWarps);
        }
        mbar_init(bar(DQB_MMADONE), 1);
        *abort_flag = 0;
        *mma_exit = 0;
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
            int g = 0, w = 0;          // KV steps loaded, items with work loaded
            int kf = 0, vf = 0;        // K and V fills issued (for the drain)
            int qfix = 0, dofix = 0;   // Q and dO fills issued
            for (int j = 0;; ++j) {
                const int slot = j & 1;
                if (j >= 2 && !wait_bounded(bar(DQB_ITEMEMPTY + slot), ((j >> 1) - 1) & 1, abort_flag, limit)) break;
                int u = *abort_flag ? -1 : atomicAdd(p.work + 1, 1);
                if (u >= n_items) u = -1;
                item_slot[slot] = u;
                mbar_arrive(bar(DQB_ITEMFULL + slot));
                if (u < 0) break;
                int b, hq, t;
                dq_item(p, u, b, hq, t);
                const int hkv = hq / (p.Hq / p.Hkv);
                const int nkv = kv_tiles_for_rows(p, t * kBM);
                if (nkv == 0) continue;
                if (w > 0 && !wait_bounded(bar(DQB_QEMPTY), (w - 1) & 1, abort_flag, limit)) break;
                mbar_arrive_expect_tx(bar(DQB_QFULL), G::kTileBytes);
                for (int h = 0; h < G::kHalves; ++h)
                    tma_load_4d(sbase + G::kFix0 + h * kHalfBytes, &tm_q, h * 64, hq, t * kBM, b, bar(DQB_QFULL),
                                pol_fix);
                ++qfix;
                if (w > 0 && !wait_bounded(bar(DQB_DOEMPTY), (w - 1) & 1, abort_flag, limit)) break;
                mbar_arrive_expect_tx(bar(DQB_DOFULL), G::kTileBytes);
                for (int h = 0; h < G::kHalves; ++h)
                    tma_load_4d(sbase + G::kFix1 + h * kHalfBytes, &tm_do, h * 64, hq, t * kBM, b, bar(DQB_DOFULL),
                                pol_fix);
                ++dofix;
                ++w;
                bool ok = true;
                for (int kt = 0; kt < nkv; ++kt, ++g) {
                    const int ks = g % G::kKStages, kuse = g / G::kKStages;
                    if (kuse > 0 && !wait_bounded(bar(DQB_KEMPTY + ks), (kuse - 1) & 1, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(DQB_KFULL + ks), G::kTileBytes);
                    for (int h = 0; h < G::kHalves; ++h)
                        tma_load_4d(sbase + G::kKRing + ks * G::kTileBytes + h * kHalfBytes, &tm_k, h * 64, hkv,
                                    kt * kBN, b, bar(DQB_KFULL + ks), pol_stream);
                    ++kf;
                    const int vs = g % G::kVStages, vuse = g / G::kVStages;
                    if (vuse > 0 && !wait_bounded(bar(DQB_VEMPTY + vs), (vuse - 1) & 1, abort_flag, limit)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(bar(DQB_VFULL + vs), G::kTileBytes);
                    for (int h = 0; h < G::kHalves; ++h)
                        tma_load_4d(sbase + G::kVRing + vs * G::kTileBytes + h * kHalfBytes, &tm_v, h * 64, hkv,
                                    kt * kBN, b, bar(DQB_VFULL + vs), pol_stream);
                    ++vf;
                }
                if (!ok) break;
            }
            // drain: every copy issued has landed before the CTA may exit
            if (qfix > 0) drain_bounded(bar(DQB_QFULL), (qfix - 1) & 1, limit);
            if (dofix > 0) drain_bounded(bar(DQB_DOFULL), (dofix - 1) & 1, limit);
            for (int s = 0; s < G::kKStages; ++s) {
                const int fills = kf > s ? (kf - 1 - s) / G::kKStages + 1 : 0;
                if (fills) drain_bounded(bar(DQB_KFULL + s), (fills - 1) & 1, limit);
            }
            for (int s = 0; s < G::kVStages; ++s) {
                const int fills = vf > s ? (vf - 1 - s) / G::kVStages + 1 : 0;
                if (fills) drain_bounded(bar(DQB_VFULL + s), (fills - 1) & 1, limit);
            }
        }
        __syncwarp();
        // release warp of the abort path: the elementwise warps' arrivals
        release_named_barriers(mma_exit, abort_flag, kBarPReady, 2, kBarReadyThreads, kComputeWarps, limit);
    } else if (warp == kMmaWarp) {
        // =========================== MMA issuer =============================
        constexpr uint32_t idesc_s = idesc_f16kind_f32(kBM, kBN, false, kF16);  // S, dP
        constexpr uint32_t idesc_acc = idesc_f16kind_f32(kBM, kD, true, kF16);  // dQ
        const uint64_t q_desc = sdesc_sw128(sbase + G::kFix0, 16, 1024);
        const uint64_t do_desc = sdesc_sw128(sbase + G::kFix1, 16, 1024);
        const uint64_t k_k0 = sdesc_sw128(sbase + G::kKRing, 16, 1024);
        const uint64_t v_k0 = sdesc_sw128(sbase + G::kVRing, 16, 1024);
        const uint64_t k_mn0 = sdesc_sw128(sbase + G::kKRing, kHalfBytes, 1024);
        const uint32_t tS = tmem_base + G::kTmemS, tDP = tmem_base + G::kTmemDP;
        const uint32_t tDQ = tmem_base + G::kTmemDQ;
        // Per item, issue order S_0, dP_0, then per KV tile n:
        //   [S_n read out] S_{n+1}, [dS_n stored] dQ_n, dP_{n+1}
        // The elementwise warps signal (P barrier) as soon as S_n is in their
        // registers, so S_{n+1} runs while they form P_n and dS_n; dP_{n+1}
        // overwrites dS_n only after dQ_n (issue order).  A V stage is released
        // right after its dP, a K stage after its dQ.  g counts KV steps over all
        // items; the P barrier is met on every step, including an item's last, so
        // the next item's S_0 never overwrites an S still being read.
        auto issue_s = [&](int gk) -> bool {  // S of global KV step gk; its K must have landed
            const int ks = gk % G::kKStages;
            if (!wait_bounded(bar(DQB_KFULL + ks), (gk / G::kKStages) & 1, abort_flag, limit)) return false;
            tc_fence_after();
            if (elect_one()) {
                mma_kmajor<kD>(tS, q_desc, k_k0 + static_cast<uint64_t>((ks * G::kTileBytes) >> 4), idesc_s);
                mma_commit(bar(DQB_SFULL));
            }
            __syncwarp();
            return true;
        };
        auto issue_dp = [&](int gk) -> bool {  // dP of global KV step gk; its V must have landed
            const int vs = gk % G::kVStages;
            if (!wait_bounded(bar(DQB_VFULL + vs), (gk / G::kVStages) & 1, abort_flag, limit)) return false;
            tc_fence_after();
            if (elect_one()) {
                mma_kmajor<kD>(tDP, do_desc, v_k0 + static_cast<uint64_t>((vs * G::kTileBytes) >> 4), idesc_s);
                mma_commit(bar(DQB_DPFULL));
                mma_commit(bar(DQB_VEMPTY + vs));
            }
            __syncwarp();
            return true;
        };
        auto commit_to = [&](int which) {
            if (elect_one()) mma_commit(bar(which));
            __syncwarp();
        };
        bool ok = true;
        int g = 0, w = 0;
        for (int j = 0; ok; ++j) {
            const int slot = j & 1;
            if (!wait_bounded(bar(DQB_ITEMFULL + slot), (j >> 1) & 1, abort_flag, limit)) break;
            const int u = item_slot[slot];
            __syncwarp();
            if (elect_one()) mbar_arrive(bar(DQB_ITEMEMPTY + slot));
            __syncwarp();
            if (u < 0) break;
            int b, hq, t;
            dq_item(p, u, b, hq, t);
            const int nkv = kv_tiles_for_rows(p, t * kBM);
            if (nkv == 0) continue;
            // the previous item's last S must have been read out before S_0 overwrites it
            if (g > 0) named_bar_sync(kBarPReady, kBarReadyThreads);
            ok = wait_bounded(bar(DQB_QFULL), w & 1, abort_flag, limit) && issue_s(g);
            if (!ok) break;
            if (nkv == 1) commit_to(DQB_QEMPTY);
            ok = wait_bounded(bar(DQB_DOFULL), w & 1, abort_flag, limit) && issue_dp(g);
            if (!ok) break;
            if (nkv == 1) commit_to(DQB_DOEMPTY);
            for (int kt = 0; ok && kt < nkv; ++kt) {
                const int gk = g + kt;
                const int ks = gk % G::kKStages;
                const uint64_t so = static_cast<uint64_t>((ks * G::kTileBytes) >> 4);
                if (kt + 1 < nkv) {
                    named_bar_sync(kBarPReady, kBarReadyThreads);  // S_kt read out of tensor memory
                    if (!issue_s(gk + 1)) {
                        ok = false;
                        break;
                    }
                    if (kt + 2 == nkv) commit_to(DQB_QEMPTY);  // the item's last S is issued
                }
                named_bar_sync(kBarDsReady, kBarReadyThreads);  // dS_kt in tensor memory
                tc_fence_after();
                if (elect_one()) {
                    mma_tmem_mn(tDQ, tDP, k_mn0 + so, idesc_acc, kt > 0);
                    mma_commit(bar(DQB_KEMPTY + ks));
                    if (kt == nkv - 1) mma_commit(bar(DQB_ACCDONE));
                }
                __syncwarp();
                if (kt + 1 < nkv) {
                    if (!issue_dp(gk + 1)) {
                        ok = false;
                        break;
                    }
                    if (kt + 2 == nkv) commit_to(DQB_DOEMPTY);  // the item's last dP is issued
                }
            }
            g += nkv;
            ++w;
        }
        // the last item's last S read-out is the one signal not yet met (each
        // other one is met before the S that follows it)
        if (ok && g > 0) named_bar_sync(kBarPReady, kBarReadyThreads);
        *mma_exit = 1;  // the release loop may stop
        if (elect_one()) {
            mma_commit(bar(DQB_MMADONE));
            drain_bounded(bar(DQB_MMADONE), 0, limit);
        }
        __syncwarp();
    } else {
        // =========================== elementwise warps ======================
        const int quarter = warp % 4, grp = warp / 4;
        const int r = quarter * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + G::kTmemS + kCols * grp;
        const uint32_t tDP = tmem_base + lane_off + G::kTmemDP + kCols * grp;
        const uint32_t tDS = tmem_base + lane_off + G::kTmemDP + kCols * grp;  // packed over own fp32 columns
        const float sl2 = p.scale_log2;
        bool ok = true;
        int g = 0, w = 0;
        for (int j = 0; ok; ++j) {
            const int slot = j & 1;
            const bool got_item = wait_bounded(bar(DQB_ITEMFULL + slot), (j >> 1) & 1, abort_flag, limit);
            if (!__all_sync(0xffffffffu, got_item)) break;
            const int u = item_slot[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(DQB_ITEMEMPTY + slot));
            if (u < 0) break;
            int b, hq, t;
            dq_item(p, u, b, hq, t);
            const int nkv = kv_tiles_for_rows(p, t * kBM);
            const int row = t * kBM + r;
            const size_t vo = (static_cast<size_t>(b) * p.Hq + hq) * p.sq_pad + row;  // row < sq_pad
            const float neg_l2 = -p.lse2[vo];
            const float dlt = p.delta[vo];
            // last visible key of this row (keys past Skv are masked too)
            const long long lim_ll =
                p.causal ? min((long long)row + p.diag, (long long)p.Skv - 1) : (long long)p.Skv - 1;
            const int lim = static_cast<int>(lim_ll < -1 ? -1 : lim_ll);
            for (int kt = 0; kt < nkv; ++kt) {
                const int gk = g + kt;
                const bool got = wait_bounded(bar(DQB_SFULL), gk & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t x[kCols];
                tmem_ld_cols<kCols>(tS, x);
                tc_fence_before();
                named_bar_arrive(kBarPReady, kBarReadyThreads);  // S may now be overwritten by the next tile's product
                float pv[kCols];
#pragma unroll
                for (int c = 0; c < kCols; c += 2) {
                    ffma2_bc(pv[c], pv[c + 1], __uint_as_float(x[c]), __uint_as_float(x[c + 1]), sl2, neg_l2);
                    pv[c] = ex2_approx(pv[c]);
                    pv[c + 1] = ex2_approx(pv[c + 1]);
                }
                const int nvis = lim - (kt * kBN + kCols * grp) + 1;  // visible columns of this group
                if (nvis < kCols) {
#pragma unroll
                    for (int c = 0; c < kCols; ++c)
                        if (c >= nvis) pv[c] = 0.f;
                }
                const bool got2 = wait_bounded(bar(DQB_DPFULL), gk & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got2)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                tmem_ld_cols<kCols>(tDP, x);
                {
                    uint32_t pk[kCols / 2];
#pragma unroll
                    for (int c = 0; c < kCols; c += 2) {
                        float d0, d1;
                        fsubmul2(d0, d1, pv[c], pv[c + 1], __uint_as_float(x[c]), __uint_as_float(x[c + 1]), dlt,
                                 dlt);
                        pk[c / 2] = pack_x2<kF16>(d0, d1);
                    }
                    tmem_st_packed<kCols>(tDS, pk);
                }
                tmem_wait_st();
                tc_fence_before();
                named_bar_arrive(kBarDsReady, kBarReadyThreads);
            }
            if (!ok) break;
            // epilogue: scale * dQ of this row, columns [grp kD/kGroups, (grp+1) kD/kGroups); the
            // accumulator is read out before this thread's next dS-barrier arrival, which gates
            // the next item's first dQ product
            const bool have = nkv > 0;
            if (have) {
                const bool got = wait_bounded(bar(DQB_ACCDONE), w & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got)) break;
                tc_fence_after();
            }
            const bool write = row < p.Sq;
            const size_t off = ((static_cast<size_t>(b) * p.Sq + (write ? row : 0)) * p.Hq + hq) * kD + grp * (kD / kGroups);
            store_acc_part<kF16, kD>(tmem_base + lane_off + G::kTmemDQ + grp * (kD / kGroups), have, p.scale, p.dq + off,
                                     write);
            if (have) {
                g += nkv;
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

}  // namespace bwd
}  // namespace attn
