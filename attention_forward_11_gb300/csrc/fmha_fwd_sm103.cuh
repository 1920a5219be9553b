// fmha_fwd_sm103.cuh -- fused attention forward for sm_103a (GB300).
//
// One CTA owns two 128-row query tiles that read the same K/V head: either two
// consecutive row tiles of one query head, or (when the GQA group has an even
// number of query heads) the same rows of two query heads of one group, so
// every K/V tile brought into shared memory feeds 256 query rows.
//
// Warp roles (320 threads):
//   warps 0-3  softmax warpgroup of tile 0 (one query row per thread)
//   warps 4-7  softmax warpgroup of tile 1
//   warp  8    MMA issuer (one thread): S_t = Q_t K^T and O_t += P_t V on tcgen05
//   warp  9    TMA producer (one thread): Q once, then K and V tiles through
//              two shared-memory rings guarded by full/empty mbarriers
//
// Tensor memory (512 columns x 128 lanes, fp32): S_0 | S_1 | O_0 | O_1, 128 columns
// each.  P_t (bf16, two per column) is written over the first 64 columns of S_t
// and is the A operand of the P.V product straight from tensor memory.
//
// The online softmax follows the Pallas page's kernel loop (`kv_loop`): the row
// maximum is kept in log2 units of the scaled logits so that each weight is one
// FMA and one ex2 (scale * log2e folded into the FMA), the running sum is
// rescaled by alpha = 2^(m_old - m_new), and O is divided by the sum once at the
// end.  The maximum used for the exponentials is only raised when the tile
// maximum exceeds it by more than 2^8; otherwise the stale maximum is kept
// (weights stay <= 256, exact in the same arithmetic since l and O share it),
// so O in tensor memory is rescaled only on the rare tiles that raise it.
//
// Causal (bottom-right aligned: key j visible from row i iff j <= i + Skv - Sq):
// KV tiles entirely above a tile's last visible key are never loaded or
// multiplied; the element mask is applied only on the tiles that cross the
// diagonal or the ragged key tail.  Row tiles are launched longest first (the
// Choreo tutorial's non-persistent schedule) so the short tiles fill the tail.
//
// Every mbarrier wait is bounded: when a wait runs out, the thread records
// ATTN_ERR_TIMEOUT in the device status word and raises a CTA abort flag; all
// roles then leave their loops, in-flight TMA loads and MMAs are drained with
// bounded waits, and tensor memory is freed before the CTA exits.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "sm103_ptx.cuh"

namespace attn {

constexpr int kBM = 128;                 // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;                 // keys per KV tile
constexpr int kHeadDim = 128;            // D
constexpr int kTiles = 2;                // query tiles per CTA
constexpr int kKStages = 2;              // K ring depth
constexpr int kVStages = 2;              // V ring depth
constexpr int kTileBytes = kBM * kHeadDim * 2;   // 32 KB bf16 tile (Q, K or V)
constexpr int kHalfBytes = kTileBytes / 2;       // one 64-column, 128-byte-swizzled half
constexpr int kSoftmaxWarps = 4 * kTiles;
constexpr int kMmaWarp = kSoftmaxWarps;
constexpr int kLoadWarp = kSoftmaxWarps + 1;
constexpr int kThreads = 32 * (kSoftmaxWarps + 2);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;           // S_t at kTmemS + 128 t
constexpr uint32_t kTmemO = 256;         // O_t at kTmemO + 128 t
constexpr float kRescaleLog2 = 8.0f;     // raise the running max only past 2^8

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kSmemQ = 0;
constexpr int kSmemK = kSmemQ + kTiles * kTileBytes;
constexpr int kSmemV = kSmemK + kKStages * kTileBytes;
constexpr int kSmemBar = kSmemV + kVStages * kTileBytes;
enum : int {
    BAR_Q = 0,
    BAR_KFULL = 1,
    BAR_KEMPTY = BAR_KFULL + kKStages,
    BAR_VFULL = BAR_KEMPTY + kKStages,
    BAR_VEMPTY = BAR_VFULL + kVStages,
    BAR_SFULL = BAR_VEMPTY + kVStages,
    BAR_PFULL = BAR_SFULL + kTiles,
    BAR_ODONE = BAR_PFULL + kTiles,
    BAR_MMADONE = BAR_ODONE + kTiles,
    BAR_COUNT
};
constexpr int kSmemTmemSlot = kSmemBar + BAR_COUNT * 8;
constexpr int kSmemAbort = kSmemTmemSlot + 4;
constexpr int kSmemUsed = kSmemAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // + slack to align the base to 1024 bytes
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");

constexpr unsigned int kStatusTimeout = 1u;

// Device status word: bit 0 = a bounded wait ran out.  Read and cleared by the host.
__device__ unsigned int g_attn_status = 0;

struct FwdParams {
    int B, Sq, Skv, Hq, Hkv;
    int causal;             // 0 or 1 (bottom-right)
    float scale_log2;       // softmax scale * log2(e)
    float* lse;             // [B, Hq, Sq] fp32, or nullptr
    int head_pairs;         // 1: the CTA's tiles are two heads of a GQA group, same rows
    int n_row_units;        // row units per (batch, head unit)
    int n_head_units;       // head units per batch
    unsigned int poll_limit;  // bound on every mbarrier poll loop
};

// Bounded wait on an mbarrier phase.  Gives up (returns false) if the CTA abort
// flag is raised, or after `limit` polls (then it raises the flag itself).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int limit) {
    for (unsigned int i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    *abort_flag = 1;
    atomicOr(&g_attn_status, kStatusTimeout);
    return false;
}

// Same, ignoring the abort flag: used to drain in-flight copies and MMAs.
__device__ __forceinline__ bool drain_bounded(uint32_t bar, uint32_t parity, unsigned int limit) {
    for (unsigned int i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    atomicOr(&g_attn_status, kStatusTimeout);
    return false;
}

// tcgen05.wait::ld that also orders the loaded registers after the wait
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.wait::ld.sync.aligned;"
        : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
          "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
          "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
          "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
          "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
          "+r"(r[31])
        :
        : "memory");
}

// Number of KV tiles a query tile [row0, row0 + 128) must visit.
__device__ __forceinline__ int kv_tiles_for(const FwdParams& p, int row0) {
    if (row0 >= p.Sq) return 0;
    const int n_all = (p.Skv + kBN - 1) / kBN;
    if (!p.causal) return n_all;
    const int last_row = min(row0 + kBM - 1, p.Sq - 1);
    const long long last_key = (long long)last_row + (p.Skv - p.Sq);
    if (last_key < 0) return 0;
    const long long n = last_key / kBN + 1;
    return n < n_all ? (int)n : n_all;
}

__global__ void __launch_bounds__(kThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    // align in the shared window (swizzle atoms and TMA boxes want 1024 bytes)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kSmemTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + kSmemBar + 8 * i; };

    // ---- work unit of this CTA (longest causal row units first)
    const int inner_count = p.B * p.n_head_units;
    const int ru = static_cast<int>(blockIdx.x) / inner_count;
    const int inner = static_cast<int>(blockIdx.x) % inner_count;
    const int b = inner / p.n_head_units;
    const int hu = inner % p.n_head_units;
    const int row_unit = p.causal ? (p.n_row_units - 1 - ru) : ru;
    int hq_t[kTiles], row0_t[kTiles], n_t[kTiles];
    if (p.head_pairs) {
        hq_t[0] = 2 * hu;
        hq_t[1] = 2 * hu + 1;
        row0_t[0] = row0_t[1] = row_unit * kBM;
    } else {
        hq_t[0] = hq_t[1] = hu;
        row0_t[0] = row_unit * (kTiles * kBM);
        row0_t[1] = row0_t[0] + kBM;
    }
    const int hkv = hq_t[0] / (p.Hq / p.Hkv);
    n_t[0] = kv_tiles_for(p, row0_t[0]);
    n_t[1] = kv_tiles_for(p, row0_t[1]);
    const int n_max = max(n_t[0], n_t[1]);

    // ---- set-up: barriers, abort flag, tensor memory
    if (warp == kLoadWarp && lane == 0) {
        mbar_init(bar(BAR_Q), 1);
        for (int s = 0; s < kKStages; ++s) {
            mbar_init(bar(BAR_KFULL + s), 1);
            mbar_init(bar(BAR_KEMPTY + s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            mbar_init(bar(BAR_VFULL + s), 1);
            mbar_init(bar(BAR_VEMPTY + s), 1);
        }
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bar(BAR_SFULL + t), 1);
            mbar_init(bar(BAR_PFULL + t), 4 * 32);
            mbar_init(bar(BAR_ODONE + t), 1);
        }
        mbar_init(bar(BAR_MMADONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const unsigned int limit = p.poll_limit;

    if (warp == kLoadWarp) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            mbar_arrive_expect_tx(bar(BAR_Q), kTiles * kTileBytes);
            for (int t = 0; t < kTiles; ++t)
                for (int h = 0; h < 2; ++h)
                    tma_load_4d(sbase + kSmemQ + t * kTileBytes + h * kHalfBytes, &tm_q, h * 64,
                                hq_t[t], row0_t[t], b, bar(BAR_Q), pol_q);
            int k_fills = 0, v_fills = 0;
            for (int kt = 0; kt < n_max; ++kt) {
                const int ks = kt % kKStages, kuse = kt / kKStages;
                if (kuse > 0 && !wait_bounded(bar(BAR_KEMPTY + ks), (kuse - 1) & 1, abort_flag, limit))
                    break;
                mbar_arrive_expect_tx(bar(BAR_KFULL + ks), kTileBytes);
                for (int h = 0; h < 2; ++h)
                    tma_load_4d(sbase + kSmemK + ks * kTileBytes + h * kHalfBytes, &tm_k, h * 64,
                                hkv, kt * kBN, b, bar(BAR_KFULL + ks), pol_kv);
                ++k_fills;
                const int vs = kt % kVStages, vuse = kt / kVStages;
                if (vuse > 0 && !wait_bounded(bar(BAR_VEMPTY + vs), (vuse - 1) & 1, abort_flag, limit))
                    break;
                mbar_arrive_expect_tx(bar(BAR_VFULL + vs), kTileBytes);
                for (int h = 0; h < 2; ++h)
                    tma_load_4d(sbase + kSmemV + vs * kTileBytes + h * kHalfBytes, &tm_v, h * 64,
                                hkv, kt * kBN, b, bar(BAR_VFULL + vs), pol_kv);
                ++v_fills;
            }
            // drain: every copy this thread issued has landed before the CTA may exit
            drain_bounded(bar(BAR_Q), 0, limit);
            for (int s = 0; s < kKStages; ++s) {
                const int fills = k_fills > s ? (k_fills - 1 - s) / kKStages + 1 : 0;
                if (fills) drain_bounded(bar(BAR_KFULL + s), (fills - 1) & 1, limit);
            }
            for (int s = 0; s < kVStages; ++s) {
                const int fills = v_fills > s ? (v_fills - 1 - s) / kVStages + 1 : 0;
                if (fills) drain_bounded(bar(BAR_VFULL + s), (fills - 1) & 1, limit);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // =========================== MMA issuer =============================
        if (lane == 0 && n_max > 0) {
            constexpr uint32_t idesc_qk = idesc_bf16_f32(kBM, kBN, false);
            constexpr uint32_t idesc_pv = idesc_bf16_f32(kBM, kHeadDim, true);
            auto issue_qk = [&](int t, int ks) {
                const uint32_t d = tmem_base + kTmemS + 128 * t;
                const uint32_t qa = sbase + kSmemQ + t * kTileBytes;
                const uint32_t kb = sbase + kSmemK + ks * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
                    mma_bf16_ss(d, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                                idesc_qk, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int vs, bool accumulate) {
                const uint32_t d = tmem_base + kTmemO + 128 * t;
                const uint32_t pa = tmem_base + kTmemS + 128 * t;
                const uint32_t vb = sbase + kSmemV + vs * kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_bf16_ts(d, pa + kk * 8, sdesc_sw128(vb + kk * 16 * 128, kHalfBytes, 1024),
                                idesc_pv, (accumulate || kk > 0) ? 1u : 0u);
            };
            bool ok = wait_bounded(bar(BAR_Q), 0, abort_flag, limit) &&
                      wait_bounded(bar(BAR_KFULL + 0), 0, abort_flag, limit);
            if (ok) {
                tc_fence_after();
                for (int t = 0; t < kTiles; ++t)
                    if (n_t[t] > 0) {
                        issue_qk(t, 0);
                        mma_commit(bar(BAR_SFULL + t));
                    }
                mma_commit(bar(BAR_KEMPTY + 0));
            }
            for (int kt = 0; ok && kt < n_max; ++kt) {
                const int vs = kt % kVStages, vuse = kt / kVStages;
                const int ks = (kt + 1) % kKStages, kuse = (kt + 1) / kKStages;
                if (!wait_bounded(bar(BAR_VFULL + vs), vuse & 1, abort_flag, limit)) break;
                tc_fence_after();
                bool k_ready = false;
                for (int t = 0; ok && t < kTiles; ++t) {
                    if (kt < n_t[t]) {
                        if (!wait_bounded(bar(BAR_PFULL + t), kt & 1, abort_flag, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_pv(t, vs, kt > 0);
                        if (kt == n_t[t] - 1) mma_commit(bar(BAR_ODONE + t));
                    }
                    if (kt + 1 < n_t[t]) {
                        if (!k_ready) {
                            if (!wait_bounded(bar(BAR_KFULL + ks), kuse & 1, abort_flag, limit)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            k_ready = true;
                        }
                        issue_qk(t, ks);
                        mma_commit(bar(BAR_SFULL + t));
                    }
                }
                if (!ok) break;
                mma_commit(bar(BAR_VEMPTY + vs));
                if (kt + 1 < n_max) mma_commit(bar(BAR_KEMPTY + ks));
            }
            // every MMA this thread issued has completed before tensor memory is freed
            mma_commit(bar(BAR_MMADONE));
            drain_bounded(bar(BAR_MMADONE), 0, limit);
        }
        __syncwarp();
    } else {
        // =========================== softmax warpgroups =====================
        const int t = warp / 4;
        const int wq = warp % 4;
        const int r = wq * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + kTmemS + 128 * t;
        const uint32_t tO = tmem_base + lane_off + kTmemO + 128 * t;
        const int row = row0_t[t] + r;
        const int nt = n_t[t];
        // last key this row may see
        const long long lim_ll =
            p.causal ? min((long long)row + (p.Skv - p.Sq), (long long)p.Skv - 1) : (long long)p.Skv - 1;
        const int lim = static_cast<int>(lim_ll < -1 ? -1 : lim_ll);
        const float sl2 = p.scale_log2;
        float m_run = -INFINITY;  // running max (log2 units of scaled logits) used by the weights
        float l_run = 0.f;        // running sum of weights
        bool ok = true;

        for (int kt = 0; kt < nt; ++kt) {
            // warp-uniform outcome: the tcgen05.ld/st below are warp-collective
            const bool got = wait_bounded(bar(BAR_SFULL + t), kt & 1, abort_flag, limit);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c)
                tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));

            const int nvis = lim - kt * kBN + 1;  // visible keys of this row in the tile
            if (nvis < kBN) {
#pragma unroll
                for (int j = 0; j < kBN; ++j)
                    if (j >= nvis) s[j] = __float_as_uint(-INFINITY);
            }
            float mx[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = __uint_as_float(s[u]);
#pragma unroll
            for (int j = 8; j < kBN; ++j) mx[j & 7] = fmaxf(mx[j & 7], __uint_as_float(s[j]));
            const float tmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
            const float m_tile = tmax * sl2;
            float alpha = 1.f;
            if (m_tile - m_run > kRescaleLog2) {  // false while both are -inf
                alpha = ex2_approx(m_run - m_tile);
                m_run = m_tile;
            }
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float p0 = ex2_approx(fmaf(__uint_as_float(s[32 * c + 2 * u]), sl2, -m_use));
                    const float p1 = ex2_approx(fmaf(__uint_as_float(s[32 * c + 2 * u + 1]), sl2, -m_use));
                    rs[c] += p0 + p1;
                    pk[u] = pack_bf16x2(p0, p1);
                }
                tmem_st16(tS + 16 * c, pk);
            }
            l_run = l_run * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
            // O_t holds P.V of tiles < kt (complete: S_t(kt) was issued after them)
            const bool need = (kt > 0) && (alpha != 1.f);
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tO + 32 * c, o);
                    tmem_wait_ld_regs(o);
#pragma unroll
                    for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
                    tmem_st32(tO + 32 * c, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(BAR_PFULL + t));
        }

        // ------------------------------ epilogue ------------------------------
        bool have = ok && nt > 0;
        if (have) have = wait_bounded(bar(BAR_ODONE + t), 0, abort_flag, limit);
        have = __all_sync(0xffffffffu, have);
        // the staging buffer is Q_t's: its TMA load must have landed (it may never
        // have been waited on when this tile had no KV tile to visit)
        drain_bounded(bar(BAR_Q), 0, limit);
        tc_fence_after();
        const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
        uint8_t* stage = smem + kSmemQ + t * kTileBytes;  // Q_t is dead once O_t is final
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            if (have) {
                tmem_ld32(tO + 32 * c, o);
                tmem_wait_ld_regs(o);
            } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) o[u] = 0u;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                uint4 val;
                val.x = pack_bf16x2(__uint_as_float(o[8 * u + 0]) * inv_l, __uint_as_float(o[8 * u + 1]) * inv_l);
                val.y = pack_bf16x2(__uint_as_float(o[8 * u + 2]) * inv_l, __uint_as_float(o[8 * u + 3]) * inv_l);
                val.z = pack_bf16x2(__uint_as_float(o[8 * u + 4]) * inv_l, __uint_as_float(o[8 * u + 5]) * inv_l);
                val.w = pack_bf16x2(__uint_as_float(o[8 * u + 6]) * inv_l, __uint_as_float(o[8 * u + 7]) * inv_l);
                const int half = c >> 1;
                const int chunk = (c & 1) * 4 + u;       // 16-byte chunk within the 128-byte row
                const int phys = chunk ^ (r & 7);         // 128-byte swizzle
                *reinterpret_cast<uint4*>(stage + half * kHalfBytes + r * 128 + phys * 16) = val;
            }
        }
        if (p.lse != nullptr && row < p.Sq) {
            const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
            p.lse[(static_cast<size_t>(b) * p.Hq + hq_t[t]) * p.Sq + row] = lse;
        }
        fence_proxy_async_smem();
        named_bar_sync(1 + t, 128);
        if (r == 0 && row0_t[t] < p.Sq && *abort_flag == 0) {
            for (int h = 0; h < 2; ++h)
                tma_store_4d(&tm_o, smem_u32(stage + h * kHalfBytes), h * 64, hq_t[t], row0_t[t], b);
            bulk_commit_group();
            bulk_wait_group0();
        }
    }

    // ---- teardown: all tensor-memory traffic is complete; free it
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing
// arrives on; the bounded wait runs out and records the timeout status.
__global__ void wait_timeout_selftest_kernel(unsigned int poll_limit) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ int abort_storage;
    if (threadIdx.x == 0) {
        abort_storage = 0;
        mbar_init(smem_u32(&bar_storage), 1);
        fence_mbar_init();
        wait_bounded(smem_u32(&bar_storage), 0, reinterpret_cast<volatile int*>(&abort_storage),
                     poll_limit);
    }
}

}  // namespace attn
