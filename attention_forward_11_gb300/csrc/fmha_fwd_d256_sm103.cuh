// fmha_fwd_d256_sm103.cuh -- attention forward for head size 256 on sm_103a.
//
// Same operation as fmha_fwd_kernel (the Pallas page's forward, with the
// caller's scale, the mask readings and the natural-log LSE), for D = 256:
// the Pallas page's benchmark sweeps head sizes 64, 128 and 256.
//
// At D = 256 one query tile's O needs 256 tensor-memory columns, so a CTA holds
// one 128-row tile and uses the rest of tensor memory to double-buffer S:
//   columns   0-127  S_0   (KV tiles 0, 2, 4, ...)
//   columns 128-255  S_1   (KV tiles 1, 3, 5, ...)
//   columns 256-511  O     (fp32, 128 rows x 256)
// The MMA warp issues S_0, S_1, then per KV tile j: [P_j stored] PV_j, S_{j+2},
// so the softmax of tile j runs while the tensor core computes S_{j+1} and
// PV_{j-1}.  P_j (bf16) is written over the first 64 columns of its S buffer,
// which S_{j+2} overwrites only after PV_j has read it (issue order).
//
// Shared memory: Q (128 x 256, four 64-column swizzled chunks, 64 KB); K and V
// tiles stream as halves of 128 keys x 128 columns (32 KB, two chunks) through
// a four-slot ring in the order the MMAs consume them: K_0, K_1, then per j
// V_j, K_{j+2} (each as two halves); a 16 KB staging chunk for the O store.
//
// Warps: 0-3 softmax (thread = query row = TMEM lane) and epilogue; warp 4
// issues the MMAs (one elected lane); warp 5 is the TMA producer.  Every
// mbarrier wait is bounded, as in the D <= 128 kernel.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "fmha_fwd_sm103.cuh"

namespace attn {
namespace d256 {

constexpr int kD = 256;
constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kSlots = 4;                      // ring of K/V halves
constexpr int kHalf = kBN * 128 * 2;           // 128 keys x 128 columns: 32 KB
constexpr int kChunk = kHalfBytes;             // 128 rows x 64 columns: 16 KB

enum : int {
    BAR_QFULL = 0,
    BAR_FULL = 1,                              // [slot]
    BAR_EMPTY = BAR_FULL + kSlots,             // [slot]
    BAR_SFULL = BAR_EMPTY + kSlots,            // [buffer]
    BAR_PFULL = BAR_SFULL + 2,                 // [buffer] (128 arrivals)
    BAR_PVDONE = BAR_PFULL + 2,                // after every PV (O rescale waits)
    BAR_ODONE = BAR_PVDONE + 1,                // after the last PV (once)
    BAR_MMADONE = BAR_ODONE + 1,
    BAR_COUNT
};

struct Geo {
    static constexpr int kSmemQ = 0;                          // 4 chunks
    static constexpr int kSmemRing = kSmemQ + 4 * kChunk;     // kSlots halves
    static constexpr int kSmemStage = kSmemRing + kSlots * kHalf;
    static constexpr int kSmemBar = kSmemStage + kChunk;
    static constexpr int kSmemTmemSlot = kSmemBar + BAR_COUNT * 8;
    static constexpr int kSmemAbort = kSmemTmemSlot + 4;
    static constexpr int kSmemBytes = kSmemAbort + 4 + 1024;
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

constexpr uint32_t kTmemO = 256;

// Work item of CTA u: query tile t of (b, hq) = u / n_t.  The CTAs of one head
// run side by side, so its K and V (4 MB at S = 4096) stay in L2 while they
// stream through them; within a head the tiles that visit the most KV tiles
// (the last ones under a causal mask) go first.
struct Item {
    int b, hq, hkv, row0, n;
};

__host__ __device__ __forceinline__ Item decode(const FwdParams& p, int u) {
    Item it;
    const int n_t = (p.Sq + kBM - 1) / kBM;
    const int bh = u / n_t;
    const int tr = u % n_t;
    const int t = p.causal ? n_t - 1 - tr : tr;
    it.b = bh / p.Hq;
    it.hq = bh % p.Hq;
    it.hkv = it.hq / (p.Hq / p.Hkv);
    it.row0 = t * kBM;
    it.n = kv_tiles_for(p, it.row0);
    return it;
}

// Ring sequence: fill f (0, 1, 2, ...) loads, in MMA consumption order,
//   K_0, K_1, then per j: V_j, K_{j+2} (when j + 2 < n), each as two halves.
// Returns the tensor (0 = K, 1 = V), KV tile and half of fill f.
__host__ __device__ __forceinline__ void fill_of(int f, int n, int& is_v, int& kv, int& half) {
    half = f & 1;
    const int g = f >> 1;  // tile load index
    if (g < 2 || n <= 2) {
        is_v = (n <= 2) ? (g >= n) : 0;
        kv = (n <= 2) ? (g < n ? g : g - n) : g;
        return;
    }
    // g >= 2 and n > 2: after K_0, K_1 the pattern is V_0, K_2, V_1, K_3, ...,
    // V_{n-3}, K_{n-1}, then V_{n-2}, V_{n-1}
    const int r = g - 2;
    const int pairs = n - 2;  // (V_j, K_{j+2}) for j < n - 2
    if (r < 2 * pairs) {
        is_v = (r & 1) == 0;
        kv = is_v ? r / 2 : r / 2 + 2;
    } else {
        is_v = 1;
        kv = n - 2 + (r - 2 * pairs);
    }
}

template <bool kF16>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_fwd_d256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Geo::kSmemAbort);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Geo::kSmemTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + Geo::kSmemBar + 8 * i; };
    const Item it = decode(p, static_cast<int>(blockIdx.x));
    const int n = it.n;
    const int n_fills = 4 * n;  // K and V of every KV tile, two halves each
    const unsigned int limit = p.poll_limit;

    if (warp == kLoadWarp && lane == 0) {
        mbar_init(bar(BAR_QFULL), 1);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar(BAR_FULL + s), 1);
            mbar_init(bar(BAR_EMPTY + s), 1);
        }
        for (int b2 = 0; b2 < 2; ++b2) {
            mbar_init(bar(BAR_SFULL + b2), 1);
            mbar_init(bar(BAR_PFULL + b2), 128);
        }
        mbar_init(bar(BAR_PVDONE), 1);
        mbar_init(bar(BAR_ODONE), 1);
        mbar_init(bar(BAR_MMADONE), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
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
        if (lane == 0 && n > 0) {
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            mbar_arrive_expect_tx(bar(BAR_QFULL), 4 * kChunk);
            for (int c = 0; c < 4; ++c)
                tma_load_4d(sbase + Geo::kSmemQ + c * kChunk, &tm_q, c * 64, it.hq, it.row0, it.b, bar(BAR_QFULL),
                            pol_q);
            int issued = 0;
            for (int f = 0; f < n_fills; ++f) {
                const int s = f % kSlots, use = f / kSlots;
                if (use > 0 && !wait_bounded(bar(BAR_EMPTY + s), (use - 1) & 1, abort_flag, limit)) break;
                int is_v, kv, half;
                fill_of(f, n, is_v, kv, half);
                mbar_arrive_expect_tx(bar(BAR_FULL + s), kHalf);
                const CUtensorMap* m = is_v ? &tm_v : &tm_k;
                for (int c = 0; c < 2; ++c)
                    tma_load_4d(sbase + Geo::kSmemRing + s * kHalf + c * kChunk, m, half * 128 + c * 64, it.hkv,
                                kv * kBN, it.b, bar(BAR_FULL + s), pol_kv);
                ++issued;
            }
            drain_bounded(bar(BAR_QFULL), 0, limit);
            for (int s = 0; s < kSlots; ++s) {
                const int fills = issued > s ? (issued - 1 - s) / kSlots + 1 : 0;
                if (fills) drain_bounded(bar(BAR_FULL + s), (fills - 1) & 1, limit);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // =========================== MMA issuer =============================
        constexpr uint32_t idesc_qk = idesc_f16kind_f32(kBM, kBN, false, kF16);
        constexpr uint32_t idesc_pv = idesc_f16kind_f32(kBM, 128, true, kF16);
        const uint64_t q_desc = sdesc_sw128(sbase + Geo::kSmemQ, 16, 1024);
        const uint64_t r_kdesc = sdesc_sw128(sbase + Geo::kSmemRing, 16, 1024);
        const uint64_t r_mndesc = sdesc_sw128(sbase + Geo::kSmemRing, kChunk, 1024);
        int f = 0;  // ring fills consumed so far
        bool ok = n > 0 && wait_bounded(bar(BAR_QFULL), 0, abort_flag, limit);
        // S_j = Q K_j^T: two halves of the head dimension, 8 k-steps each
        auto issue_s = [&](int j) -> bool {
            const uint32_t d = tmem_base + 128 * (j & 1);
            for (int h = 0; h < 2; ++h, ++f) {
                const int s = f % kSlots;
                if (!wait_bounded(bar(BAR_FULL + s), (f / kSlots) & 1, abort_flag, limit)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t qoff = static_cast<uint64_t>(((2 * h + (kk >> 2)) * kChunk + (kk & 3) * 32) >> 4);
                        const uint64_t koff = static_cast<uint64_t>((s * kHalf + (kk >> 2) * kChunk + (kk & 3) * 32) >> 4);
                        mma_bf16_ss(d, q_desc + qoff, r_kdesc + koff, idesc_qk, (h > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(BAR_EMPTY + s));
                    if (h == 1) mma_commit(bar(BAR_SFULL + (j & 1)));
                }
                __syncwarp();
            }
            return true;
        };
        // O[:, 128 h .. 128 h + 128) (+)= P_j V_j[:, 128 h .. 128 h + 128)
        auto issue_pv = [&](int j) -> bool {
            const uint32_t pa = tmem_base + 128 * (j & 1);
            for (int h = 0; h < 2; ++h, ++f) {
                const int s = f % kSlots;
                if (!wait_bounded(bar(BAR_FULL + s), (f / kSlots) & 1, abort_flag, limit)) return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_bf16_ts(tmem_base + kTmemO + 128 * h, pa + kk * 8,
                                    r_mndesc + static_cast<uint64_t>((s * kHalf + kk * 16 * 128) >> 4), idesc_pv,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(BAR_EMPTY + s));
                    if (h == 1) mma_commit(bar(BAR_PVDONE));
                }
                __syncwarp();
            }
            return true;
        };
        if (ok) ok = issue_s(0);
        if (ok && n > 1) ok = issue_s(1);
        for (int j = 0; ok && j < n; ++j) {
            // P_j stored by the softmax warps (and O rescaled, if it had to be)
            if (!wait_bounded(bar(BAR_PFULL + (j & 1)), (j >> 1) & 1, abort_flag, limit)) break;
            tc_fence_after();
            if (!issue_pv(j)) break;
            if (j == n - 1) {
                if (elect_one()) mma_commit(bar(BAR_ODONE));
                __syncwarp();
            }
            if (j + 2 < n && !issue_s(j + 2)) break;
        }
        if (elect_one()) {
            mma_commit(bar(BAR_MMADONE));
            drain_bounded(bar(BAR_MMADONE), 0, limit);
        }
        __syncwarp();
    } else {
        // =========================== softmax and epilogue ===================
        const int r = warp * 32 + lane;  // query row within the tile = TMEM lane
        const int row = it.row0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const uint32_t tO = tmem_base + lane_off + kTmemO;
        const float sl2 = p.scale_log2;
        const long long lim_ll = p.causal ? min((long long)row + p.diag, (long long)p.Skv - 1) : (long long)p.Skv - 1;
        const int lim = static_cast<int>(lim_ll < -1 ? -1 : lim_ll);  // last visible key
        float m_run = -INFINITY, l_run = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const uint32_t tS = tmem_base + lane_off + 128 * (j & 1);
            const bool got = wait_bounded(bar(BAR_SFULL + (j & 1)), (j >> 1) & 1, abort_flag, limit);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t s[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
            const int nvis = lim - j * kBN + 1;
            if (nvis < kBN) {
#pragma unroll
                for (int jj = 0; jj < kBN; ++jj)
                    if (jj >= nvis) s[jj] = __float_as_uint(-INFINITY);
            }
            float mx[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                mx[q] = fmax3(__uint_as_float(s[q]), __uint_as_float(s[8 + q]), __uint_as_float(s[16 + q]));
#pragma unroll
            for (int base = 24; base < kBN; base += 16)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    mx[q] = fmax3(mx[q], __uint_as_float(s[base + q]), __uint_as_float(s[base + 8 + q]));
            const float m_tile = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) * sl2;
            float alpha = 1.f;
            if (m_tile - m_run > kRescaleLog2) {
                alpha = ex2_approx(m_run - m_tile);
                m_run = m_tile;
            }
            const float m_use = m_run == -INFINITY ? 0.f : m_run;
            // O holds PV_0 .. PV_{j-1}; rescale it (rare: only when the running max
            // rose) after PV_{j-1} has completed and before PV_j is issued.  S_j
            // completing implies PV_{j-2} completed, so PVDONE is at most one phase
            // behind and its parity identifies PV_{j-1}.
            const bool need = (j > 0) && (alpha != 1.f);
            if (__any_sync(0xffffffffu, need)) {
                const bool pv = wait_bounded(bar(BAR_PVDONE), (j - 1) & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, pv)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < kD / 16; ++c) {
                    uint32_t o[16];
                    tmem_ld16(tO + 16 * c, o);
                    tmem_wait_ld_regs16(o);
#pragma unroll
                    for (int q = 0; q < 16; q += 2) {
                        float x0, x1;
                        fmul2_b(x0, x1, __uint_as_float(o[q]), __uint_as_float(o[q + 1]), alpha);
                        o[q] = __float_as_uint(x0);
                        o[q + 1] = __float_as_uint(x1);
                    }
                    tmem_st16(tO + 16 * c, o);
                }
            }
            float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int q = 0; q < 16; q += 2) {
                    const int e = 32 * c + 2 * q;
                    float a0, a1, b0, b1;
                    ffma2_bc(a0, a1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]), sl2, -m_use);
                    ffma2_bc(b0, b1, __uint_as_float(s[e + 2]), __uint_as_float(s[e + 3]), sl2, -m_use);
                    a0 = ex2_approx(a0);
                    a1 = ex2_approx(a1);
                    b0 = ex2_approx(b0);
                    b1 = ex2_approx(b1);
                    if (q & 2) {
                        fadd2_acc(rs2, rs3, a0, a1);
                        fadd2_acc(rs2, rs3, b0, b1);
                    } else {
                        fadd2_acc(rs0, rs1, a0, a1);
                        fadd2_acc(rs0, rs1, b0, b1);
                    }
                    pk[q] = pack_x2<kF16>(a0, a1);
                    pk[q + 1] = pack_x2<kF16>(b0, b1);
                }
                tmem_st16(tS + 16 * c, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(BAR_PFULL + (j & 1)));
            l_run = l_run * alpha + ((rs0 + rs1) + (rs2 + rs3));
        }
        // epilogue: O (after the last PV) times 1/l, four 64-column chunks through
        // the swizzled staging buffer and a TMA store each; LSE
        if (ok) {
            bool have = n > 0;
            if (have) {
                // a dedicated once-per-CTA barrier: PVDONE may still be two phases behind here
                const bool got = wait_bounded(bar(BAR_ODONE), 0, abort_flag, limit);
                have = __all_sync(0xffffffffu, got);
                ok = have;
                tc_fence_after();
            }
            const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
            uint8_t* stage = smem + Geo::kSmemStage;
            for (int c = 0; ok && c < 4; ++c) {
                uint32_t o[64];
                if (have) {
                    tmem_ld32(tO + 64 * c, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                    tmem_ld32(tO + 64 * c + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                    tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                    tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) o[e] = 0u;
                }
                if (r == 0) bulk_wait_group_read0();  // the previous store has read the staging
                named_bar_sync(1, 128);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float fo[8];
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        fmul2_b(fo[e], fo[e + 1], __uint_as_float(o[8 * q + e]), __uint_as_float(o[8 * q + e + 1]),
                                inv_l);
                    *reinterpret_cast<uint4*>(stage + r * 128 + ((q ^ (r & 7)) * 16)) =
                        make_uint4(pack_x2<kF16>(fo[0], fo[1]), pack_x2<kF16>(fo[2], fo[3]),
                                   pack_x2<kF16>(fo[4], fo[5]), pack_x2<kF16>(fo[6], fo[7]));
                }
                fence_proxy_async_smem();
                named_bar_sync(1, 128);
                if (r == 0 && it.row0 < p.Sq) {
                    tma_store_4d(&tm_o, smem_u32(stage), c * 64, it.hq, it.row0, it.b);
                    bulk_commit_group();
                }
            }
            if (ok && row < p.Sq && p.lse != nullptr) {
                const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
                p.lse[(static_cast<size_t>(it.b) * p.Hq + it.hq) * p.Sq + row] = lse;
            }
            if (r == 0) bulk_wait_group0();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace d256
}  // namespace attn
