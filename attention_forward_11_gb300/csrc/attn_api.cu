// attn_api.cu -- host side of libattn: argument validation, TMA descriptor
// encoding, work decomposition and the launch of the sm_103a kernels.  The
// checks mirror the Pallas page's `_attention_forward` (shapes, GQA
// divisibility, dtype, head size) but accept any sequence length: ragged
// tails are handled inside the kernel by TMA zero-fill and key masking.
#include <attn.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <memory>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fmha_bwd_sm103.cuh"
#include "fmha_fwd_d256_sm103.cuh"
#include "fmha_bwd_d256_sm103.cuh"
#include "fmha_fwd_sm103.cuh"
#include "unit_rates_sm103.cuh"

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::atomic<unsigned long long> g_launches{0};
constexpr unsigned int kDefaultPollLimit = 1u << 26;
constexpr int kMaxDevices = 64;

EncodeTiledFn encoder() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 4-d view [B, S, H, D] of a bf16 tensor (D innermost), 128-row x 64-column
// boxes with 128-byte swizzle: the layout the tcgen05 K-major / MN-major
// shared-memory descriptors expect.
bool encode_bshd(CUtensorMap* map, const void* ptr, int B, int S, int H, int D, bool f16 = false) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                   (cuuint64_t)S * H * D * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)attn::kBM, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <class Sched, bool kF16, int kD>
bool opt_in_smem() {
    return cudaFuncSetAttribute(attn::fmha_fwd_kernel<Sched, kF16, kD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::Geo<kD>::kSmemBytes) == cudaSuccess;
}

template <bool kF16, int kD>
bool opt_in_smem_bwd() {
    constexpr int bytes = attn::bwd::BwdGeo<kD>::kSmemBytes;
    return cudaFuncSetAttribute(attn::bwd::fmha_bwd_dkdv_kernel<kF16, kD>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
           cudaFuncSetAttribute(attn::bwd::fmha_bwd_dq_kernel<kF16, kD>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::bwd::DqGeo<kD>::kSmemBytes) == cudaSuccess;
}

template <int kRole, bool kF16>
bool opt_in_smem_bwd256() {
    return cudaFuncSetAttribute(attn::bwd256::fmha_bwd_d256_kernel<kRole, kF16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                attn::bwd256::Geo<kRole>::kSmemBytes) == cudaSuccess;
}

template <bool kF16>
bool opt_in_smem_bwd256_all() {
    using namespace attn::bwd256;
    return opt_in_smem_bwd256<kRoleDV, kF16>() && opt_in_smem_bwd256<kRoleDK, kF16>() &&
           opt_in_smem_bwd256<kRoleDQ, kF16>();
}

// Per-device one-time set-up: the kernels' shared-memory opt-in and the SM count.
bool device_setup(int dev, int* sm_count) {
    static std::mutex mu;
    static int sms[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0) {
        int n = 0;
        if (!opt_in_smem<attn::PlainSched, false, 128>() || !opt_in_smem<attn::PlainSched, true, 128>() ||
            !opt_in_smem<attn::SplitSched, false, 128>() || !opt_in_smem<attn::PlainSched, false, 64>() ||
            !opt_in_smem<attn::PlainSched, true, 64>() || !opt_in_smem<attn::SplitSched, false, 64>() ||
            !opt_in_smem<attn::TableSched, false, 128>() || !opt_in_smem<attn::TableSched, true, 128>() ||
            !opt_in_smem_bwd<false, 128>() || !opt_in_smem_bwd<true, 128>() || !opt_in_smem_bwd<false, 64>() ||
            !opt_in_smem_bwd<true, 64>() || !opt_in_smem_bwd256_all<false>() || !opt_in_smem_bwd256_all<true>() ||
            cudaFuncSetAttribute(attn::d256::fmha_fwd_d256_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 attn::d256::Geo::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(attn::d256::fmha_fwd_d256_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 attn::d256::Geo::kSmemBytes) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            return false;
        sms[dev] = n;
    }
    *sm_count = sms[dev];
    return true;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

// Size checks shared by every entry point (mirrors the Pallas page's
// `_attention_forward`): sizes, GQA divisibility, mask mode, scale, head size.
attn_status_t check_sizes(int B, int Sq, int Skv, int Hq, int Hkv, int D, int causal) {
    if (B < 1 || Sq < 1 || Skv < 1 || Hq < 1 || Hkv < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (causal < 0 || causal > 2) return ATTN_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// Pointer checks: non-null, 16-byte aligned (TMA), outputs not aliasing inputs.
attn_status_t check_pointers(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             int B, int Sq, int Skv, int Hq, int Hkv, int D) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    for (const void* ptr : {q, k, v, o})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return ATTN_ERR_INVALID_ARG;
    if (lse && reinterpret_cast<uintptr_t>(lse) % 4 != 0) return ATTN_ERR_INVALID_ARG;
    const size_t q_bytes = (size_t)B * Sq * Hq * D * 2;
    const size_t kv_bytes = (size_t)B * Skv * Hkv * D * 2;
    if (ranges_overlap(o, q_bytes, q, q_bytes) || ranges_overlap(o, q_bytes, k, kv_bytes) ||
        ranges_overlap(o, q_bytes, v, kv_bytes))
        return ATTN_ERR_INVALID_ARG;
    const size_t lse_bytes = (size_t)B * Hq * Sq * 4;
    if (lse && (ranges_overlap(lse, lse_bytes, o, q_bytes) || ranges_overlap(lse, lse_bytes, q, q_bytes) ||
                ranges_overlap(lse, lse_bytes, k, kv_bytes) || ranges_overlap(lse, lse_bytes, v, kv_bytes)))
        return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// Work decomposition: two 128-row query tiles per unit sharing one K/V head.
attn_status_t make_params(int B, int Sq, int Skv, int Hq, int Hkv, int causal, float scale, void* o,
                          float* lse, attn::FwdParams* out, int D = 128) {
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    attn::FwdParams p{};
    p.B = B;
    p.Sq = Sq;
    p.Skv = Skv;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.D = D;
    p.causal = causal;
    p.diag = causal == 1 ? Skv - Sq : 0;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.lse = lse;
    p.poll_limit = kDefaultPollLimit;
    const int group = Hq / Hkv;
    p.head_pairs = (group % 2 == 0) ? 1 : 0;
    if (p.head_pairs) {
        p.n_head_units = Hq / 2;
        p.n_row_units = (Sq + attn::kBM - 1) / attn::kBM;
    } else {
        p.n_head_units = Hq;
        p.n_row_units = (Sq + attn::kTiles * attn::kBM - 1) / (attn::kTiles * attn::kBM);
    }
    const long long n_units = (long long)p.n_row_units * B * p.n_head_units;
    if (n_units > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
    p.n_units = static_cast<int>(n_units);
    p.o = static_cast<uint16_t*>(o);
    *out = p;
    return ATTN_OK;
}

bool encode_maps(const void* q, const void* k, const void* v, const void* o, int B, int Sq, int Skv, int Hq,
                 int Hkv, int D, CUtensorMap* tm, bool f16 = false) {
    return encode_bshd(&tm[0], q, B, Sq, Hq, D, f16) && encode_bshd(&tm[1], k, B, Skv, Hkv, D, f16) &&
           encode_bshd(&tm[2], v, B, Skv, Hkv, D, f16) && encode_bshd(&tm[3], o, B, Sq, Hq, D, f16);
}

// ---- split-KV plan: equal contiguous shares of the (unit, KV tile) iterations
struct SplitPlan {
    bool split = false;      // false: the whole-unit schedule is used (no workspace)
    int grid = 0;
    int n_slots = 0;
    attn::SplitSched sched{};
    attn::CombineTable comb{};
};
constexpr size_t kWorkspaceAlign = 256;
// Split only when the whole-unit makespan is at least ATTN_SPLIT_MARGIN_PCT percent
// of the split share plus ATTN_SPLIT_MIN_STEPS KV iterations.  Measured on GB300
// over few-tile shapes (Sq 1-2048, Skv 8K-128K, GQA 8/1, 32/8, 64/8, MHA 16): every
// shape with a ratio of 2.4 or more gained 1.5-19x from the split; between 1.15
// and 1.33 the outcome ranged from 0.89x to 1.34x (the benchmark's chunked
// prefill, 1.19: 0.96x), so those keep the whole-unit schedule.  (Building with
// both set to 0 splits wherever the plan can: how the crossover was measured.)
#ifndef ATTN_SPLIT_MARGIN_PCT
#define ATTN_SPLIT_MARGIN_PCT 135
#endif
#ifndef ATTN_SPLIT_MIN_STEPS
#define ATTN_SPLIT_MIN_STEPS 4
#endif
constexpr long long kSplitMarginPct = ATTN_SPLIT_MARGIN_PCT, kSplitMinSteps = ATTN_SPLIT_MIN_STEPS;

size_t workspace_bytes_for(int n_slots, int D) {
    const size_t o_bytes = (size_t)n_slots * attn::kTiles * attn::kBM * D * sizeof(float);
    const size_t ml_bytes = (size_t)n_slots * attn::kTiles * attn::kBM * sizeof(float2);
    const size_t o_pad = (o_bytes + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign;
    return o_pad + ml_bytes;
}

// The split plan: the (unit, KV tile) iterations, units in the plain schedule's
// order, cut into G = min(#SMs, total) equal contiguous shares, one per CTA; a
// unit that straddles shares becomes one piece per share, each with a workspace
// slot, merged afterwards by the combine kernel.  Fixed-size storage only (no
// heap), so every split-KV entry point, the no-allocation one included, runs
// this one planner.
void build_split_plan(const attn::FwdParams& p, int sms, SplitPlan* plan) {
    plan->split = false;
    if (p.D == 256) return;  // head size 256 runs its own one-tile-per-CTA kernel, unsplit
    if (p.n_units < 1 || p.n_units > attn::kMaxPieces) return;
    int W[attn::kMaxPieces];
    long long bnd[attn::kMaxSplitCtas + 1];
    unsigned short piece_cta[attn::kMaxPieces];
    long long T = 0;
    for (int u = 0; u < p.n_units; ++u) {
        W[u] = attn::decode_unit(p, u).nmax();
        if (W[u] > 0xFFFF) return;
        T += W[u];
    }
    const int G = static_cast<int>(std::min<long long>(std::min(sms, attn::kMaxSplitCtas), T));
    if (G < 1) return;
    // Does a split pay?  The whole-unit schedule takes as long as its busiest CTA
    // (units in the snake order over min(#units, #SMs) CTAs); the split one about
    // ceil(T / G) iterations, but its shares start at different KV positions, so the
    // L2 sharing of each K/V tile between the units of a head that run side by side
    // is lost, and a merge kernel follows.  Split only when the whole-unit makespan
    // exceeds the share by the measured margin.
    {
        const int Gp = std::min(p.n_units, std::min(sms, attn::kMaxPieces));
        long long load[attn::kMaxPieces] = {};
        long long makespan = 0;
        for (int u = 0; u < p.n_units; ++u) {
            const int r = u / Gp, c = u % Gp;
            const int cta = (r & 1) ? Gp - 1 - c : c;
            load[cta] += W[u];
            makespan = std::max(makespan, load[cta]);
        }
        const long long share = (T + G - 1) / G;
        if (makespan * 100 < share * kSplitMarginPct + kSplitMinSteps * 100) return;
    }
    for (int c = 0; c <= G; ++c) bnd[c] = (long long)c * T / G;
    attn::SplitSched& sc = plan->sched;
    attn::CombineTable& cb = plan->comb;
    int n_pieces = 0, n_slots = 0, n_comb = 0, c = 0;
    long long off = 0;
    auto add = [&](int u, int kb, int ke, int slot, int cta) -> bool {
        if (n_pieces >= attn::kMaxPieces) return false;
        sc.piece[n_pieces] = attn::Piece{u, static_cast<unsigned int>(kb) | (static_cast<unsigned int>(ke) << 16),
                                         slot};
        piece_cta[n_pieces++] = static_cast<unsigned short>(cta);
        return true;
    };
    for (int u = 0; u < p.n_units; ++u) {
        const long long a = off, e = off + W[u];
        while (c < G - 1 && a >= bnd[c + 1]) ++c;
        if (W[u] == 0) {
            if (!add(u, 0, 0, -1, c)) return;  // no KV tile at all: still writes O = 0, LSE = -inf
            continue;
        }
        int c1 = c;
        while (c1 < G - 1 && e > bnd[c1 + 1]) ++c1;
        if (c1 == c) {
            if (!add(u, 0, W[u], -1, c)) return;
        } else {
            if (n_comb >= attn::kMaxCombine) return;
            cb.e[n_comb++] = attn::CombineEntry{u, n_slots, c1 - c + 1};
            for (int cc = c; cc <= c1; ++cc) {
                const long long kb = std::max(a, bnd[cc]) - a, ke = std::min(e, bnd[cc + 1]) - a;
                if (!add(u, static_cast<int>(kb), static_cast<int>(ke), n_slots++, cc)) return;
            }
        }
        off = e;
    }
    if (n_comb == 0) return;  // no unit straddles two shares: the whole-unit schedule is as good
    // first piece of each CTA (pieces are in non-decreasing CTA order)
    int i = 0;
    for (int cc = 0; cc <= G; ++cc) {
        while (i < n_pieces && piece_cta[i] < cc) ++i;
        sc.cta_begin[cc] = static_cast<unsigned short>(i);
    }
    sc.n_pieces = n_pieces;
    cb.n = n_comb;
    plan->grid = G;
    plan->n_slots = n_slots;
    plan->split = true;
}

// The whole-unit schedule's table for causal shapes (TableSched): units in blocks
// of K/V heads whose K and V together take at most kTableBlockBytes, longest first
// within a block; each unit in turn goes to the least-loaded CTA (its KV tiles
// plus one for the unit's own start-up), which keeps the CTAs' totals within a
// unit of each other while a block's heads run side by side and their K and V
// stay in L2.  Returns false where the snake order is used instead: unmasked
// shapes (already numbered head-major) and shapes beyond the table's size.
constexpr long long kTableBlockBytes = 48ll << 20;
bool build_plain_table(const attn::FwdParams& p, int grid, attn::TableSched* sc) {
    if (!p.causal || p.n_units > attn::kMaxTable || grid < 1 || grid > attn::kMaxSplitCtas) return false;
    const int inner_count = p.B * p.n_head_units;              // (batch, head unit) pairs
    const int units_per_kv = p.n_head_units / p.Hkv > 0 ? p.n_head_units / p.Hkv : 1;
    const long long kv_bytes = 4ll * p.Skv * p.D;               // K and V of one K/V head
    const long long kv_per_block = std::max<long long>(1, kTableBlockBytes / std::max<long long>(1, kv_bytes));
    const int block = static_cast<int>(std::min<long long>(inner_count, kv_per_block * units_per_kv));
    long long load[attn::kMaxSplitCtas] = {};
    unsigned short count[attn::kMaxSplitCtas] = {};
    unsigned short owner[attn::kMaxTable];
    unsigned short order[attn::kMaxTable];
    int n = 0;
    for (int s = 0; s < inner_count; s += block)
        for (int ru = 0; ru < p.n_row_units; ++ru)
            for (int inner = s; inner < std::min(inner_count, s + block); ++inner) {
                const int u = ru * inner_count + inner;
                int c = 0;
                for (int k = 1; k < grid; ++k)
                    if (load[k] < load[c]) c = k;
                load[c] += attn::decode_unit(p, u).nmax() + 1;
                owner[n] = static_cast<unsigned short>(c);
                order[n] = static_cast<unsigned short>(u);
                ++count[c];
                ++n;
            }
    if (n != p.n_units) return false;
    int pos = 0;
    for (int c = 0; c < grid; ++c) {
        sc->cta_begin[c] = static_cast<unsigned short>(pos);
        pos += count[c];
    }
    sc->cta_begin[grid] = static_cast<unsigned short>(pos);
    unsigned short fill[attn::kMaxSplitCtas] = {};
    for (int i = 0; i < n; ++i) {  // each CTA's units in the order they were handed out
        const int c = owner[i];
        sc->unit[sc->cta_begin[c] + fill[c]++] = order[i];
    }
    return true;
}

// build_plain_table for the last few shapes, so a repeated call costs a copy
// (the greedy assignment takes ~units x CTAs steps on the host)
bool plain_table_cached(const attn::FwdParams& p, int grid, attn::TableSched* out) {
    struct Entry {
        int key[9];
        bool ok;
        attn::TableSched sched;
    };
    constexpr int kEntries = 8;
    static Entry cache[kEntries];
    static int used = 0, next = 0;
    static std::mutex mu;
    const int key[9] = {p.B, p.Sq, p.Skv, p.Hq, p.Hkv, p.D, p.causal, grid, p.n_units};
    std::lock_guard<std::mutex> lock(mu);
    for (int e = 0; e < used; ++e)
        if (std::memcmp(cache[e].key, key, sizeof(key)) == 0) {
            if (cache[e].ok) std::memcpy(out, &cache[e].sched, sizeof(*out));
            return cache[e].ok;
        }
    const bool ok = build_plain_table(p, grid, out);
    Entry& slot = cache[next];
    std::memcpy(slot.key, key, sizeof(key));
    slot.ok = ok;
    if (ok) std::memcpy(&slot.sched, out, sizeof(*out));
    next = (next + 1) % kEntries;
    if (used < kEntries) ++used;
    return ok;
}

template <bool kF16 = false>
attn_status_t launch_plain(const CUtensorMap* tm, const attn::FwdParams& p, int sms, cudaStream_t stream) {
    if (p.D == 256) {
        // one 128-row query tile per CTA (its O fills half of tensor memory)
        const long long tiles = (long long)p.B * p.Hq * ((p.Sq + attn::kBM - 1) / attn::kBM);
        if (tiles > 0x7fffffffLL) return ATTN_ERR_INVALID_ARG;
        attn::d256::fmha_fwd_d256_kernel<kF16><<<static_cast<unsigned int>(tiles), attn::d256::kThreads,
                                                 attn::d256::Geo::kSmemBytes, stream>>>(tm[0], tm[1], tm[2], tm[3], p);
        if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return ATTN_OK;
    }
    // persistent grid: at most one CTA per SM (the CTA holds all 512 TMEM columns)
    const int grid = p.n_units < sms ? p.n_units : sms;
    static thread_local attn::TableSched table;  // 4.6 KB: kept off the stack
    if (p.D == 64)
        attn::fmha_fwd_kernel<attn::PlainSched, kF16, 64><<<static_cast<unsigned int>(grid), attn::kThreads,
                                                            attn::Geo<64>::kSmemBytes, stream>>>(
            tm[0], tm[1], tm[2], tm[3], p, attn::PlainSched{0});
    else if (plain_table_cached(p, grid, &table))  // head size 128, causal: the head-blocked table
        attn::fmha_fwd_kernel<attn::TableSched, kF16, 128><<<static_cast<unsigned int>(grid), attn::kThreads,
                                                             attn::Geo<128>::kSmemBytes, stream>>>(
            tm[0], tm[1], tm[2], tm[3], p, table);
    else
        attn::fmha_fwd_kernel<attn::PlainSched, kF16, 128><<<static_cast<unsigned int>(grid), attn::kThreads,
                                                             attn::Geo<128>::kSmemBytes, stream>>>(
            tm[0], tm[1], tm[2], tm[3], p, attn::PlainSched{0});
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ATTN_OK;
}

attn_status_t launch_split(const CUtensorMap* tm, const attn::FwdParams& p, SplitPlan& plan, void* workspace,
                           cudaStream_t stream) {
    const size_t o_bytes = (size_t)plan.n_slots * attn::kTiles * attn::kBM * p.D * sizeof(float);
    const size_t o_pad = (o_bytes + kWorkspaceAlign - 1) / kWorkspaceAlign * kWorkspaceAlign;
    plan.sched.ws_o = static_cast<float*>(workspace);
    plan.sched.ws_ml = reinterpret_cast<float2*>(static_cast<char*>(workspace) + o_pad);
    if (p.D == 64)
        attn::fmha_fwd_kernel<attn::SplitSched, false, 64><<<static_cast<unsigned int>(plan.grid), attn::kThreads,
                                                             attn::Geo<64>::kSmemBytes, stream>>>(
            tm[0], tm[1], tm[2], tm[3], p, plan.sched);
    else
        attn::fmha_fwd_kernel<attn::SplitSched, false, 128><<<static_cast<unsigned int>(plan.grid), attn::kThreads,
                                                              attn::Geo<128>::kSmemBytes, stream>>>(
            tm[0], tm[1], tm[2], tm[3], p, plan.sched);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    plan.comb.ws_o = plan.sched.ws_o;
    plan.comb.ws_ml = plan.sched.ws_ml;
    plan.comb.o = p.o;
    const long long warps = (long long)plan.comb.n * attn::kTiles * attn::kBM;
    const unsigned int blocks = static_cast<unsigned int>((warps + attn::kCombineWarps - 1) / attn::kCombineWarps);
    if (p.D == 64)
        attn::splitkv_combine_kernel<false, 64><<<blocks, 32 * attn::kCombineWarps, 0, stream>>>(p, plan.comb);
    else
        attn::splitkv_combine_kernel<false, 128><<<blocks, 32 * attn::kCombineWarps, 0, stream>>>(p, plan.comb);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ATTN_OK;
}

}  // namespace

namespace {

attn_status_t fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Sq, int Skv,
                       int Hq, int Hkv, int D, int causal, float scale, bool f16, cudaStream_t stream) {
    // ---- validation: nothing is launched on any error
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_sizes(B, Sq, Skv, Hq, Hkv, D, causal);
    if (st == ATTN_ERR_INVALID_ARG) return st;
    const attn_status_t sp = check_pointers(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D > 0 ? D : 1);
    if (sp != ATTN_OK) return sp;
    attn::FwdParams p{};
    const attn_status_t sm = make_params(B, Sq, Skv, Hq, Hkv, causal, scale, o, lse, &p, D);
    if (sm != ATTN_OK) return sm;
    if (st != ATTN_OK) return st;  // valid request, unsupported head size
    CUtensorMap tm[4];
    if (!encode_maps(q, k, v, o, B, Sq, Skv, Hq, Hkv, D, tm, f16)) return ATTN_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_setup(dev, &sms)) return ATTN_ERR_CUDA;
    return f16 ? launch_plain<true>(tm, p, sms, stream) : launch_plain<false>(tm, p, sms, stream);
}

}  // namespace

extern "C" attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int Sq, int Skv, int Hq, int Hkv, int D, int causal,
                                  float scale, cudaStream_t stream) {
    return fwd_impl(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D, causal, scale, false, stream);
}

extern "C" attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                     int Sq, int Skv, int Hq, int Hkv, int D, int causal, float scale, int dtype,
                                     cudaStream_t stream) {
    if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_F16) return ATTN_ERR_INVALID_ARG;
    return fwd_impl(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D, causal, scale, dtype == ATTN_DTYPE_F16, stream);
}

extern "C" attn_status_t attn_fwd_splitkv_workspace_size(int B, int Sq, int Skv, int Hq, int Hkv, int D,
                                                         int causal, size_t* bytes) {
    if (!bytes) return ATTN_ERR_INVALID_ARG;
    *bytes = 0;
    const attn_status_t st = check_sizes(B, Sq, Skv, Hq, Hkv, D, causal);
    if (st != ATTN_OK) return st;
    attn::FwdParams p{};
    const attn_status_t sm = make_params(B, Sq, Skv, Hq, Hkv, causal, 1.0f, nullptr, nullptr, &p, D);
    if (sm != ATTN_OK) return sm;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_setup(dev, &sms)) return ATTN_ERR_CUDA;
    std::unique_ptr<SplitPlan> plan(new SplitPlan());
    build_split_plan(p, sms, plan.get());
    *bytes = plan->split ? workspace_bytes_for(plan->n_slots, D) : 0;
    return ATTN_OK;
}

extern "C" attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                                          int Sq, int Skv, int Hq, int Hkv, int D, int causal, float scale,
                                          void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_sizes(B, Sq, Skv, Hq, Hkv, D, causal);
    if (st == ATTN_ERR_INVALID_ARG) return st;
    const attn_status_t sp = check_pointers(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D > 0 ? D : 1);
    if (sp != ATTN_OK) return sp;
    if (workspace && reinterpret_cast<uintptr_t>(workspace) % kWorkspaceAlign != 0) return ATTN_ERR_INVALID_ARG;
    attn::FwdParams p{};
    const attn_status_t sm = make_params(B, Sq, Skv, Hq, Hkv, causal, scale, o, lse, &p, D);
    if (sm != ATTN_OK) return sm;
    if (st != ATTN_OK) return st;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_setup(dev, &sms)) return ATTN_ERR_CUDA;
    std::unique_ptr<SplitPlan> plan(new SplitPlan());
    build_split_plan(p, sms, plan.get());
    if (plan->split) {
        const size_t need = workspace_bytes_for(plan->n_slots, D);
        if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
        const size_t q_bytes = (size_t)B * Sq * Hq * D * 2, kv_bytes = (size_t)B * Skv * Hkv * D * 2;
        if (ranges_overlap(workspace, need, q, q_bytes) || ranges_overlap(workspace, need, k, kv_bytes) ||
            ranges_overlap(workspace, need, v, kv_bytes) || ranges_overlap(workspace, need, o, q_bytes) ||
            (lse && ranges_overlap(workspace, need, lse, (size_t)B * Hq * Sq * 4)))
            return ATTN_ERR_INVALID_ARG;
    }
    CUtensorMap tm[4];
    if (!encode_maps(q, k, v, o, B, Sq, Skv, Hq, Hkv, D, tm)) return ATTN_ERR_CUDA;
    return plan->split ? launch_split(tm, p, *plan, workspace, stream) : launch_plain(tm, p, sms, stream);
}

// ---- split-KV without any allocation: scratch in a static device array
//
// For callers that cannot allocate device memory at the point they run
// attention -- for example code whose device memory all belongs to another
// allocator (a framework's caching pool, a fixed arena set up at start-up) or
// runtimes that forbid allocation once serving has begun.  The split-KV scratch
// then lives in this file-scope array instead of a caller workspace.  Every GPU
// that loads the library holds the array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(40) << 20;  // 40 MiB
static __device__ __align__(256) unsigned char g_splitkv_scratch[kStaticScratchBytes];

namespace {

// Device address of the static scratch on `dev` (the current device), looked up
// once per device: in host code the array's name is only a stand-in.
void* static_scratch_address(int dev) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_splitkv_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
        addr[dev] = ptr;
    }
    return addr[dev];
}

}  // namespace

extern "C" attn_status_t attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                                  float* lse, int B, int Sq, int Skv, int Hq, int Hkv, int D,
                                                  int causal, float scale, cudaStream_t stream) {
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_sizes(B, Sq, Skv, Hq, Hkv, D, causal);
    if (st == ATTN_ERR_INVALID_ARG) return st;
    const attn_status_t sp = check_pointers(q, k, v, o, lse, B, Sq, Skv, Hq, Hkv, D > 0 ? D : 1);
    if (sp != ATTN_OK) return sp;
    attn::FwdParams p{};
    const attn_status_t sm = make_params(B, Sq, Skv, Hq, Hkv, causal, scale, o, lse, &p, D);
    if (sm != ATTN_OK) return sm;
    if (st != ATTN_OK) return st;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_setup(dev, &sms)) return ATTN_ERR_CUDA;
    void* scratch = static_scratch_address(dev);  // first call on a device: one-time look-up
    if (scratch == nullptr) return ATTN_ERR_CUDA;
    // the plan lives in static storage: one call at a time builds and launches it
    static std::mutex plan_mu;
    static SplitPlan plan;
    std::lock_guard<std::mutex> lock(plan_mu);
    build_split_plan(p, sms, &plan);
    if (plan.split && workspace_bytes_for(plan.n_slots, D) > kStaticScratchBytes) return ATTN_ERR_UNSUPPORTED;
    CUtensorMap tm[4];
    if (!encode_maps(q, k, v, o, B, Sq, Skv, Hq, Hkv, D, tm)) return ATTN_ERR_CUDA;
    return plan.split ? launch_split(tm, p, plan, scratch, stream) : launch_plain(tm, p, sms, stream);
}

// ---- backward
namespace {

constexpr size_t kBwdAlign = 256;

size_t bwd_vec_bytes(int B, int Sq, int Hq) {
    const size_t sq_pad = (static_cast<size_t>(Sq) + attn::kBM - 1) / attn::kBM * attn::kBM;
    const size_t v = static_cast<size_t>(B) * Hq * sq_pad * sizeof(float);
    return (v + kBwdAlign - 1) / kBwdAlign * kBwdAlign;
}

template <bool kF16, int kD>
attn_status_t launch_bwd(const CUtensorMap* tm, const void* o, const void* dO, const float* lse,
                         const attn::bwd::BwdParams& p, int sms, cudaStream_t stream) {
    using namespace attn::bwd;
    const long long rows = (long long)p.Hq * p.sq_pad;  // per batch entry
    const long long per_block = 8LL * prep_rows_per_warp<kD>();
    const dim3 prep_grid(static_cast<unsigned int>((rows + per_block - 1) / per_block), static_cast<unsigned int>(p.B));
    bwd_prep_kernel<kF16, kD><<<prep_grid, 256, 0, stream>>>(
        static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dO), lse, p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    // persistent: at most one CTA per SM, items taken from the queue the prep kernel reset
    const int n_items = p.B * p.Hkv * p.n_kv_tiles;
    const unsigned int g_kv = static_cast<unsigned int>(n_items < sms ? n_items : sms);
    fmha_bwd_dkdv_kernel<kF16, kD><<<g_kv, kThreads, BwdGeo<kD>::kSmemBytes, stream>>>(tm[0], tm[1], tm[2], tm[3], p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const int n_q_items = p.B * p.Hq * p.n_q_tiles;
    const unsigned int g_q = static_cast<unsigned int>(n_q_items < sms ? n_q_items : sms);
    fmha_bwd_dq_kernel<kF16, kD><<<g_q, kThreads, DqGeo<kD>::kSmemBytes, stream>>>(tm[0], tm[1], tm[2], tm[3], p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ATTN_OK;
}

// Head size 256: the prep kernel, then the dV, dK and dQ launches of the one
// D = 256 kernel (each persistent, on its own work counter).
template <bool kF16>
attn_status_t launch_bwd256(const CUtensorMap* tm, const void* o, const void* dO, const float* lse,
                            const attn::bwd::BwdParams& p, int sms, cudaStream_t stream) {
    using namespace attn::bwd256;
    constexpr int kD = 256;
    const long long rows = (long long)p.Hq * p.sq_pad;  // per batch entry
    const long long per_block = 8LL * attn::bwd::prep_rows_per_warp<kD>();
    const dim3 prep_grid(static_cast<unsigned int>((rows + per_block - 1) / per_block), static_cast<unsigned int>(p.B));
    attn::bwd::bwd_prep_kernel<kF16, kD><<<prep_grid, 256, 0, stream>>>(
        static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dO), lse, p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    auto grid_of = [&](int n) { return static_cast<unsigned int>(n < sms ? n : sms); };
    fmha_bwd_d256_kernel<kRoleDV, kF16><<<grid_of(n_items_of<kRoleDV>(p)), kThreads, Geo<kRoleDV>::kSmemBytes,
                                          stream>>>(tm[0], tm[1], tm[2], tm[3], p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    fmha_bwd_d256_kernel<kRoleDK, kF16><<<grid_of(n_items_of<kRoleDK>(p)), kThreads, Geo<kRoleDK>::kSmemBytes,
                                          stream>>>(tm[0], tm[1], tm[2], tm[3], p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    fmha_bwd_d256_kernel<kRoleDQ, kF16><<<grid_of(n_items_of<kRoleDQ>(p)), kThreads, Geo<kRoleDQ>::kSmemBytes,
                                          stream>>>(tm[0], tm[1], tm[2], tm[3], p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_bwd_workspace_size(int B, int Sq, int Skv, int Hq, int Hkv, int D, size_t* bytes) {
    if (!bytes) return ATTN_ERR_INVALID_ARG;
    *bytes = 0;
    const attn_status_t st = check_sizes(B, Sq, Skv, Hq, Hkv, D, 0);
    if (st != ATTN_OK) return st;
    *bytes = 2 * bwd_vec_bytes(B, Sq, Hq) + kBwdAlign;  // + the kernels' work counters
    return ATTN_OK;
}

extern "C" attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                  const void* dO, void* dq, void* dk, void* dv, int B, int Sq, int Skv, int Hq,
                                  int Hkv, int D, int causal, float scale, int dtype, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
    // ---- validation: nothing is launched on any error
    if (!q || !k || !v || !o || !lse || !dO || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_F16) return ATTN_ERR_INVALID_ARG;
    attn_status_t st = check_sizes(B, Sq, Skv, Hq, Hkv, D, causal);
    if (st == ATTN_ERR_INVALID_ARG) return st;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    for (const void* ptr : {q, k, v, o, dO, static_cast<const void*>(dq), static_cast<const void*>(dk),
                            static_cast<const void*>(dv)})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(lse) % 4 != 0 || reinterpret_cast<uintptr_t>(workspace) % kBwdAlign != 0)
        return ATTN_ERR_INVALID_ARG;
    const int Dn = D > 0 ? D : 1;
    const size_t q_bytes = (size_t)B * Sq * Hq * Dn * 2, kv_bytes = (size_t)B * Skv * Hkv * Dn * 2;
    const size_t lse_bytes = (size_t)B * Hq * Sq * 4;
    const size_t need = 2 * bwd_vec_bytes(B, Sq, Hq) + kBwdAlign;
    if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
    // the outputs and the workspace overlap no input and no other output
    const void* out_p[4] = {dq, dk, dv, workspace};
    const size_t out_n[4] = {q_bytes, kv_bytes, kv_bytes, need};
    const void* in_p[6] = {q, k, v, o, lse, dO};
    const size_t in_n[6] = {q_bytes, kv_bytes, kv_bytes, q_bytes, lse_bytes, q_bytes};
    for (int a = 0; a < 4; ++a) {
        for (int c = 0; c < 6; ++c)
            if (ranges_overlap(out_p[a], out_n[a], in_p[c], in_n[c])) return ATTN_ERR_INVALID_ARG;
        for (int c = a + 1; c < 4; ++c)
            if (ranges_overlap(out_p[a], out_n[a], out_p[c], out_n[c])) return ATTN_ERR_INVALID_ARG;
    }
    if (st != ATTN_OK) return st;  // valid request, unsupported head size
    attn::bwd::BwdParams p{};
    p.B = B;
    p.Sq = Sq;
    p.Skv = Skv;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.D = D;
    p.causal = causal;
    p.diag = causal == 1 ? Skv - Sq : 0;
    p.n_q_tiles = (Sq + attn::kBM - 1) / attn::kBM;
    p.n_kv_tiles = (Skv + attn::kBN - 1) / attn::kBN;
    p.sq_pad = p.n_q_tiles * attn::kBM;
    if ((long long)B * Hkv * p.n_kv_tiles > 0x7fffffffLL || (long long)B * Hq * p.n_q_tiles > 0x7fffffffLL ||
        (long long)Hq * p.sq_pad > 0x7fffffffLL - 1024 || B > 65535)
        return ATTN_ERR_INVALID_ARG;
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.lse2 = static_cast<float*>(workspace);
    p.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + bwd_vec_bytes(B, Sq, Hq));
    p.work = reinterpret_cast<int*>(static_cast<char*>(workspace) + 2 * bwd_vec_bytes(B, Sq, Hq));
    p.dq = static_cast<uint16_t*>(dq);
    p.dk = static_cast<uint16_t*>(dk);
    p.dv = static_cast<uint16_t*>(dv);
    p.poll_limit = kDefaultPollLimit;
    const bool f16 = dtype == ATTN_DTYPE_F16;
    CUtensorMap tm[4];
    if (!encode_bshd(&tm[0], q, B, Sq, Hq, D, f16) || !encode_bshd(&tm[1], dO, B, Sq, Hq, D, f16) ||
        !encode_bshd(&tm[2], k, B, Skv, Hkv, D, f16) || !encode_bshd(&tm[3], v, B, Skv, Hkv, D, f16))
        return ATTN_ERR_CUDA;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_setup(dev, &sms)) return ATTN_ERR_CUDA;
    if (D == 256)
        return f16 ? launch_bwd256<true>(tm, o, dO, lse, p, sms, stream)
                   : launch_bwd256<false>(tm, o, dO, lse, p, sms, stream);
    if (D == 64)
        return f16 ? launch_bwd<true, 64>(tm, o, dO, lse, p, sms, stream)
                   : launch_bwd<false, 64>(tm, o, dO, lse, p, sms, stream);
    return f16 ? launch_bwd<true, 128>(tm, o, dO, lse, p, sms, stream)
               : launch_bwd<false, 128>(tm, o, dO, lse, p, sms, stream);
}

extern "C" const char* attn_status_str(attn_status_t status) {
    switch (status) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
    }
    return "ATTN_UNKNOWN_STATUS";
}

namespace {

// Reads and clears the current device's status word (the caller has synchronised
// whatever work it wants covered).
attn_status_t read_and_clear_status() {
    unsigned int word = 0;
    if (cudaMemcpyFromSymbol(&word, attn::g_attn_status, sizeof word) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbol(attn::g_attn_status, &zero, sizeof zero) != cudaSuccess)
            return ATTN_ERR_CUDA;
    }
    return (word & attn::kStatusTimeout) ? ATTN_ERR_TIMEOUT : ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_check_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
    return read_and_clear_status();
}

extern "C" attn_status_t attn_last_device_status(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
    return read_and_clear_status();
}

extern "C" unsigned long long attn_kernel_launches(void) {
    return g_launches.load(std::memory_order_relaxed);
}

extern "C" attn_status_t attn_debug_wait_timeout(unsigned int poll_limit, cudaStream_t stream) {
    if (poll_limit < 1 || poll_limit > (1u << 20)) return ATTN_ERR_INVALID_ARG;
    attn::wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(poll_limit);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ATTN_OK;
}

// ---- measured unit rates (diagnostic)
namespace {
template <int kMode>
attn_status_t run_mma_rate(int sms, cudaStream_t stream, double* clocks_per_mma) {
    auto kern = attn::rates::mma_rate_kernel<kMode>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, attn::rates::kMmaSmem) !=
        cudaSuccess)
        return ATTN_ERR_CUDA;
    kern<<<sms, 128, attn::rates::kMmaSmem, stream>>>();
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    long long c[attn::rates::kMaxSms];
    if (cudaMemcpyFromSymbolAsync(c, attn::rates::g_rate_clocks, sizeof(long long) * sms, 0,
                                  cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    double mean = 0.0;
    for (int i = 0; i < sms; ++i) mean += static_cast<double>(c[i]);
    *clocks_per_mma = mean / sms / (8.0 * attn::rates::kMmaIters);
    return ATTN_OK;
}
}  // namespace

extern "C" attn_status_t attn_debug_unit_schedule(int B, int Sq, int Skv, int Hq, int Hkv, int D, int causal,
                                                   int sms, int* cta_begin, int* units, int cap, int* n_units_out) {
    const attn_status_t sz = check_sizes(B, Sq, Skv, Hq, Hkv, D, causal);
    if (sz != ATTN_OK) return sz;
    if (sms < 1 || sms > attn::kMaxSplitCtas || !cta_begin || !units || !n_units_out) return ATTN_ERR_INVALID_ARG;
    attn::FwdParams p;
    static int dummy_o;
    const attn_status_t pr = make_params(B, Sq, Skv, Hq, Hkv, causal, 1.0f, &dummy_o, nullptr, &p, D);
    if (pr != ATTN_OK) return pr;
    *n_units_out = 0;
    if (D != 128) return ATTN_OK;  // head size 64 keeps the snake order; 256 runs its own kernel
    const int grid = p.n_units < sms ? p.n_units : sms;
    attn::TableSched table;
    if (!build_plain_table(p, grid, &table)) return ATTN_OK;
    if (cap < p.n_units) return ATTN_ERR_INVALID_ARG;
    for (int c = 0; c <= grid; ++c) cta_begin[c] = table.cta_begin[c];
    for (int i = 0; i < p.n_units; ++i) units[i] = table.unit[i];
    *n_units_out = p.n_units;
    return ATTN_OK;
}

extern "C" attn_status_t attn_debug_unit_rates(double* out, int n, cudaStream_t stream) {
    if (out == nullptr || n < ATTN_UNIT_RATES) return ATTN_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
    if (sms < 1 || sms > attn::rates::kMaxSms) return ATTN_ERR_UNSUPPORTED;
    // an earlier kernel's timeout is kept and reported, not wiped by this diagnostic
    const attn_status_t earlier = attn_check_device_status(stream);
    if (earlier == ATTN_ERR_CUDA) return earlier;
    attn_status_t st;
    if ((st = run_mma_rate<0>(sms, stream, &out[0])) != ATTN_OK) return st;
    if ((st = run_mma_rate<1>(sms, stream, &out[1])) != ATTN_OK) return st;
    if ((st = run_mma_rate<2>(sms, stream, &out[2])) != ATTN_OK) return st;
    if ((st = run_mma_rate<3>(sms, stream, &out[3])) != ATTN_OK) return st;
    if ((st = run_mma_rate<4>(sms, stream, &out[4])) != ATTN_OK) return st;
    attn::rates::ex2_rate_kernel<<<sms, attn::rates::kEx2Threads, 0, stream>>>(0.01f);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    long long c[attn::rates::kMaxSms];
    if (cudaMemcpyFromSymbolAsync(c, attn::rates::g_rate_clocks, sizeof(long long) * sms,
                                  sizeof(long long) * attn::rates::kMaxSms, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return ATTN_ERR_CUDA;
    double mean = 0.0;
    for (int i = 0; i < sms; ++i) mean += static_cast<double>(c[i]);
    mean /= sms;
    // warp-level ex2 instructions per SM sub-partition: its warps x iterations x chains
    const double per_smsp = (attn::rates::kEx2Threads / 32 / 4) * static_cast<double>(attn::rates::kEx2Iters) *
                            attn::rates::kEx2Chains;
    out[5] = mean / per_smsp;
    out[6] = 4.0 * 32.0 / out[5];
    out[7] = static_cast<double>(sms);
    const attn_status_t now = attn_check_device_status(stream);
    return now != ATTN_OK ? now : earlier;
}
