// fmha_fwd_sm103.cuh -- fused attention forward for sm_103a (GB300).
//
// Work unit = two 128-row query tiles that read the same K/V head: either two
// consecutive row tiles of one query head, or (when the GQA group has an even
// number of query heads) the same rows of two query heads of one group, so
// every K/V tile brought into shared memory feeds 256 query rows.  Under a causal
// mask units are numbered longest first (row tiles near the end of the sequence
// visit the most KV tiles -- the Choreo tutorial's non-persistent schedule);
// without one every unit is equally long and they are numbered head-major, so
// the units of one K/V head run side by side and its K and V stay in L2; a
// persistent grid of at most one CTA per SM takes them in a snake order
// (round r: CTA c takes unit r*G + c, or r*G + G-1-c on odd rounds), so the
// next unit's Q is loaded while the current one finishes.
//
// Warp roles (512 threads, four warpgroups):
//   warps 0-3    softmax warpgroup of tile 0 (one query row per thread)
//   warps 4-7    softmax warpgroup of tile 1
//   warps 8-11   epilogue warpgroup: O_t out of tensor memory, times 1/l, bf16,
//                TMA store; LSE.  It runs while the softmax warpgroups start the
//                next unit, so the store never sits on the softmax critical path.
//   warp  12     MMA issuer (one elected lane): S_t = Q_t K^T and O_t += P_t V
//   warp  13     TMA producer (one thread): Q of each unit (plus an L2 prefetch of
//                the next unit's Q), K and V tiles in stages: stage g carries V of
//                KV tile g-1 and K of KV tile g (tiles numbered across units), so the
//                MMA warp waits once per KV step, for both operands of that step
//                (P.V with V_j, then S_{j+1} with K_{j+1}), and releases both with
//                one commit
//   warp  14     release warp: once any bounded wait of the CTA has run out, it
//                completes the MMA warp's P barriers (below) until that warp has
//                left its loop
//   warp  15     idle
// Registers are split with setmaxnreg: softmax 176, epilogue 88, MMA/producer 72
// per thread (2*176 + 88 + 72 = 4 * 128, the launch allocation of 128 per thread).
//
// Tensor memory (512 columns x 128 lanes, fp32): S_0 | S_1 | O_0 | O_1, 128 columns
// each.  P_t (bf16, two per column) is written over the first 64 columns of S_t
// and is the A operand of the P.V product straight from tensor memory.
//
// The online softmax follows the Pallas page's kernel loop (`kv_loop`): the row
// maximum is kept in log2 units of the scaled logits so that each weight is one
// FMA and one ex2 (scale * log2e folded into the FMA), the running sum is
// rescaled by alpha = 2^(m_old - m_new), and O is divided by the sum once at the
// end.  The maximum used for the exponentials is only raised when a tile's
// maximum exceeds it by more than 15 (log2 units); otherwise the stale maximum
// is kept (weights stay <= 2^15, inside the fp16 range of P; l and O share it, so
// the quotient is the same), and O in tensor memory is rescaled only on the rare
// tiles that raise it.
// The weights of a tile are handed to the MMA warp in two halves of 64 keys, so
// the first half of O += P.V runs while the second half's exponentials are made.
// That hand-off uses hardware named barriers (softmax warps arrive, the MMA warp
// syncs), not mbarriers: an mbarrier poll by the warp that issued tcgen05.mma
// returns only after that warp's queued MMAs have drained, which left the tensor
// core idle between every group of MMAs, while a named barrier does not wait for
// them.  Each such barrier completes once per (tile, half, KV step): the softmax
// warps of a tile can arrive for step k+1 only after S_t(k+1) exists, which the
// MMA warp issues after its sync for step k, so generations never mix.
//
// Causal masks (bottom-right aligned: key j visible from row i iff j <= i + Skv - Sq;
// top-left aligned: iff j <= i): KV tiles entirely above a tile's last visible key
// are never loaded or multiplied; the element mask is applied only on the tiles that cross the
// diagonal or the ragged key tail.
//
// Every mbarrier wait is bounded: when a wait runs out, the thread records
// ATTN_ERR_TIMEOUT in the device status word and raises a CTA abort flag; all
// roles then leave their loops, in-flight TMA loads and MMAs are drained with
// bounded waits, and tensor memory is freed before the CTA exits.  A named
// barrier cannot time out, so once the abort flag is up the release warp keeps
// arriving on the MMA warp's P barriers (with the softmax warps' thread count)
// until the MMA warp reports that it has left its loop.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda.h>

#include "sm103_ptx.cuh"


namespace attn {

constexpr int kBM = 128;                 // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;                 // keys per KV tile
constexpr int kTiles = 2;                // query tiles per unit
constexpr int kStages = 2;              // K/V stages in flight (one K slot and one V slot each)
constexpr int kHalfBytes = kBM * 64 * 2;         // 128 rows x one 64-column, 128-byte-swizzled half
constexpr int kSoftmaxWarps = 4 * kTiles;          // warpgroups 0 and 1
constexpr int kEpilogueWarp0 = kSoftmaxWarps;      // warpgroup 2
constexpr int kMmaWarp = kEpilogueWarp0 + 4;       // warpgroup 3
constexpr int kLoadWarp = kMmaWarp + 1;
constexpr int kReleaseWarp = kMmaWarp + 2;
// named barriers: 1 = epilogue staging; kBarP + 2 t + h = P_t half h in tensor memory
// (the tile's four softmax warps arrive, the MMA warp syncs)
constexpr uint32_t kBarP = 2;
constexpr uint32_t kBarPThreads = 4 * 32 + 32;
constexpr int kThreads = 512;
constexpr int kRegsSoftmax = 176, kRegsEpilogue = 88, kRegsOther = 72;
static_assert(2 * kRegsSoftmax + kRegsEpilogue + kRegsOther <= 4 * (65536 / kThreads),
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;           // S_t at kTmemS + 128 t
constexpr uint32_t kTmemO = 256;         // O_t at kTmemO + 128 t
constexpr float kRescaleLog2 = 15.0f;    // raise the running max only past 2^15 (fp16 P holds 2^15)

enum : int {
    BAR_QFULL = 0,
    BAR_QEMPTY = BAR_QFULL + kTiles,
    BAR_KVFULL = BAR_QEMPTY + kTiles,        // [stage]: V_{g-1} and K_g landed
    BAR_KVEMPTY = BAR_KVFULL + kStages,      // [stage]: both read by their last MMA
    BAR_SFULL = BAR_KVEMPTY + kStages,
    BAR_ODONE = BAR_SFULL + kTiles,
    BAR_OFREE = BAR_ODONE + kTiles,
    BAR_STATSFULL = BAR_OFREE + kTiles,
    BAR_STATSFREE = BAR_STATSFULL + kTiles,
    BAR_MMADONE = BAR_STATSFREE + kTiles,
    BAR_COUNT
};
// Shared-memory map for head size kD (offsets from a 1024-byte aligned base).
// Every row of a Q, K or V tile is kD / 64 halves of 64 columns, each half a
// 128-row x 128-byte block in the 128-byte swizzle (TMA box and UMMA atom).
template <int kD>
struct Geo {
    static_assert(kD == 64 || kD == 128, "head size 64 or 128");
    static constexpr int kHalves = kD / 64;
    static constexpr int kTileBytes = kBM * kD * 2;  // Q, K or V tile
    static constexpr int kSmemQ = 0;
    static constexpr int kSmemK = kSmemQ + kTiles * kTileBytes;
    static constexpr int kSmemV = kSmemK + kStages * kTileBytes;
    static constexpr int kSmemStage = kSmemV + kStages * kTileBytes;  // O staging: one half
    static constexpr int kSmemStats = kSmemStage + kHalfBytes;         // per tile and row: (m, l)
    static constexpr int kSmemBar = kSmemStats + kTiles * kBM * 8;
    static constexpr int kSmemTmemSlot = kSmemBar + BAR_COUNT * 8;
    static constexpr int kSmemAbort = kSmemTmemSlot + 4;
    static constexpr int kSmemMmaExit = kSmemAbort + 4;  // set once the MMA warp left its loop
    static constexpr int kSmemUsed = kSmemMmaExit + 4;
    static constexpr int kSmemBytes = kSmemUsed + 1024;  // + slack to align the base to 1024 bytes
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-CTA shared memory limit");
};

constexpr unsigned int kStatusTimeout = 1u;

// Device status word: bit 0 = a bounded wait ran out.  Read and cleared by the host.
__device__ unsigned int g_attn_status = 0;

struct FwdParams {
    int B, Sq, Skv, Hq, Hkv;
    int D;                  // head size (64 or 128); selects the kernel instance
    int causal;             // 0: none; 1: bottom-right; 2: top-left
    int diag;               // key j visible from row i iff j <= i + diag (when causal)
    float scale_log2;       // softmax scale * log2(e)
    uint16_t* o;            // [B, Sq, Hq, D] bf16
    float* lse;             // [B, Hq, Sq] fp32, or nullptr
    int head_pairs;         // 1: a unit's tiles are two heads of a GQA group, same rows
    int n_row_units;        // row units per (batch, head unit)
    int n_head_units;       // head units per batch
    int n_units;            // n_row_units * B * n_head_units
    unsigned int poll_limit;  // bound on every mbarrier poll loop
};

// Bounded wait on an mbarrier phase.  Gives up (returns false) if the CTA abort
// flag is raised, or after `limit` polls (then it raises the flag itself).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                             unsigned int limit) {
    for (unsigned int i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 15u) == 15u && *abort_flag) return false;
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

__device__ __forceinline__ void tmem_wait_ld_regs16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
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
__host__ __device__ __forceinline__ int kv_tiles_for(const FwdParams& p, int row0) {
    if (row0 >= p.Sq) return 0;
    const int n_all = (p.Skv + kBN - 1) / kBN;
    if (!p.causal) return n_all;
    const int last_row = row0 + kBM - 1 < p.Sq - 1 ? row0 + kBM - 1 : p.Sq - 1;
    const long long last_key = (long long)last_row + p.diag;
    if (last_key < 0) return 0;
    const long long n = last_key / kBN + 1;
    return n < n_all ? (int)n : n_all;
}

// Decoded work item: a unit, or (split-KV) the KV tiles [kb, kb + nmax) of a unit.
struct Unit {
    int b, hkv;
    int hq0, hq1;      // query heads of tile 0 / tile 1
    int row0, row1;    // first query row of tile 0 / tile 1
    int n0, n1;        // KV tiles each tile visits in this item (from kb on)
    int kb;            // first KV tile of the item
    int slot;          // split-KV: workspace slot of a partial item; -1: final output
    __host__ __device__ __forceinline__ int hq(int t) const { return t ? hq1 : hq0; }
    __host__ __device__ __forceinline__ int row(int t) const { return t ? row1 : row0; }
    __host__ __device__ __forceinline__ int n(int t) const { return t ? n1 : n0; }
    __host__ __device__ __forceinline__ int nmax() const { return n0 > n1 ? n0 : n1; }
};

__host__ __device__ __forceinline__ Unit decode_unit(const FwdParams& p, int u) {
    Unit w;
    int ru, inner;
    if (p.causal) {
        // longest first: row units outermost (descending), then batch and head unit
        const int inner_count = p.B * p.n_head_units;
        ru = u / inner_count;
        inner = u % inner_count;
    } else {
        // every unit visits every KV tile: head-major, so the units of one K/V head
        // run side by side and its K and V stay in L2
        ru = u % p.n_row_units;
        inner = u / p.n_row_units;
    }
    w.b = inner / p.n_head_units;
    const int hu = inner % p.n_head_units;
    const int row_unit = p.causal ? (p.n_row_units - 1 - ru) : ru;
    if (p.head_pairs) {
        w.hq0 = 2 * hu;
        w.hq1 = 2 * hu + 1;
        w.row0 = w.row1 = row_unit * kBM;
    } else {
        w.hq0 = w.hq1 = hu;
        w.row0 = row_unit * (kTiles * kBM);
        w.row1 = w.row0 + kBM;
    }
    w.hkv = w.hq0 / (p.Hq / p.Hkv);
    w.n0 = kv_tiles_for(p, w.row0);
    w.n1 = kv_tiles_for(p, w.row1);
    w.kb = 0;
    w.slot = -1;
    return w;
}

// j-th unit of this CTA in the snake order, or -1 when there is none.
__device__ __forceinline__ int unit_of(const FwdParams& p, int j) {
    const int G = static_cast<int>(gridDim.x);
    const int c = static_cast<int>(blockIdx.x);
    const long long u = (long long)j * G + ((j & 1) ? (G - 1 - c) : c);
    return u < p.n_units ? static_cast<int>(u) : -1;
}

// ---- schedules of work items over the persistent grid
constexpr int kMaxSplitCtas = 256;
// Whole units in the order above, in the snake order of unit_of().
struct PlainSched {
    int unused;
};
// Whole units from a table (causal shapes of up to kMaxTable units): per CTA, the
// units the host assigned to it, in the order it takes them.  The host orders
// the units in blocks of heads whose K and V together fit in part of L2, longest
// first within each block, and hands each unit in turn to the least-loaded CTA,
// so the heads of one block run side by side (their K and V are read from DRAM
// about once) and the CTAs still finish together.
constexpr int kMaxTable = 2048;
struct TableSched {
    unsigned short cta_begin[kMaxSplitCtas + 1];
    unsigned short unit[kMaxTable];
};

// Split-KV: the host cuts the sequence of (unit, KV tile) iterations into equal
// contiguous shares, one per CTA.  A unit that straddles shares becomes several
// pieces; each writes its raw fp32 accumulator and (m, l) to a workspace slot and
// the combine kernel merges them.  Units inside one share write O directly.
struct Piece {
    int unit;
    unsigned int krange;  // first KV tile | (end KV tile << 16)
    int slot;             // workspace slot, or -1 for a whole unit
};
constexpr int kMaxPieces = 1024;
struct SplitSched {
    float* ws_o;          // [slot][tile][row][D] fp32 raw accumulators
    float2* ws_ml;        // [slot][tile][row] (running max in log2 units, row sum)
    int n_pieces;
    unsigned short cta_begin[kMaxSplitCtas + 1];
    Piece piece[kMaxPieces];
};

__device__ __forceinline__ bool get_work(const FwdParams& p, const PlainSched&, int j, Unit& w) {
    const int u = unit_of(p, j);
    if (u < 0) return false;
    w = decode_unit(p, u);
    return true;
}

__device__ __forceinline__ bool get_work(const FwdParams& p, const TableSched& sc, int j, Unit& w) {
    const int i = sc.cta_begin[blockIdx.x] + j;
    if (i >= sc.cta_begin[blockIdx.x + 1]) return false;
    w = decode_unit(p, sc.unit[i]);
    return true;
}

__device__ __forceinline__ bool get_work(const FwdParams& p, const SplitSched& sc, int j, Unit& w) {
    const int i = sc.cta_begin[blockIdx.x] + j;
    if (i >= sc.cta_begin[blockIdx.x + 1]) return false;
    const Piece pc = sc.piece[i];
    w = decode_unit(p, pc.unit);
    const int kb = static_cast<int>(pc.krange & 0xFFFFu), ke = static_cast<int>(pc.krange >> 16);
    w.n0 = max(0, min(w.n0, ke) - kb);
    w.n1 = max(0, min(w.n1, ke) - kb);
    w.kb = kb;
    w.slot = pc.slot;
    return true;
}

// kF16: Q, K, V, O are IEEE binary16 instead of bf16 (P follows the operands).
// kD: head size (64 or 128).
template <class Sched, bool kF16, int kD>
__global__ void __launch_bounds__(kThreads, 1)
    fmha_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p, const __grid_constant__ Sched sched) {
    using G = Geo<kD>;
    extern __shared__ uint8_t smem_raw[];
    // align in the shared window (swizzle atoms and TMA boxes want 1024 bytes)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x) / 32, 0);
    const int lane = static_cast<int>(threadIdx.x) & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::kSmemAbort);
    volatile int* mma_exit = reinterpret_cast<volatile int*>(smem + G::kSmemMmaExit);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kSmemTmemSlot);
    auto bar = [&](int i) -> uint32_t { return sbase + G::kSmemBar + 8 * i; };

    // ---- set-up: barriers, abort flag, tensor memory
    if (warp == kLoadWarp && lane == 0) {
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bar(BAR_QFULL + t), 1);
            mbar_init(bar(BAR_QEMPTY + t), 1);
            mbar_init(bar(BAR_SFULL + t), 1);
            mbar_init(bar(BAR_ODONE + t), 1);
            mbar_init(bar(BAR_OFREE + t), 4 * 32);
            mbar_init(bar(BAR_STATSFULL + t), 4 * 32);
            mbar_init(bar(BAR_STATSFREE + t), 4 * 32);
        }
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(BAR_KVFULL + s), 1);
            mbar_init(bar(BAR_KVEMPTY + s), 1);
        }
        mbar_init(bar(BAR_MMADONE), 1);
        *abort_flag = 0;
        *mma_exit = 0;
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
    const int wg = warp / 4;

    if (wg == 3) {
      regs_dec<kRegsOther>();  // warpgroup-wide, before the warps take their roles
      if (warp == kLoadWarp) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            // K and V stream as stages: stage g holds V of fill g-1 and K of fill g
            // (fills numbered across units), both released by the same MMA commit
            // (the end of the KV step that reads V_{g-1} with P.V and K_g with the
            // next S); barrier pair KVFULL/KVEMPTY[g % kStages].  The Q tiles of a
            // unit are loaded right after the stage that brings its K_0.
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            int g = 0;                       // stages issued
            int q_issued[kTiles] = {0, 0};   // Q_t fills issued so far
            int jq = 0;                      // next unit whose Q is to be loaded
            bool ok = true;
            auto issue_q_upto = [&](int jmax) -> bool {
                for (; jq <= jmax; ++jq) {
                    Unit w;
                    if (!get_work(p, sched, jq, w)) return true;
                    for (int t = 0; t < kTiles; ++t) {
                        if (jq > 0 && !wait_bounded(bar(BAR_QEMPTY + t), (jq - 1) & 1, abort_flag, limit))
                            return false;
                        mbar_arrive_expect_tx(bar(BAR_QFULL + t), G::kTileBytes);
                        for (int h = 0; h < G::kHalves; ++h)
                            tma_load_4d(sbase + G::kSmemQ + t * G::kTileBytes + h * kHalfBytes, &tm_q, h * 64,
                                        w.hq(t), w.row(t), w.b, bar(BAR_QFULL + t), pol_q);
                        ++q_issued[t];
                    }
                    Unit wn;
                    if (get_work(p, sched, jq + 1, wn)) {  // warm L2 with the next unit's Q meanwhile
                        for (int t = 0; t < kTiles; ++t)
                            for (int h = 0; h < G::kHalves; ++h)
                                tma_prefetch_l2_4d(&tm_q, h * 64, wn.hq(t), wn.row(t), wn.b);
                    }
                }
                return true;
            };
            // K cursor (the fill of the next stage's K) and V cursor (the previous one)
            int jk = 0, ktk = 0;
            Unit wk;
            bool have_k = get_work(p, sched, 0, wk);
            while (have_k && ktk >= wk.nmax()) {
                ++jk;
                ktk = 0;
                have_k = get_work(p, sched, jk, wk);
            }
            Unit wv = wk;
            int ktv = 0;
            bool have_v = false;
            while (ok && (have_k || have_v)) {
                const int st = g % kStages, use = g / kStages;
                if (use > 0 && !wait_bounded(bar(BAR_KVEMPTY + st), (use - 1) & 1, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(bar(BAR_KVFULL + st), ((have_k ? 1 : 0) + (have_v ? 1 : 0)) * G::kTileBytes);
                if (have_v) {
                    const int vs = (g - 1) % kStages;
                    for (int h = 0; h < G::kHalves; ++h)
                        tma_load_4d(sbase + G::kSmemV + vs * G::kTileBytes + h * kHalfBytes, &tm_v, h * 64,
                                    wv.hkv, (wv.kb + ktv) * kBN, wv.b, bar(BAR_KVFULL + st), pol_kv);
                }
                if (have_k) {
                    for (int h = 0; h < G::kHalves; ++h)
                        tma_load_4d(sbase + G::kSmemK + st * G::kTileBytes + h * kHalfBytes, &tm_k, h * 64,
                                    wk.hkv, (wk.kb + ktk) * kBN, wk.b, bar(BAR_KVFULL + st), pol_kv);
                }
                ++g;  // counted before anything can fail: the drain below waits for these copies
                if (have_k && ktk == 0 && !issue_q_upto(jk)) {
                    ok = false;
                    break;
                }
                have_v = have_k;
                wv = wk;
                ktv = ktk;
                if (have_k) {
                    ++ktk;
                    while (have_k && ktk >= wk.nmax()) {
                        ++jk;
                        ktk = 0;
                        have_k = get_work(p, sched, jk, wk);
                    }
                }
            }
            if (ok) issue_q_upto(0x7fffffff);  // units after the last fill (without KV work) still need Q
            // drain: every copy this thread issued has landed before the CTA may exit
            for (int t = 0; t < kTiles; ++t)
                if (q_issued[t] > 0) drain_bounded(bar(BAR_QFULL + t), (q_issued[t] - 1) & 1, limit);
            for (int st = 0; st < kStages; ++st) {
                const int fills = g > st ? (g - 1 - st) / kStages + 1 : 0;
                if (fills) drain_bounded(bar(BAR_KVFULL + st), (fills - 1) & 1, limit);
            }
        }
        __syncwarp();
      } else if (warp == kMmaWarp) {
        // =========================== MMA issuer =============================
        // The whole warp runs the control flow (so descriptors and stage indices stay
        // warp-uniform); one elected lane issues each group of MMAs and its commits.
        constexpr uint32_t idesc_qk = idesc_f16kind_f32(kBM, kBN, false, kF16);
        constexpr uint32_t idesc_pv = idesc_f16kind_f32(kBM, kD, true, kF16);
        // descriptor of k-step kk = base descriptor + constant start-address offset (>> 4)
        const uint64_t q_desc0 = sdesc_sw128(sbase + G::kSmemQ, 16, 1024);
        const uint64_t k_desc0 = sdesc_sw128(sbase + G::kSmemK, 16, 1024);
        const uint64_t v_desc0 = sdesc_sw128(sbase + G::kSmemV, kHalfBytes, 1024);
        auto issue_qk = [&](int t, int ks) {
            const uint32_t d = tmem_base + kTmemS + 128 * t;
            const uint64_t qd = q_desc0 + static_cast<uint64_t>((t * G::kTileBytes) >> 4);
            const uint64_t kd = k_desc0 + static_cast<uint64_t>((ks * G::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
                const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4);
                mma_bf16_ss(d, qd + off, kd + off, idesc_qk, kk > 0 ? 1u : 0u);
            }
        };
        // O_t (+)= P_t V over keys [64 h, 64 h + 64) of the KV tile
        auto issue_pv = [&](int t, int vs, int h, bool accumulate) {
            const uint32_t d = tmem_base + kTmemO + 128 * t;
            const uint32_t pa = tmem_base + kTmemS + 128 * t;
            const uint64_t vd = v_desc0 + static_cast<uint64_t>((vs * G::kTileBytes) >> 4);
#pragma unroll
            for (int q = 0; q < kBN / 32; ++q) {
                const int kk = h * (kBN / 32) + q;
                mma_bf16_ts(d, pa + kk * 8, vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_pv,
                            (accumulate || kk > 0) ? 1u : 0u);
            }
        };
        int kv = 0;                 // KV tiles consumed so far (stage kv carries K_kv)
        bool ok = true;
        for (int j = 0; ok; ++j) {
            Unit w;
            if (!get_work(p, sched, j, w)) break;
            const int nm = w.nmax();
            // S_t(0) for each tile that has work; Q_t must have landed, and stage kv
            // (this unit's K_0, with V of the previous unit's last KV tile)
            bool k_ready = false;
            for (int t = 0; t < kTiles && ok; ++t) {
                ok = wait_bounded(bar(BAR_QFULL + t), j & 1, abort_flag, limit);
                if (!ok) break;
                if (w.n(t) > 0 && !k_ready) {
                    ok = wait_bounded(bar(BAR_KVFULL + kv % kStages), (kv / kStages) & 1, abort_flag, limit);
                    if (!ok) break;
                    k_ready = true;
                }
                tc_fence_after();
                if (elect_one()) {
                    if (w.n(t) > 0) {
                        issue_qk(t, kv % kStages);
                        mma_commit(bar(BAR_SFULL + t));
                    }
                    if (w.n(t) <= 1) mma_commit(bar(BAR_QEMPTY + t));  // Q_t no longer read
                }
                __syncwarp();
            }
            if (!ok) break;
            if (nm > 0) {  // stage kv: its V was read by the previous unit's last P.V, its K now
                if (elect_one()) mma_commit(bar(BAR_KVEMPTY + kv % kStages));
                __syncwarp();
            }
            for (int kt = 0; ok && kt < nm; ++kt) {
                const int vs = kv % kStages;
                const int kn = kv + 1;  // stage kn: V_{kt} and K_{kt+1} (or the next unit's K_0)
                if (!wait_bounded(bar(BAR_KVFULL + kn % kStages), (kn / kStages) & 1, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int t = 0; t < kTiles; ++t) {
                    const int nt = w.n(t);
                    if (kt < nt) {
                        // the first P.V of a unit overwrites O_t: the previous unit's
                        // epilogue must have read it out of tensor memory
                        if (kt == 0 && j > 0 &&
                            !wait_bounded(bar(BAR_OFREE + t), (j - 1) & 1, abort_flag, limit)) {
                            ok = false;
                            break;
                        }
                        // P_t(kt) arrives in two halves of 64 keys; each half's P.V starts
                        // as soon as the softmax warpgroup has stored it
                        for (int h = 0; h < 2; ++h) {
                            named_bar_sync(kBarP + 2 * t + h, kBarPThreads);
                            tc_fence_after();
                            if (elect_one()) {
                                issue_pv(t, vs, h, kt > 0);
                                if (h == 1 && kt == nt - 1) mma_commit(bar(BAR_ODONE + t));  // O_t final
                            }
                            __syncwarp();
                        }
                        if (!ok) break;
                    } else if (nt == 0 && kt == 0) {
                        // tile without work: its (all-zero) O_t is "final" now, but only after
                        // the previous unit's O_t was read, which keeps this barrier's phases
                        // in step with the epilogue that waits on them
                        if (j > 0 && !wait_bounded(bar(BAR_OFREE + t), (j - 1) & 1, abort_flag, limit)) {
                            ok = false;
                            break;
                        }
                        if (elect_one()) mma_commit(bar(BAR_ODONE + t));
                        __syncwarp();
                    }
                    if (kt + 1 < nt) {
                        if (elect_one()) {
                            issue_qk(t, kn % kStages);
                            mma_commit(bar(BAR_SFULL + t));
                            if (kt + 2 == nt) mma_commit(bar(BAR_QEMPTY + t));  // last S_t of the unit
                        }
                        __syncwarp();
                    }
                }
                if (!ok) break;
                // stage kn is free once V_kt and K_{kt+1} have been read; after the unit's
                // last step its K belongs to the next unit and is released there
                if (kt + 1 < nm && elect_one()) mma_commit(bar(BAR_KVEMPTY + kn % kStages));
                __syncwarp();
                ++kv;
            }
            for (int t = 0; ok && nm == 0 && t < kTiles; ++t) {  // unit without any work
                if (j > 0 && !wait_bounded(bar(BAR_OFREE + t), (j - 1) & 1, abort_flag, limit)) {
                    ok = false;
                    break;
                }
                if (elect_one()) mma_commit(bar(BAR_ODONE + t));
                __syncwarp();
            }
        }
        *mma_exit = 1;  // the release warp may stop
        // every MMA this warp issued has completed before tensor memory is freed
        if (elect_one()) {
            mma_commit(bar(BAR_MMADONE));
            drain_bounded(bar(BAR_MMADONE), 0, limit);
        }
        __syncwarp();
      } else if (warp == kReleaseWarp) {
        // =========================== release warp ===========================
        // Sleeps until the MMA warp leaves its loop; if the abort flag goes up first,
        // it arrives on every P barrier (as the softmax warps would) so that an MMA
        // warp waiting there moves on, sees the abort at its next bounded wait and
        // leaves.  Surplus arrivals only complete generations nobody waits for.
        const unsigned long long cap = 64ull * limit;
        unsigned long long i = 0;
        for (; i < cap && !*mma_exit; ++i) {
            if (*abort_flag) {
                for (int b = 0; b < 2 * kTiles; ++b)
                    for (int k = 0; k < 4; ++k) named_bar_arrive(kBarP + b, kBarPThreads);
            } else {
                nanosleep_ns(1024);
            }
        }
        if (i == cap) atomicOr(&g_attn_status, kStatusTimeout);
      }
    } else if (wg < 2) {
        // =========================== softmax warpgroups =====================
        regs_inc<kRegsSoftmax>();
        const int t = warp / 4;
        const int wq = warp % 4;
        const int r = wq * 32 + lane;  // row within the tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem_base + lane_off + kTmemS + 128 * t;
        const uint32_t tO = tmem_base + lane_off + kTmemO + 128 * t;
        const float sl2 = p.scale_log2;
        int sc = 0;  // S_t products consumed so far
        bool ok = true;

        for (int j = 0; ok; ++j) {
            Unit w;
            if (!get_work(p, sched, j, w)) break;
            const int nt = w.n(t);
            const int row = w.row(t) + r;
            const long long lim_ll = p.causal ? min((long long)row + p.diag, (long long)p.Skv - 1)
                                              : (long long)p.Skv - 1;
            const int lim = static_cast<int>(lim_ll < -1 ? -1 : lim_ll);  // last visible key
            float m_run = -INFINITY;  // running max (log2 units of scaled logits) used by the weights
            float l_run = 0.f;        // running sum of weights

            for (int kt = 0; kt < nt; ++kt, ++sc) {
                // warp-uniform outcome: the tcgen05.ld/st below are warp-collective
                const bool got = wait_bounded(bar(BAR_SFULL + t), sc & 1, abort_flag, limit);
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

                const int nvis = lim - (w.kb + kt) * kBN + 1;  // visible keys of this row in the tile
                if (nvis < kBN) {
#pragma unroll
                    for (int jj = 0; jj < kBN; ++jj)
                        if (jj >= nvis) s[jj] = __float_as_uint(-INFINITY);
                }
                // tile maximum (three-input max, 8 independent chains)
                float mx[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    mx[q] = fmax3(__uint_as_float(s[q]), __uint_as_float(s[8 + q]), __uint_as_float(s[16 + q]));
#pragma unroll
                for (int base = 24; base < kBN; base += 16)
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        mx[q] = fmax3(mx[q], __uint_as_float(s[base + q]), __uint_as_float(s[base + 8 + q]));
                const float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                         fmaxf(mx[6], mx[7]));
                const float m_tile = tmax * sl2;

                // raise the running max only when the tile max exceeds it by more than 2^15
                // (always on the first tile with a visible key: then alpha = 0)
                float alpha = 1.f;
                if (m_tile - m_run > kRescaleLog2) {
                    alpha = ex2_approx(m_run - m_tile);
                    m_run = m_tile;
                }
                const float m_use = m_run == -INFINITY ? 0.f : m_run;
                // O_t holds P.V of tiles < kt (complete: S_t(kt) was issued after them);
                // rescale it before this tile's first P.V half may start
                const bool need = (kt > 0) && (alpha != 1.f);
                if (__any_sync(0xffffffffu, need)) {
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
                // weights 2^(s*scale*log2e - m_use), their row sum, packed to bf16 pairs and
                // stored as P_t in two halves of 64 keys (32 columns); each half is handed
                // to the MMA warp as soon as it is in tensor memory
                float rs0 = 0.f, rs1 = 0.f, rs2 = 0.f, rs3 = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
#pragma unroll
                    for (int c = 2 * h; c < 2 * h + 2; ++c) {
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
                    named_bar_arrive(kBarP + 2 * t + h, kBarPThreads);
                }
                l_run = l_run * alpha + ((rs0 + rs1) + (rs2 + rs3));
            }
            if (!ok) break;

            // hand (m, l) of every row to the epilogue warpgroup and start the next unit
            if (j > 0 && !wait_bounded(bar(BAR_STATSFREE + t), (j - 1) & 1, abort_flag, limit)) {
                ok = false;
                break;
            }
            reinterpret_cast<float2*>(smem + G::kSmemStats)[t * kBM + r] = make_float2(m_run, l_run);
            mbar_arrive(bar(BAR_STATSFULL + t));
        }
    } else if (wg == 2) {
        // =========================== epilogue warpgroup =====================
        regs_dec<kRegsEpilogue>();
        const int wq = warp % 4;
        const int r = wq * 32 + lane;  // row within a tile = TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        uint8_t* stage = smem + G::kSmemStage;
        bool ok = true;
        for (int j = 0; ok; ++j) {
            Unit w;
            if (!get_work(p, sched, j, w)) break;
            for (int t = 0; t < kTiles; ++t) {
                // O_t final (every P.V of the unit completed) and (m, l) of its rows
                const bool got = wait_bounded(bar(BAR_ODONE + t), j & 1, abort_flag, limit) &&
                                 wait_bounded(bar(BAR_STATSFULL + t), j & 1, abort_flag, limit);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float2 ml = reinterpret_cast<const float2*>(smem + G::kSmemStats)[t * kBM + r];
                mbar_arrive(bar(BAR_STATSFREE + t));
                const float m_run = ml.x, l_run = ml.y;
                const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
                const int nt = w.n(t);
                const int row = w.row(t) + r;
                const uint32_t tO = tmem_base + lane_off + kTmemO + 128 * t;
                const bool tile_in_range = w.row(t) < p.Sq;
                if constexpr (std::is_same<Sched, SplitSched>::value) {
                    if (w.slot >= 0) {
                        // a piece of a split unit: the raw fp32 accumulator and (m, l) of
                        // every row go to its workspace slot for the combine kernel
                        const size_t rr = (static_cast<size_t>(w.slot) * kTiles + t) * kBM + r;
                        uint4* dst = reinterpret_cast<uint4*>(sched.ws_o + rr * kD);
#pragma unroll
                        for (int h = 0; h < G::kHalves; ++h) {
                            uint32_t o[64];
                            if (nt > 0) {
                                tmem_ld32(tO + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                                tmem_ld32(tO + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                                tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                                tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                            } else {
#pragma unroll
                                for (int e = 0; e < 64; ++e) o[e] = 0u;
                            }
                            if (h == G::kHalves - 1) {  // O_t may now be overwritten by the next item's first P.V
                                tc_fence_before();
                                mbar_arrive(bar(BAR_OFREE + t));
                            }
#pragma unroll
                            for (int q = 0; q < 16; ++q)
                                dst[16 * h + q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
                        }
                        sched.ws_ml[rr] = make_float2(m_run, l_run);
                        continue;
                    }
                }
                // two 64-column halves: TMEM -> registers -> (1/l) -> bf16 -> swizzled
                // staging -> one TMA store each (rows past Sq are clipped by the store)
#pragma unroll
                for (int h = 0; h < G::kHalves; ++h) {
                    uint32_t o[64];
                    if (nt > 0) {
                        tmem_ld32(tO + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                        tmem_ld32(tO + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                        tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&o[0]));
                        tmem_wait_ld_regs(*reinterpret_cast<uint32_t(*)[32]>(&o[32]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 64; ++e) o[e] = 0u;
                    }
                    if (h == G::kHalves - 1) {  // O_t may now be overwritten by the next unit's first P.V
                        tc_fence_before();
                        mbar_arrive(bar(BAR_OFREE + t));
                    }
                    if (r == 0) bulk_wait_group_read0();  // the previous store has read the staging
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {  // 16-byte chunk q of this row's half
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; e += 2)
                            fmul2_b(f[e], f[e + 1], __uint_as_float(o[8 * q + e]), __uint_as_float(o[8 * q + e + 1]),
                                    inv_l);
                        *reinterpret_cast<uint4*>(stage + r * 128 + ((q ^ (r & 7)) * 16)) =
                            make_uint4(pack_x2<kF16>(f[0], f[1]), pack_x2<kF16>(f[2], f[3]),
                                       pack_x2<kF16>(f[4], f[5]), pack_x2<kF16>(f[6], f[7]));
                    }
                    fence_proxy_async_smem();
                    named_bar_sync(1, 128);
                    if (r == 0 && tile_in_range) {
                        tma_store_4d(&tm_o, smem_u32(stage), h * 64, w.hq(t), w.row(t), w.b);
                        bulk_commit_group();
                    }
                }
                if (row < p.Sq && p.lse != nullptr) {
                    const float lse = l_run > 0.f ? (m_run + log2f(l_run)) * 0.69314718055994531f : -INFINITY;
                    p.lse[(static_cast<size_t>(w.b) * p.Hq + w.hq(t)) * p.Sq + row] = lse;
                }
            }
        }
        if (r == 0) bulk_wait_group0();  // every O store has completed before the CTA exits
    }

    // ---- teardown: all tensor-memory traffic is complete; free it
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---- split-KV combine
// Merges the partial (m, l, O) of the pieces of each split unit -- the rule of the
// kernbench page's `_merge_running`, in log2 units:
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  O = sum_s O_s 2^(m_s - M) / L,
//   LSE = (M + log2 L) ln 2;  a row no piece saw a key of gets O = 0, LSE = -inf.
// One warp per (split unit, tile, row); lane i owns columns [i D/32, (i+1) D/32).
struct CombineEntry {
    int unit;
    int first_slot;
    int n_slots;
};
constexpr int kMaxCombine = 512;
constexpr int kCombineWarps = 8;
struct CombineTable {
    const float* ws_o;
    const float2* ws_ml;
    uint16_t* o;          // [B, Sq, Hq, D] bf16 or f16
    int n;
    CombineEntry e[kMaxCombine];
};

template <bool kF16, int kD>
__global__ void __launch_bounds__(32 * kCombineWarps)
    splitkv_combine_kernel(const FwdParams p, const __grid_constant__ CombineTable ct) {
    const int gw = static_cast<int>(blockIdx.x) * kCombineWarps + static_cast<int>(threadIdx.x) / 32;
    const int lane = static_cast<int>(threadIdx.x) & 31;
    const int entry = gw / (kTiles * kBM);
    if (entry >= ct.n) return;
    const int t = (gw / kBM) % kTiles;
    const int r = gw % kBM;
    const CombineEntry e = ct.e[entry];
    const Unit w = decode_unit(p, e.unit);
    const int row = w.row(t) + r;
    if (row >= p.Sq) return;
    float M = -INFINITY;
    for (int sl = 0; sl < e.n_slots; ++sl) {
        const float2 ml = ct.ws_ml[((static_cast<size_t>(e.first_slot) + sl) * kTiles + t) * kBM + r];
        if (ml.y > 0.f) M = fmaxf(M, ml.x);
    }
    constexpr int kPer = kD / 32;  // columns per lane (4 or 2)
    float L = 0.f;
    float acc[kPer] = {};
    for (int sl = 0; sl < e.n_slots; ++sl) {
        const size_t rr = ((static_cast<size_t>(e.first_slot) + sl) * kTiles + t) * kBM + r;
        const float2 ml = ct.ws_ml[rr];
        if (!(ml.y > 0.f)) continue;  // this piece saw no key of the row
        const float a = exp2f(ml.x - M);
        const float* src = ct.ws_o + rr * kD + kPer * lane;
        float v[kPer];
        if constexpr (kPer == 4) {
            const float4 x = *reinterpret_cast<const float4*>(src);
            v[0] = x.x, v[1] = x.y, v[2] = x.z, v[3] = x.w;
        } else {
            const float2 x = *reinterpret_cast<const float2*>(src);
            v[0] = x.x, v[1] = x.y;
        }
        L += ml.y * a;
#pragma unroll
        for (int i = 0; i < kPer; ++i) acc[i] += v[i] * a;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* dst = ct.o + ((static_cast<size_t>(w.b) * p.Sq + row) * p.Hq + w.hq(t)) * kD + kPer * lane;
    if constexpr (kPer == 4) {
        uint2 out;
        out.x = pack_x2<kF16>(acc[0] * inv, acc[1] * inv);
        out.y = pack_x2<kF16>(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(dst) = out;
    } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_x2<kF16>(acc[0] * inv, acc[1] * inv);
    }
    if (lane == 0 && p.lse != nullptr)
        p.lse[(static_cast<size_t>(w.b) * p.Hq + w.hq(t)) * p.Sq + row] =
            L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
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
