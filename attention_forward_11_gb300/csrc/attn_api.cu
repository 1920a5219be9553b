// attn_api.cu -- host side of libattn: argument validation, TMA descriptor
// encoding, work decomposition and the launch of the sm_103a kernels.  The
// checks mirror the Pallas page's `_attention_forward` (shapes, GQA
// divisibility, dtype, head size) but accept any sequence length: ragged
// tails are handled inside the kernel by TMA zero-fill and key masking.
#include <attn.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "fmha_fwd_sm103.cuh"

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
bool encode_bshd(CUtensorMap* map, const void* ptr, int B, int S, int H, int D) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2,
                                   (cuuint64_t)S * H * D * 2};
    const cuuint32_t box[4] = {64, 1, (cuuint32_t)attn::kBM, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device one-time set-up: the kernel's shared-memory opt-in and the SM count.
bool device_setup(int dev, int* sm_count) {
    static std::mutex mu;
    static int sms[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (sms[dev] == 0) {
        int n = 0;
        if (cudaFuncSetAttribute(attn::fmha_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 attn::kSmemBytes) != cudaSuccess ||
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

}  // namespace

extern "C" attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                                  int B, int Sq, int Skv, int Hq, int Hkv, int D, int causal,
                                  float scale, cudaStream_t stream) {
    // ---- validation: nothing is launched on any error
    if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || Sq < 1 || Skv < 1 || Hq < 1 || Hkv < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    for (const void* ptr : {q, k, v, static_cast<const void*>(o)})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return ATTN_ERR_INVALID_ARG;
    if (lse && reinterpret_cast<uintptr_t>(lse) % 4 != 0) return ATTN_ERR_INVALID_ARG;
    const size_t q_bytes = (size_t)B * Sq * Hq * D * 2;
    const size_t kv_bytes = (size_t)B * Skv * Hkv * D * 2;
    if (ranges_overlap(o, q_bytes, q, q_bytes) || ranges_overlap(o, q_bytes, k, kv_bytes) ||
        ranges_overlap(o, q_bytes, v, kv_bytes))
        return ATTN_ERR_INVALID_ARG;
    if (lse && (ranges_overlap(lse, (size_t)B * Hq * Sq * 4, o, q_bytes) ||
                ranges_overlap(lse, (size_t)B * Hq * Sq * 4, q, q_bytes)))
        return ATTN_ERR_INVALID_ARG;
    if (D != attn::kHeadDim) return ATTN_ERR_UNSUPPORTED;

    // ---- work decomposition: two 128-row query tiles per CTA sharing one K/V head
    attn::FwdParams p{};
    p.B = B;
    p.Sq = Sq;
    p.Skv = Skv;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.causal = causal;
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

    CUtensorMap tm_q, tm_k, tm_v, tm_o;
    if (!encode_bshd(&tm_q, q, B, Sq, Hq, D) || !encode_bshd(&tm_k, k, B, Skv, Hkv, D) ||
        !encode_bshd(&tm_v, v, B, Skv, Hkv, D) || !encode_bshd(&tm_o, o, B, Sq, Hq, D))
        return ATTN_ERR_CUDA;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || !device_setup(dev, &sms)) return ATTN_ERR_CUDA;
    // persistent grid: at most one CTA per SM (the CTA holds all 512 TMEM columns)
    const int grid = static_cast<int>(n_units < sms ? n_units : sms);
    attn::fmha_fwd_kernel<<<static_cast<unsigned int>(grid), attn::kThreads, attn::kSmemBytes,
                            stream>>>(tm_q, tm_k, tm_v, tm_o, p);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return ATTN_OK;
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

extern "C" attn_status_t attn_check_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
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
