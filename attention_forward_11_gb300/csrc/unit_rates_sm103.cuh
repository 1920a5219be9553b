// unit_rates_sm103.cuh -- measured issue rates of the two units the attention
// loop leans on: the tensor pipe (tcgen05.mma kind::f16, M = 128, K = 16, for
// the operand sources and N the kernels use) and the exponential unit
// (ex2.approx.ftz.f32).  The forward's tile costs 2 x 8 MMAs of 128x128x16 and
// 16384 ex2 per 128x128 tile; whether the exponentials can hide under the
// products decides whether part of them must move to the FMA pipe (a
// polynomial exp2, as the CuTe-DSL FA4 design does on B200).
//
// Both kernels run one CTA per SM (the dynamic shared memory request keeps a
// second CTA off the SM) and time themselves with the SM clock.
#pragma once
#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {
namespace rates {

constexpr int kMmaIters = 1000;          // groups of 8 MMAs (one K = 128 chain each)
constexpr int kMmaSmem = 140000;         // > half an SM's shared memory: one CTA per SM
constexpr int kEx2Iters = 4096;
constexpr int kEx2Chains = 16;           // independent exponentials per thread per iteration
constexpr int kEx2Threads = 256;         // two warps per SM sub-partition
constexpr int kMaxSms = 1024;            // bound of the per-CTA result array
constexpr unsigned int kWaitLimit = 1u << 26;

// Per-CTA clock counts of the last run: [0, kMaxSms) MMA kernel, [kMaxSms, 2 kMaxSms) ex2 kernel.
__device__ long long g_rate_clocks[2 * kMaxSms];
__device__ float g_rate_sink;

// kMode: 0 SS N=128, 1 TS N=128 (A in tensor memory), 2 SS N=256, 3 SS N=64, 4 TS N=64.
// The operands are zeros (the MMA's duration does not depend on the values).
template <int kMode>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel() {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t a_smem = sbase, b_smem = sbase + 32768;   // A 128x128, B up to 256x128 bf16
    const uint32_t bar = sbase + 98304;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 98304 + 8);
    const int warp = static_cast<int>(threadIdx.x) / 32;
    for (int i = static_cast<int>(threadIdx.x); i < 98304 / 16; i += 128)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    fence_proxy_async_smem();  // the zeros are read by the tensor core (async proxy)
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    volatile int* mma_done = reinterpret_cast<volatile int*>(smem + 98304 + 12);
    constexpr bool kTS = kMode == 1 || kMode == 4;
    constexpr uint32_t kN = kMode == 2 ? 256 : (kMode == 3 || kMode == 4) ? 64 : 128;
    if (threadIdx.x == 0) {
        constexpr uint32_t idesc = idesc_f16kind_f32(128, kN, false, false);
        const uint64_t ad = sdesc_sw128(a_smem, 16, 1024), bd = sdesc_sw128(b_smem, 16, 1024);
        const long long t0 = clock64();
        for (int it = 0; it < kMmaIters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t aoff = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                const uint64_t boff = static_cast<uint64_t>(((kk >> 2) * (kN * 128) + (kk & 3) * 32) >> 4);
                const uint32_t acc = (it | kk) ? 1u : 0u;
                if (kTS)
                    mma_bf16_ts(tmem, tmem + 256 + kk * 8, bd + boff, idesc, acc);
                else
                    mma_bf16_ss(tmem, ad + aoff, bd + boff, idesc, acc);
            }
        }
        mma_commit(bar);
        bool done = false;
        for (unsigned int i = 0; i < kWaitLimit && !done; ++i) done = mbar_try_wait(bar, 0);
        g_rate_clocks[blockIdx.x] = clock64() - t0;
        if (!done) {
            atomicOr(&g_attn_status, kStatusTimeout);
            // a second bounded wait: the MMAs may still be reading shared memory
            // and writing tensor memory, which must not be freed under them
            for (unsigned int i = 0; i < kWaitLimit && !done; ++i) done = mbar_try_wait(bar, 0);
        }
        *mma_done = done ? 1 : 0;
    }
    tc_fence_before();
    __syncthreads();
    // freed only when every MMA is known complete; otherwise the status word
    // already reports the timeout and the columns are left to the CTA's exit
    if (warp == 0 && *mma_done) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// kEx2Chains independent chains of exponentials per thread, each step feeding
// the next (x <- -2^x, which stays in (-1, 0)), so that no two exponentials
// have the same input and none can be merged or hoisted by the assembler; the
// sums keep the results live.  Two warps per SM sub-partition keep the unit fed.
__global__ void __launch_bounds__(kEx2Threads, 1) ex2_rate_kernel(float seed) {
    float x[kEx2Chains], acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kEx2Chains; ++k) x[k] = -seed * static_cast<float>(k + 1 + (threadIdx.x & 7));
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < kEx2Iters; ++it) {
#pragma unroll
        for (int k = 0; k < kEx2Chains; ++k) {
            float y;
            asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x[k]));
            x[k] = -y;
            acc[k & 3] += y;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) g_rate_clocks[kMaxSms + blockIdx.x] = clock64() - t0;
    const float s = (acc[0] + acc[1]) + (acc[2] + acc[3]);
    if (s == 12345.f) g_rate_sink = s;  // keeps the sums (and so the ex2) live
}

}  // namespace rates
}  // namespace attn
