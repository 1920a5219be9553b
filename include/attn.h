/*
 * attn.h -- C ABI of libattn, a GB300 (sm_103a) fused attention forward pass.
 *
 * The operation is scaled-dot-product attention as the JAX Pallas page
 * (attention_mgpu.py) defines it in `attention_reference`, with the caller's
 * softmax scale applied to the logits, grouped-query heads mapped as in that
 * page's `_attention_forward` (kv_head = q_head / (Hq / Hkv)), and the
 * log-sum-exp residual that page stores for the backward pass:
 *
 *     S   = scale * Q K^T              (per batch b, query head h, kv head g)
 *     O   = softmax(S [+ causal mask]) V
 *     LSE = ln sum_j exp(S_ij)         (natural log, fp32)
 *
 * It is computed tile by tile with an online softmax (running row max m, row
 * sum l and an fp32 accumulator, exp2 of pre-scaled logits, one final division
 * by l), the schedule of the Pallas page's kernel loop and of the Choreo
 * tutorial's non-persistent FA kernel, on Blackwell tensor cores (tcgen05).
 *
 * Plain pointers and sizes only; no framework types.  All functions are
 * thread-safe.  The library allocates no device memory.
 */
#ifndef LIBATTN_ATTN_H_
#define LIBATTN_ATTN_H_

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment, scale or flag; nothing launched */
    ATTN_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (D != 128)      */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or the kernel launch failed       */
    ATTN_ERR_TIMEOUT = 4      /* a device-side bounded wait ran out (see attn_check_device_status) */
} attn_status_t;

/*
 * attn_fwd -- O = softmax(scale * Q K^T [+ mask]) V and LSE, asynchronously on `stream`.
 *
 * q    device pointer, bf16, [B, Sq, Hq, D], D contiguous (row stride Hq*D elements)
 * k, v device pointers, bf16, [B, Skv, Hkv, D]
 * o    device pointer, bf16, [B, Sq, Hq, D]   (written; round-to-nearest-even of O)
 * lse  device pointer, fp32, [B, Hq, Sq], or NULL to skip it
 * B, Sq, Skv, Hq, Hkv, D  sizes; every one >= 1, Hq a multiple of Hkv, D == 128.
 *      Sq and Skv may be any length (ragged tails are handled in the kernel).
 * causal 0: every key visible.  1: key j visible from query i iff
 *      j <= i + (Skv - Sq) (bottom-right aligned; the top-left rule of the
 *      Pallas page when Sq == Skv).  A query row that sees no key gets O = 0
 *      and LSE = -inf.
 * scale  finite, > 0 (typically 1/sqrt(D)).
 * stream CUDA stream the kernel runs on (0 = legacy default stream).
 *
 * Ownership: the caller owns every buffer; nothing is retained after return.
 * q, k, v, o must be 16-byte aligned (TMA).  o must not alias q, k or v.
 * Returns ATTN_OK once the kernel is enqueued; a device-side wait that runs out
 * is reported later through attn_check_device_status.  On any error return,
 * nothing was launched and no output was written.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Sq, int Skv, int Hq, int Hkv, int D, int causal, float scale,
                       cudaStream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char* attn_status_str(attn_status_t status);

/*
 * Synchronises `stream`, then reads and clears this device's kernel status
 * word.  Returns ATTN_ERR_TIMEOUT if any libattn kernel on the current device
 * gave up a bounded wait since the last check (its outputs are then invalid),
 * ATTN_ERR_CUDA if synchronisation itself failed, else ATTN_OK.
 */
attn_status_t attn_check_device_status(cudaStream_t stream);

/* Number of kernels libattn has enqueued in this process (all devices). */
unsigned long long attn_kernel_launches(void);

/*
 * Self-test of the bounded-wait path (failure detection without a GPU fault):
 * launches one CTA that waits on an mbarrier nothing ever arrives on, for at
 * most `poll_limit` polls, then records ATTN_ERR_TIMEOUT in the device status
 * word and returns normally.  The caller then sees ATTN_ERR_TIMEOUT from
 * attn_check_device_status.  poll_limit must be in [1, 1<<20].
 */
attn_status_t attn_debug_wait_timeout(unsigned int poll_limit, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_ATTN_H_ */
