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
 * thread-safe.  No call allocates device memory: scratch memory, where a path
 * needs some, is passed in by the caller.  The library's own device state is
 * static: a 4-byte status word and the 40 MiB scratch array of
 * attn_fwd_splitkv_noalloc, which every GPU that loads the library holds until
 * the process exits (one copy per GPU), whether or not that entry point is
 * ever called.
 */
#ifndef LIBATTN_ATTN_H_
#define LIBATTN_ATTN_H_

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment, scale or flag; nothing launched */
    ATTN_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (head size)  */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or the kernel launch failed       */
    ATTN_ERR_TIMEOUT = 4      /* a device-side bounded wait ran out (see attn_last_device_status) */
} attn_status_t;

/*
 * attn_fwd -- O = softmax(scale * Q K^T [+ mask]) V and LSE, asynchronously on `stream`.
 *
 * q    device pointer, bf16, [B, Sq, Hq, D], D contiguous (row stride Hq*D elements)
 * k, v device pointers, bf16, [B, Skv, Hkv, D]
 * o    device pointer, bf16, [B, Sq, Hq, D]   (written; round-to-nearest-even of O)
 * lse  device pointer, fp32, [B, Hq, Sq], or NULL to skip it
 * B, Sq, Skv, Hq, Hkv, D  sizes; every one >= 1, Hq a multiple of Hkv, D 64, 128 or 256
 *      (other head sizes: ATTN_ERR_UNSUPPORTED).
 *      Sq and Skv may be any length (ragged tails are handled in the kernel).
 * causal 0: every key visible.  1: key j visible from query i iff
 *      j <= i + (Skv - Sq) (bottom-right aligned, as in chunked prefill).
 *      2: iff j <= i (top-left aligned, the Pallas page's reference mask).
 *      1 and 2 coincide when Sq == Skv.  A query row that sees no key gets
 *      O = 0 and LSE = -inf.
 * scale  finite, > 0 (typically 1/sqrt(D)).
 * stream CUDA stream the kernel runs on (0 = legacy default stream).
 *
 * Ownership: the caller owns every buffer; nothing is retained after return.
 * q, k, v, o must be 16-byte aligned (TMA).  o must not alias q, k or v.
 * Returns ATTN_OK once the kernel is enqueued; a device-side wait that runs out
 * is reported later through attn_last_device_status.  On any error return,
 * nothing was launched and no output was written.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Sq, int Skv, int Hq, int Hkv, int D, int causal, float scale,
                       cudaStream_t stream);

/* Element type of q, k, v and o for attn_fwd_ex. */
typedef enum {
    ATTN_DTYPE_BF16 = 0, /* bfloat16 (what attn_fwd takes) */
    ATTN_DTYPE_F16 = 1   /* IEEE binary16 */
} attn_dtype_t;

/*
 * attn_fwd_ex -- attn_fwd with a choice of 16-bit element type for q, k, v and
 * o (the Pallas page's forward accepts float16 and bfloat16 alike).  `dtype`
 * is an attn_dtype_t; anything else returns ATTN_ERR_INVALID_ARG.  P is rounded
 * to the same type before the P.V product; accumulation, softmax and LSE stay
 * fp32; O is rounded to nearest-even in that type.  Everything else, including
 * errors, as attn_fwd.
 */
attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Sq, int Skv, int Hq, int Hkv, int D, int causal, float scale,
                          int dtype, cudaStream_t stream);

/*
 * Split-KV forward for problems with too few query tiles to fill the GPU
 * (short query blocks against long key ranges, e.g. chunked prefill).  The
 * same operation and arguments as attn_fwd (bf16), plus a device workspace the
 * caller allocates.  This is the single-GPU form of the kernbench page's group
 * sequence parallelism (`_gqa_attention_prefill_short.py`): the iterations over
 * (query tile pair, KV tile) are cut into equal contiguous shares, one per SM; a
 * tile pair whose KV range straddles shares is computed in pieces whose partial
 * (m, l, O) are merged by that page's `_merge_running` rule in a second kernel.
 *
 * attn_fwd_splitkv_workspace_size: bytes of workspace attn_fwd_splitkv needs
 *   for this problem on the current device (it depends on the SM count); 0 when
 *   no split pays off, and then attn_fwd_splitkv runs exactly what attn_fwd runs.
 *   A split is chosen only when the whole-unit schedule's busiest SM would run at
 *   least 1.35x the KV iterations of an equal share (plus 4): the crossover
 *   measured on GB300 (decode rows and short prefill chunks against long key
 *   ranges split and run several times faster; shapes that already fill the GPU
 *   do not).  This is the entry point to call when scratch can be supplied.
 * attn_fwd_splitkv: workspace device pointer (256-byte aligned, not aliasing
 *   any other argument) of at least that many bytes, or NULL when the size is 0.
 *   The workspace is scratch: its contents are undefined before and after the
 *   call, and two calls that overlap in time on the GPU must not share one.
 *   Errors as attn_fwd; ATTN_ERR_INVALID_ARG also for a missing or short workspace.
 */
attn_status_t attn_fwd_splitkv_workspace_size(int B, int Sq, int Skv, int Hq, int Hkv, int D,
                                              int causal, size_t* bytes);
attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int Sq, int Skv, int Hq, int Hkv, int D, int causal,
                               float scale, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * attn_fwd_splitkv_noalloc -- attn_fwd_splitkv for callers that cannot
 * allocate device memory where they call attention: code whose device memory
 * all belongs to another allocator (a framework's caching pool, a fixed arena
 * reserved at start-up) or that runs where allocation is not allowed once
 * serving has begun.  The pages have no counterpart of this entry point.
 *
 * Same arguments, semantics and errors as attn_fwd_splitkv, without the
 * workspace: the split-KV scratch is a static 40 MiB device array inside
 * libattn, which every GPU that loads the library holds until the process
 * exits.  The call allocates nothing, on the device or on the host.
 *   - The first call on a device looks up that array's device address (once per
 *     device, with the device current); make that first call before any stream
 *     capture begins.
 *   - Problems whose scratch would exceed 40 MiB return ATTN_ERR_UNSUPPORTED
 *     (on a 152-SM GPU the split plan never needs more than about 38.4 MiB).
 *   - Each GPU has its own copy of the array; every call on one GPU shares that
 *     copy, which keeps the last call's contents.  Nothing in it needs to start
 *     at zero (each call writes every partial slot before it reads it).  Calls
 *     that overlap in time on the same GPU (for example on different streams)
 *     race on it and must be serialised; calls on different GPUs do not share
 *     scratch.
 */
attn_status_t attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int Sq, int Skv, int Hq, int Hkv, int D,
                                       int causal, float scale, cudaStream_t stream);

/*
 * attn_bwd -- gradients of the attention forward: given dO, the gradient of
 * L = sum dO * O, with O = softmax(scale * Q K^T [+ mask]) V as in attn_fwd
 * (the Pallas page, attention_mgpu.py, `_attention_bwd`):
 *   P = exp(scale * Q K^T - LSE) (masked pairs 0), delta = rowsum(O * dO),
 *   dP = dO V^T, dS = P * (dP - delta),
 *   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO,
 * with dK and dV summed over the query heads that share a key/value head.
 *
 * q, k, v   device pointers, the forward's inputs (layouts as attn_fwd).
 * o         device pointer, [B, Sq, Hq, D]: the forward's output.
 * lse       device pointer, fp32 [B, Hq, Sq]: the forward's natural-log LSE
 *           (-inf for rows that see no key).
 * dO        device pointer, [B, Sq, Hq, D]: gradient of the output.
 * dq        device pointer, [B, Sq, Hq, D]     (written)
 * dk, dv    device pointers, [B, Skv, Hkv, D]  (written; every element, zero for
 *           keys no query row sees)
 * B .. scale  as attn_fwd (the same causal mode and scale as the forward call;
 *           the page's backward has no mask, this one applies the forward's);
 *           D 64, 128 or 256; B <= 65535.
 * dtype     ATTN_DTYPE_BF16 or ATTN_DTYPE_F16: the element type of q, k, v, o,
 *           dO, dq, dk and dv.
 * workspace device pointer, 256-byte aligned, of at least
 *           attn_bwd_workspace_size bytes (per-row delta and base-2 LSE);
 *           scratch, contents undefined before and after the call.
 *
 * Arithmetic: operands and P, dS in the element type, fp32 accumulation in
 * tensor memory, fp32 delta; outputs rounded to nearest even once.
 * Ownership: the caller owns every buffer.  q, k, v, o, dO, dq, dk, dv must be
 * 16-byte aligned; lse 4-byte aligned.  dq, dk, dv and the workspace must not
 * overlap any input or each other.  Three kernels are enqueued on `stream`
 * (prep, dK/dV, dQ), four at D = 256 (prep, dV, dK, dQ); errors are reported
 * as for attn_fwd (nothing is launched on any error return; a device-side
 * timeout shows in attn_last_device_status).
 */
attn_status_t attn_bwd_workspace_size(int B, int Sq, int Skv, int Hq, int Hkv, int D, size_t* bytes);
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dO, void* dq, void* dk, void* dv, int B, int Sq, int Skv, int Hq,
                       int Hkv, int D, int causal, float scale, int dtype, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);

/* Static, human-readable name of a status code (never NULL). */
const char* attn_status_str(attn_status_t status);

/*
 * attn_last_device_status -- the device-side outcome of the calls made so far.
 * Every libattn kernel records a bounded wait that ran out in one status word
 * per device (the Pallas page's host boundary returns errors only at call
 * time; this word carries the ones found later, on the GPU).  Waits until all
 * work submitted to the current device has completed (cudaDeviceSynchronize),
 * then reads and clears that device's word.  Returns ATTN_ERR_TIMEOUT if any
 * libattn kernel on the current device gave up a bounded wait since the word
 * was last read (that call's outputs are then invalid), ATTN_ERR_CUDA if
 * synchronisation or the read failed, else ATTN_OK.  The word is per device,
 * not per calling thread: a timeout is reported once, to whichever caller
 * reads it first.
 */
attn_status_t attn_last_device_status(void);

/*
 * attn_check_device_status -- attn_last_device_status that waits only for
 * `stream` (cudaStreamSynchronize) instead of the whole device, for callers
 * whose libattn work all ran on that stream.  Same word, same return values.
 */
attn_status_t attn_check_device_status(cudaStream_t stream);

/* Number of kernels libattn has enqueued in this process (all devices). */
unsigned long long attn_kernel_launches(void);

/*
 * Self-test of the bounded-wait path (failure detection without a GPU fault):
 * launches one CTA that waits on an mbarrier nothing ever arrives on, for at
 * most `poll_limit` polls, then records ATTN_ERR_TIMEOUT in the device status
 * word and returns normally.  The caller then sees ATTN_ERR_TIMEOUT from
 * attn_last_device_status.  poll_limit must be in [1, 1<<20].
 */
attn_status_t attn_debug_wait_timeout(unsigned int poll_limit, cudaStream_t stream);

/*
 * Measured issue rates of the units the attention loop leans on (diagnostic;
 * no page defines it: it checks the design's assumption that the forward's
 * 16384 exponentials per 128x128 tile fit under its 2 x 8 tensor-core products,
 * so that no exponential has to move to the FMA pipe).  Runs one CTA per SM of
 * the current device on `stream` and synchronises it.  out (host, n >=
 * ATTN_UNIT_RATES doubles) receives:
 *   out[0..4]  SM clock cycles per tcgen05.mma kind::f16 with M = 128, K = 16,
 *              bf16 operands, fp32 accumulator, issued back to back by one
 *              thread: [0] both operands in shared memory, N = 128; [1] A in
 *              tensor memory, N = 128; [2] shared memory, N = 256; [3] shared
 *              memory, N = 64; [4] A in tensor memory, N = 64
 *   out[5]     cycles per warp-wide ex2.approx.ftz.f32 on one SM sub-partition
 *              (two warps of independent exponentials per sub-partition)
 *   out[6]     exponentials per cycle per SM (= 4 x 32 / out[5])
 *   out[7]     number of SMs measured
 * Returns ATTN_ERR_INVALID_ARG for a NULL `out` or n < ATTN_UNIT_RATES (nothing
 * is launched), ATTN_ERR_CUDA on a launch or copy failure, ATTN_ERR_TIMEOUT if
 * the MMA completion wait ran out or if an earlier libattn kernel on this device
 * had already recorded a timeout (that earlier timeout is reported here, not
 * lost: the status word is read and cleared before the first rate kernel and
 * again after the last, as attn_check_device_status(stream) does), else ATTN_OK.
 */
#define ATTN_UNIT_RATES 8
attn_status_t attn_debug_unit_rates(double* out, int n, cudaStream_t stream);

/*
 * The forward's unit schedule for a shape (diagnostic; host only, launches
 * nothing).  attn_fwd runs two 128-row query tiles per work unit on a
 * persistent grid of min(#units, sms) CTAs.  For causal shapes of head size
 * 128 with at most 2048 units it takes the units from a table: the units in
 * blocks of heads whose K and V together take at most 48 MB, longest first
 * within a block, each unit handed to the least-loaded CTA.  Otherwise each
 * CTA takes units in a snake order and no table exists.
 *   sms          number of SMs to plan for, in [1, 256]
 *   cta_begin    (host, >= grid + 1 ints, grid = min(#units, sms)) receives
 *                the table's per-CTA start offsets into `units`
 *   units        (host, `cap` ints) receives the unit indices, CTA after CTA,
 *                each CTA's in the order it takes them
 *   n_units_out  receives the number of units in the table, or 0 when the
 *                snake order is used (cta_begin and units are then untouched)
 * Returns ATTN_ERR_INVALID_ARG for invalid sizes, sms out of range, a NULL
 * pointer, or a `cap` smaller than the table; ATTN_ERR_UNSUPPORTED for a head
 * size other than 64, 128 or 256; else ATTN_OK.
 */
attn_status_t attn_debug_unit_schedule(int B, int Sq, int Skv, int Hq, int Hkv, int D, int causal, int sms,
                                       int* cta_begin, int* units, int cap, int* n_units_out);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_ATTN_H_ */
