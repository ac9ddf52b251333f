/*
 * fa_gb300: fused, tiled self-attention forward (LLM prefill) for NVIDIA GB300 (sm_103a).
 *
 * C ABI. All entry points are plain C; pointers are device pointers unless stated.
 *
 * Operation (fa_forward). For every batch b, head h and query row i:
 *
 *   s_ij  = scale * sum_d Q[b,h,i,d] * K[b,h,j,d]        j in J(i)
 *   O[b,h,i,:] = sum_j exp(s_ij - max_j s_ij) V[b,h,j,:] / sum_j exp(s_ij - max_j s_ij)
 *   LSE[b,h,i] = ln sum_j exp(s_ij)
 *
 * with J(i) = {0..N-1}, or {0..i} when causal (top-left aligned: query i sees keys 0..i).
 * This is the attention forward pass S = QK^T, P = softmax(S), O = PV of "Android
 * Transformer Optimization: Attention and Mobile GPU Bottlenecks" (section "The
 * Self-Attention Bottleneck Is Memory Traffic, Not Compute"), with the scale applied to the
 * scores as the SGEMM alpha of "Flash Attention on Android: tiled SGEMM with RenderScript"
 * (section "Architecture: tiled attention with RenderScript BLAS"). It is computed with the
 * tiled loop and online softmax of the first page (sections "The Essence of FlashAttention:
 * Reordering the Computation" and "A Complete Tile Loop"): S is never written to memory.
 * The causal mask and the log-sum-exp output are not on the pages; they follow the usual
 * prefill conventions stated above.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O. Accumulation is always fp32. */
enum fa_dtype { FA_DTYPE_FP16 = 0, FA_DTYPE_BF16 = 1 };

/* Return codes. */
enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null pointer, B/H/N < 1, or O overlapping Q/K/V/LSE */
  FA_ERR_UNSUPPORTED = -2, /* D not 64 or 128, unknown dtype, or the device is not sm_103 */
  FA_ERR_ALIGN = -3,       /* Q/K/V/O not 16-byte aligned, or LSE not 4-byte aligned */
  FA_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed; see fa_last_cuda_error() */
  FA_ERR_TIMEOUT = -5,     /* a device-side wait exceeded the watchdog limit */
  FA_ERR_TOO_LARGE = -6    /* sizes exceed the 32-bit index ranges the kernel uses */
};

/*
 * fa_forward — attention forward pass.
 *
 *   q, k, v  [B, H, N, D] dense row-major (D contiguous, then N, then H, then B), element
 *            type `dtype`. Device memory, 16-byte aligned, read only.
 *   o        [B, H, N, D] same type and layout; written. Must not overlap q, k, v or lse.
 *   lse      [B, H, N] fp32, natural-log units of the scaled scores; written. May be NULL
 *            (then not written). 4-byte aligned.
 *   B, H, N  >= 1. Any N (no multiple-of-tile requirement). N <= 2^30 and B*H*ceil(N/256)
 *            < 2^31.
 *   D        64 or 128.
 *   scale    multiplies q.k before the softmax; scale <= 0, NaN or Inf selects 1/sqrt(D).
 *   causal   0: every query sees every key; nonzero: query i sees keys 0..i.
 *   dtype    FA_DTYPE_FP16 or FA_DTYPE_BF16.
 *   stream   a cudaStream_t (NULL = the legacy default stream) of the current device.
 *
 * Ownership: the caller owns every buffer; the call allocates no device memory. It is
 * asynchronous: it validates arguments on the host, encodes the tensor descriptors and
 * enqueues one kernel on `stream`, then returns. O and LSE are valid once the stream has
 * reached that point. Errors are returned before anything is enqueued, except FA_ERR_CUDA
 * for a failed launch and device-side timeouts, which fa_check_device_status() reports.
 * Thread-safe; one-time per-device setup runs on first use.
 */
FA_API int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
               float scale, int causal, int dtype, void* stream);

/* Static description of a return code. Never NULL. */
FA_API const char* fa_error_string(int code);

/* Library version as major*10000 + minor*100 + patch. */
FA_API int fa_version(void);

/*
 * Synchronises the current device, then returns FA_OK, or FA_ERR_TIMEOUT if any kernel of
 * this library on the current device gave up on a bounded wait since the last call (the
 * flag is cleared). FA_ERR_CUDA if the synchronisation itself fails.
 */
FA_API int fa_check_device_status(void);

/*
 * Sets the device-side wait limit, in nanoseconds, for launches that follow (process-wide).
 * 0 restores the default (2 s). Returns FA_OK.
 */
FA_API int fa_set_watchdog_ns(unsigned long long ns);

/*
 * Work decomposition for launches that follow (process-wide):
 *   FA_DECOMP_AUTO (0)      choose by problem size (default);
 *   FA_DECOMP_TWO_TILES (1) each work item is 256 query rows, two 128-row query tiles that
 *                           share every K/V tile (half the K/V traffic per query row);
 *   FA_DECOMP_SPLIT_KV (2)  each work item is one 128-row query tile whose K/V tiles are split
 *                           between the two softmax warpgroups and merged at the end (twice
 *                           the items, half the serial chain: for short or few sequences).
 * All three compute the same result (up to floating-point rounding order). Returns FA_OK or
 * FA_ERR_INVALID_ARG for an unknown value.
 */
enum fa_decomposition { FA_DECOMP_AUTO = 0, FA_DECOMP_TWO_TILES = 1, FA_DECOMP_SPLIT_KV = 2 };
FA_API int fa_set_decomposition(int mode);

/*
 * Test hook for failure detection (process-wide, for launches that follow): when `on` is
 * nonzero the MMA warp of every CTA first waits on a barrier that nothing arrives on, so the
 * device-side wait limit (fa_set_watchdog_ns) must run out; the kernel then records a
 * timeout, drains its in-flight copies and MMAs, frees tensor memory and returns. Outputs of
 * such launches are not valid. Returns FA_OK.
 */
FA_API int fa_debug_force_stall(int on);

/* The cudaError_t value behind the most recent FA_ERR_CUDA returned on this host thread. */
FA_API int fa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
