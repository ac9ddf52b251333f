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

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O, and of partial outputs. Accumulation is always fp32. For
 * FA_DTYPE_FP32 tensors fa_forward multiplies on the tensor cores in tf32 (the fp32-storage
 * variant of "Android Transformer Optimization: Attention and Mobile GPU Bottlenecks", section
 * "Pitfalls I Hit"): operands read from memory keep their top 19 bits (tf32: 8-bit exponent,
 * 10-bit mantissa), P is rounded to tf32, and the key tiles are 64 keys instead of 128. */
enum fa_dtype { FA_DTYPE_FP16 = 0, FA_DTYPE_BF16 = 1, FA_DTYPE_FP32 = 2 };

/* Return codes. */
enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1, /* null pointer, B/H/N < 1, or O overlapping Q/K/V/LSE */
  FA_ERR_UNSUPPORTED = -2, /* D not 64 or 128, a dtype the entry point does not take, or not sm_103 */
  FA_ERR_ALIGN = -3,       /* Q/K/V/O not 16-byte aligned, or LSE not 4-byte aligned */
  FA_ERR_CUDA = -4,        /* a CUDA runtime/driver call failed; see fa_last_cuda_error() */
  FA_ERR_TIMEOUT = -5,     /* a device-side wait exceeded the watchdog limit */
  FA_ERR_TOO_LARGE = -6,   /* sizes exceed the 32-bit index ranges the kernel uses */
  FA_ERR_WORKSPACE = -7,   /* split-KV workspace missing, misaligned or too small */
  FA_ERR_SCRATCH = -8,     /* split-KV partials larger than the built-in scratch (noalloc) */
  FA_ERR_LIBRARY = -9      /* naive baseline: cuBLAS could not be loaded or failed */
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
 *   dtype    FA_DTYPE_FP16, FA_DTYPE_BF16, or FA_DTYPE_FP32 (tf32 tensor-core products).
 *   stream   a cudaStream_t (NULL = the legacy default stream) of the current device.
 *
 * Ownership: the caller owns every buffer; the call allocates no device memory. It is
 * asynchronous: it validates arguments on the host, encodes the tensor descriptors and
 * enqueues one kernel on `stream`, then returns. O and LSE are valid once the stream has
 * reached that point. Errors are returned before anything is enqueued, except FA_ERR_CUDA
 * for a failed launch and device-side timeouts, which fa_check_device_status() reports.
 * Thread-safe; one-time per-device setup runs on first use. Causal problems with more than
 * two waves of work items run on a persistent grid from a per-shape work table. The first
 * call of such a shape builds the table on the host and copies it into the library's module
 * memory (a few KB, no allocation) with cudaMemcpyAsync on `stream`, then records an event;
 * until that event is seen complete, later calls of the shape on any stream first make their
 * stream wait on it. A call that would need the table while its stream is being captured (the
 * shape's first call, or one whose stream cannot wait yet) runs correctly without it, with one
 * CTA per work item; so does a call when the table pool (4 MB per device, kept for the life of
 * the process) is full. fa_schedule_pool_status reports both.
 *
 * Device addresses in module memory (status word, work tables, the no-alloc scratch) and the
 * per-thread launch parameters are cached for the life of the process: after
 * cudaDeviceReset, or any other destruction of the primary context, the library must not be
 * used again in the same process.
 */
FA_API int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int D,
               float scale, int causal, int dtype, void* stream);

/*
 * Split-KV forward and the merge of partial results.
 *
 * The keys of attention decompose: if the keys J(i) of row i are split into disjoint sets
 * K_1..K_S, the partial result of each set, (O_s, lse_s) = the same formulas as above with
 * j restricted to K_s, combines into the full result by the online-softmax update of
 * "Android Transformer Optimization: Attention and Mobile GPU Bottlenecks" (section "The
 * Essence of FlashAttention: Reordering the Computation") applied to whole sets:
 *
 *   m = max_s lse_s,   w_s = exp(lse_s - m),   O = sum_s w_s O_s / sum_s w_s,
 *   LSE = m + ln sum_s w_s,
 *
 * where a set with no key (lse_s = -inf) has weight 0 and its O_s is never read.
 *
 * fa_forward_splitkv computes the same O and LSE as fa_forward (arguments as there; dtype
 * FA_DTYPE_FP16 or FA_DTYPE_BF16 only), but
 * divides the 128-key tiles of every 128-row query tile into num_splits contiguous ranges
 * and processes each range as its own work item, so that one query tile can occupy several
 * SMs. That shortens the longest work items (the last query tiles of a causal sequence) and
 * fills the GPU when B*H*ceil(N/128) is small. Each item writes its partial result to
 * `workspace`; a second kernel, on the same stream, merges them into O and LSE.
 *
 *   num_splits       1..256, or 0 to choose automatically (fa_splitkv_num_splits). With 1
 *                    split this is fa_forward (the workspace is not used and may be NULL).
 *   workspace        device memory of at least fa_splitkv_workspace_bytes(B, H, N, D,
 *                    splits) bytes for the split count used, 256-byte aligned, not
 *                    overlapping any other argument; owned by the caller; its contents on
 *                    entry do not matter (nothing in it has to start at zero). Its layout is
 *                    partial O [splits, B*H, N, D] fp32, then, at the next 256-byte boundary,
 *                    partial lse [splits, B*H, N] fp32. Range s of the query tile qt (with
 *                    n = qt + 1 key tiles when causal, else ceil(N/128)) holds the key tiles
 *                    [s*n/splits, (s+1)*n/splits) (integer division); an empty range has lse
 *                    -inf and an unspecified O.
 *   workspace_bytes  its size in bytes.
 *
 * Two calls that share a workspace race unless the stream orders them. Returns FA_OK,
 * FA_ERR_WORKSPACE, or the codes of fa_forward (FA_ERR_INVALID_ARG also for num_splits
 * outside 0..256 or a workspace overlapping another argument).
 */
FA_API int fa_forward_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                              int D, float scale, int causal, int dtype, int num_splits, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * fa_forward_splitkv_noalloc — fa_forward_splitkv without a caller workspace and without any
 * allocation: the partial results go to a scratch array that is part of the library's device
 * code (a static __device__ array of 32 MiB = 33554432 bytes per device, 256-byte aligned).
 * This entry point is an engineering convenience; the pages have no counterpart to it.
 *
 *   arguments   as fa_forward_splitkv, minus workspace and workspace_bytes.
 *   limit       a given split count must need at most 32 MiB, i.e.
 *               fa_splitkv_workspace_bytes(B, H, N, D, splits) <= 33554432; otherwise
 *               FA_ERR_SCRATCH and nothing is enqueued. With num_splits 0 the count is
 *               fa_splitkv_num_splits's choice lowered, if needed, to the largest that fits
 *               (down to one split, which needs no scratch), so it never fails for size.
 *   zeroing     nothing in the scratch has to start at zero; every partial that the merge
 *               reads is written by the same call first.
 *   setup       the first call on a device does one-time setup (the device checks of
 *               fa_forward, then cudaGetSymbolAddress of the scratch with that device
 *               current); make that first call outside any stream capture.
 *   races       there is one scratch per device: two calls whose execution overlaps (on two
 *               streams, or from two threads) race on it and give wrong results. Calls
 *               ordered on one stream are fine.
 *
 * Allocates no memory (no cudaMalloc, cudaFree or allocating library call). Returns the codes
 * of fa_forward_splitkv except FA_ERR_WORKSPACE, plus FA_ERR_SCRATCH.
 */
FA_API int fa_forward_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                                      int N, int D, float scale, int causal, int dtype, int num_splits, void* stream);

/* Workspace bytes fa_forward_splitkv needs for `num_splits` (>= 1) splits; 0 for one split
 * or invalid arguments. Host only. */
FA_API size_t fa_splitkv_workspace_bytes(int B, int H, int N, int D, int num_splits);

/* The split count fa_forward_splitkv uses when given 0: a cost model of the whole job (item
 * lengths against the current device's SM count, plus the merge). >= 1, or a negative
 * fa_status. */
FA_API int fa_splitkv_num_splits(int B, int H, int N, int D, int causal);

/*
 * fa_merge_partials — combines num_parts partial results (formula above).
 *
 *   o_parts    [num_parts, B, H, N, D] of parts_dtype (FA_DTYPE_FP16, _BF16 or _FP32),
 *              16-byte aligned; read only.
 *   lse_parts  [num_parts, B, H, N] fp32 (-inf: the part has no key for that row); read only.
 *   o          [B, H, N, D] of dtype (FA_DTYPE_FP16 or _BF16), 16-byte aligned; written. Rows
 *              without a key in any part get 0.
 *   lse        [B, H, N] fp32 (-inf for rows without a key) or NULL.
 *   D          64 or 128.
 *
 * Asynchronous on `stream`, allocates nothing. Outputs must not overlap inputs. Returns
 * FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_ALIGN, FA_ERR_TOO_LARGE or
 * FA_ERR_CUDA.
 */
FA_API int fa_merge_partials(const void* o_parts, const float* lse_parts, int num_parts, int parts_dtype, void* o,
                             float* lse, int B, int H, int N, int D, int dtype, void* stream);

/*
 * fa_naive_forward — the unfused baseline: the same O and LSE computed the way the pages'
 * "naive" attention does it ("Android Transformer Optimization: Attention and Mobile GPU
 * Bottlenecks", section "The Self-Attention Bottleneck Is Memory Traffic, Not Compute"), with
 * the whole score matrix in memory: S = scale Q K^T by a batched library GEMM (cuBLAS, the
 * scale as alpha, as the SGEMM of "Flash Attention on Android: tiled SGEMM with
 * RenderScript"), a row softmax kernel that writes P over S (and LSE), and O = P V by a second
 * batched GEMM. It exists to measure what the fused kernel saves; it is not a fast path.
 *
 *   arguments  as fa_forward; dtype must be FA_DTYPE_FP16 (S and P are stored in fp16, as
 *              in the pages' size claims).
 *   workspace  caller-owned device memory of at least fa_naive_workspace_bytes(B, H, N) bytes
 *              (S and then P, [B*H, N, N] fp16), 256-byte aligned, not overlapping any other
 *              argument; its contents on entry do not matter.
 *
 * cuBLAS (libcublas.so.13) is loaded on first use; FA_ERR_LIBRARY if it cannot be loaded or
 * a GEMM fails (fa_naive_last_library_error gives the cublasStatus_t). The first call on each
 * host thread creates a cuBLAS handle (which allocates). Enqueues three kernels or more (the
 * library picks its GEMM kernels) on `stream`.
 */
FA_API int fa_naive_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
                            int D, float scale, int causal, int dtype, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Bytes of S/P the naive baseline needs: 2 * B * H * N * N rounded up to 256; 0 if invalid. */
FA_API size_t fa_naive_workspace_bytes(int B, int H, int N);

/* The cublasStatus_t behind the most recent FA_ERR_LIBRARY on this host thread. */
FA_API int fa_naive_last_library_error(void);

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
 *                           A causal launch at D = 64 with between one and two such items
 *                           per SM runs them in pairs: each CTA takes a long and a short query
 *                           tile at once and divides their K/V tiles evenly between the
 *                           warpgroups;
 *   FA_DECOMP_SPLIT_KV_SERIAL (3)  the same items, never paired (one after another).
 * All four compute the same result (up to floating-point rounding order). Returns FA_OK or
 * FA_ERR_INVALID_ARG for an unknown value.
 */
enum fa_decomposition {
  FA_DECOMP_AUTO = 0,
  FA_DECOMP_TWO_TILES = 1,
  FA_DECOMP_SPLIT_KV = 2,
  FA_DECOMP_SPLIT_KV_SERIAL = 3
};
FA_API int fa_set_decomposition(int mode);

/*
 * Test hook for failure detection (process-wide, for launches that follow): when `on` is
 * nonzero the MMA warp of every CTA first waits on a barrier that nothing arrives on, so the
 * device-side wait limit (fa_set_watchdog_ns) must run out; the kernel then records a
 * timeout, drains its in-flight copies and MMAs, frees tensor memory and returns. Outputs of
 * such launches are not valid. Returns FA_OK.
 */
FA_API int fa_debug_force_stall(int on);

/*
 * Inspection hook for the work schedule (host only, no CUDA call): causal problems with more
 * than two waves of work items run on a persistent grid of num_sms CTAs whose item lists
 * reproduce one-CTA-per-item hardware dispatch in the item order (each item goes to the CTA
 * that frees up first under an estimated cost). This returns the lists fa_forward would use
 * for this shape on a GPU with num_sms SMs, with the current fa_set_decomposition mode:
 * out[0 .. num_sms] are offsets, and CTA c processes the items out[num_sms + 1 + i] for i in
 * [out[c], out[c + 1]), in that order. Items are numbered in the kernel's order (per head
 * section, row blocks longest first). Returns the number of ints (num_sms + 1 + items),
 * 0 when the shape uses no schedule (the items are then strided over the CTAs), the same
 * count without writing when out is NULL, FA_ERR_INVALID_ARG for bad sizes or when capacity
 * is too small, FA_ERR_UNSUPPORTED for D or dtype, FA_ERR_TOO_LARGE past the item limit.
 */
FA_API int fa_debug_work_schedule(int B, int H, int N, int D, int causal, int dtype, int num_sms, int* out,
                                  int capacity);

/*
 * Inspection hook for the work decomposition (host only, no CUDA call) of a fa_forward of
 * this shape on a GPU with num_sms SMs, with the current fa_set_decomposition mode.
 * plan[0..4] (required) receive: the number of work items; 1 if an item is one 128-row
 * query tile (else two); 1 if the launch is paired; 1 if it follows a dispatch-order
 * schedule (fa_debug_work_schedule); the grid size (with a schedule: num_sms). A paired
 * launch is causal, fp16 or bf16 at D = 64, with single-query-tile items, more than num_sms
 * and at most 2 num_sms of them: CTA c of a grid of G runs items c and 2 G - 1 - c at once.
 * For a paired launch,
 * units (when not NULL) receives 6 ints per CTA: item a (the one with more K/V tiles), item
 * b (-1 when the CTA has one item), the K/V tiles of a and of b, and the tiles warpgroup 0
 * and warpgroup 1 process (warpgroup 0 takes a's first ones; warpgroup 1 all of b, then the
 * rest of a). Returns the number of unit ints (6 G; 0 when not paired), the same count
 * without writing when units is NULL, FA_ERR_INVALID_ARG for bad sizes, a NULL plan or a
 * too small capacity, FA_ERR_UNSUPPORTED for D or dtype, FA_ERR_TOO_LARGE past the item
 * limit.
 */
FA_API int fa_debug_work_plan(int B, int H, int N, int D, int causal, int dtype, int num_sms, int* plan, int* units,
                              int capacity);

/*
 * Inspection hook for the split count (host only, no CUDA call) on a GPU with num_sms SMs:
 * the count fa_splitkv_num_splits gives for this shape (for_noalloc 0), or the count
 * fa_forward_splitkv_noalloc runs with num_splits 0 (for_noalloc 1: that count lowered to the
 * largest whose partials fit the 32 MiB scratch, down to 1). Returns the count (>= 1),
 * FA_ERR_INVALID_ARG for bad sizes or num_sms < 1, FA_ERR_UNSUPPORTED for D.
 */
FA_API int fa_debug_num_splits(int B, int H, int N, int D, int causal, int num_sms, int for_noalloc);

/*
 * The per-device pool of work tables that causal multi-wave launches use (fa_forward). Host
 * only; the one CUDA call is cudaGetDevice (for used_bytes).
 *   used_bytes, capacity_bytes  (either may be NULL) bytes of the current device's 4 MB pool
 *                               in use and in total;
 *   fallbacks                   (may be NULL) launches in this process, on any device, that
 *                               needed a table but ran without one (one CTA per work item:
 *                               the same result, slower): the pool was full, or the stream
 *                               was being captured before the table's copy was known complete.
 * Returns FA_OK or FA_ERR_CUDA.
 */
FA_API int fa_schedule_pool_status(size_t* used_bytes, size_t* capacity_bytes, unsigned long long* fallbacks);

/* The cudaError_t value behind the most recent FA_ERR_CUDA returned on this host thread. */
FA_API int fa_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
