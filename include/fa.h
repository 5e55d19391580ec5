/*
 * fa.h -- C ABI of libfa.so: exact, IO-aware tiled attention on GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [EXPL] "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *          IO-Awareness" (paper explainer page).
 *   [MATH] "Mathematical Properties Behind FlashAttention - Streaming
 *          Transformations for Memory-Efficient Computation" (blog).
 *
 * Conventions shared by every entry point
 *   - Tensors Q, K, V, O, dO, dQ, dK, dV are bf16 (stored as 16-bit words),
 *     contiguous row-major [B, H, N, d]; lse is float32 [B, H, N].  The
 *     pages fix no layout; this one keeps each head's N x d matrix
 *     contiguous, so one (b, h) is a plain N x d operand of [EXPL] "Method".
 *   - All tensor pointers are DEVICE pointers owned by the caller, and must be
 *     16-byte aligned (TMA requirement).  The library never frees them.
 *   - d is 64 or 128 (separate kernels for each).  N >= 1, B >= 1, H >= 1,
 *     B*H*N < 2^31.
 *   - scale multiplies Q K^T (S = scale * Q K^T); it must be finite and > 0.
 *   - causal != 0 keeps key j for query i iff j <= i (top-left aligned).
 *   - kv_len: NULL, or a DEVICE int32 array [B]; keys j >= kv_len[b] of batch b
 *     are masked (values are clamped to [0, N]).  Query rows are never masked.
 *   - block_mask: NULL, or a DEVICE uint8 array [nb * nb], nb = ceil(N / 128),
 *     row-major; entry (I, J) = 0 removes the 128 x 128 block of query tile I
 *     and key tile J for every (b, h) ([EXPL] "Extension: Block-Sparse
 *     FlashAttention": a fixed mask over N/B_r x N/B_c blocks; here
 *     B_r = B_c = 128).
 *   - Masks combine by AND.  A query row with no allowed key gets O = 0,
 *     lse = -inf, dQ = 0, and adds nothing to dK, dV.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call is asynchronous on it; outputs are fully overwritten, never
 *     accumulated.
 *   - The library's kernels let the next kernel on the stream begin
 *     launching while they finish (programmatic dependent launch); each reads
 *     its inputs only once the previous kernel has completed.  The one
 *     exception is fa_bwd's workspace (see there).
 *   - fa_fwd and fa_bwd may be captured into a CUDA graph on `stream` and the
 *     graph replayed (each replay resets the backward's counters in its
 *     workspace); make one call on the shapes outside the capture first,
 *     which configures the kernels.
 *   - Every argument is validated before anything is launched; a failed call
 *     launches nothing.  There is no CPU fallback and no other backend.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1,  /* null pointer, bad size, non-finite or non-positive scale */
    FA_ERR_UNSUPPORTED = -2,  /* d not 64 or 128, N > 65535 * 128, N > 1024 * 128 with
                                 a block mask, N > 131072 with dropout, or no sm_103
                                 device */
    FA_ERR_MISALIGNED = -3,   /* a tensor pointer is not 16-byte aligned */
    FA_ERR_CUDA = -4,         /* a CUDA runtime / driver call failed */
    FA_ERR_TIMEOUT = -5,      /* a kernel's bounded wait ran out (reported by fa_check) */
    FA_ERR_WORKSPACE = -6     /* workspace NULL, misaligned or smaller than required */
} fa_status;

/*
 * Forward pass ([EXPL] "Method", online softmax tracking and steps 1-4;
 * [MATH] section 7).  For each query tile the kernel streams the allowed
 * key/value tiles, computes S_ij = scale * Q_i K_j^T on chip, keeps the
 * running row maximum m and exponential sum l, rescales the partial output
 * and accumulates P~_ij V_j.  Only O and the per-row statistic are written
 * ([EXPL] "Key ideas": O plus (l, m) are kept, O(N) extra memory).
 *   q, k, v  in : bf16 [B, H, N, d]
 *   o        out: bf16 [B, H, N, d], O = softmax(scale Q K^T, masked) V
 *   lse      out: fp32 [B, H, N], lse_i = m_i + ln(l_i) (natural log; the pages'
 *                 (m, l) pair folded into one number)
 * Returns FA_OK once the kernel is enqueued.
 */
FA_API fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int H, int N, int d, float scale, int causal,
                 const int32_t *kv_len, const uint8_t *block_mask, void *stream);

/*
 * Bytes of device workspace fa_bwd needs for this shape: per (b, h) and
 * query row (padded to a multiple of 128) one fp32 D_i = <dO_i, O_i>, one
 * fp32 base-2 log-sum-exp, and d fp32 dQ accumulators; O(N) per head
 * ([EXPL] "Complexity analysis": O(N) extra memory).  Plus, for the
 * block-sparse schedule, one int32 count, up to nt int16 query-tile indices
 * and one int16 place in the longest-first order per key tile (nt =
 * ceil(N / 128), capped at 1024), and one int32 work counter.  Returns 0 for
 * invalid sizes.
 */
FA_API size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass by recomputation ([EXPL] "Key ideas", recomputation; [MATH]
 * section 5): S and P are rebuilt tile by tile from Q, K, V and lse; the
 * N x N matrices are never stored.  Gradient of L = <dO, O> for
 * O = softmax(scale Q K^T) V:
 *     dV = P^T dO, dP = dO V^T, D = rowsum(dO o O), dS = P o (dP - D),
 *     dQ = scale dS K, dK = scale dS^T Q.
 *   q, k, v, o, dO in : bf16 [B, H, N, d]; o is fa_fwd's output for the same
 *                       inputs and masks
 *   lse            in : fp32 [B, H, N], fa_fwd's output
 *   dq, dk, dv     out: bf16 [B, H, N, d]
 *   workspace      in : device scratch of >= fa_bwd_workspace_size() bytes,
 *                       16-byte aligned, owned by the caller; its contents
 *                       on entry do not matter and are garbage on return.
 *                       For d = 128, or N <= 2048, and no block mask,
 *                       fa_bwd starts zeroing part of it while the previous
 *                       kernel on the stream, if it is one of this
 *                       library's, may still be running: the workspace must
 *                       not share memory with
 *                       anything that call's kernels read or write (a
 *                       buffer released to a stream-ordered allocator after
 *                       that call and handed back as the workspace does).
 *                       Successive fa_bwd calls may share one workspace.
 * Masks and scale must be the ones given to fa_fwd.
 */
FA_API fa_status fa_bwd(const void *q, const void *k, const void *v, const void *o,
                 const float *lse, const void *dout, void *dq, void *dk, void *dv,
                 int B, int H, int N, int d, float scale, int causal,
                 const int32_t *kv_len, const uint8_t *block_mask,
                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Attention dropout fused into both passes ([EXPL] "Key ideas", kernel fusion:
 * matmul, masking, softmax and dropout in one kernel).  With P the masked
 * softmax of fa_fwd and Z a keep mask,
 *     O = (P o Z / (1 - p')) V,      lse as in fa_fwd (from P, before dropout),
 * and the backward is the gradient of that O for the same Z:
 *     dV = (P o Z)^T dO / (1 - p'),  dP~ = dO V^T,  D = rowsum(dO o O),
 *     dS = P o (Z o dP~ / (1 - p') - D),  dQ = scale dS K,  dK = scale dS^T Q.
 * Z is regenerated from (seed, b*H + h, i, j) in both passes, never stored:
 *     pcg(x):  s = x * 747796405 + 2891336453;
 *              w = ((s >> ((s >> 28) + 4)) ^ s) * 277803737;  return (w >> 22) ^ w
 *              (the 32-bit "PCG hash", Jarzynski and Olano, "Hash Functions for
 *              GPU Rendering", JCGT 9(3), 2020; all arithmetic mod 2^32)
 *     kb    = pcg(pcg(pcg(seed_lo) ^ seed_hi) ^ (b*H + h))
 *     r     = pcg(kb ^ ((i >> 1) << 16 | (j >> 1)))     (one word per 2x2 block)
 *     u     = byte ((i & 1) * 2 + (j & 1)) of r (byte 0 = least significant)
 *     Z_ij  = (u >= p8),  p8 = p * 256 rounded to nearest (ties to even), at most
 *             255,  p' = p8 / 256.
 *   p       in : drop probability in [0, 1); p8 = 0 gives exactly fa_fwd / fa_bwd.
 *   seed    in : 64-bit seed (seed_lo = low 32 bits, seed_hi = high 32 bits).
 * Other arguments, layouts and errors as fa_fwd / fa_bwd; FA_ERR_INVALID_ARG for
 * p outside [0, 1) or non-finite, FA_ERR_UNSUPPORTED for p8 > 0 with
 * N > 131072 (i >> 1 and j >> 1 must fit 16 bits).  fa_bwd_dropout must get the
 * p, seed, masks and scale given to fa_fwd_dropout and its outputs.
 */
FA_API fa_status fa_fwd_dropout(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int H, int N, int d, float scale, int causal,
                                const int32_t *kv_len, const uint8_t *block_mask, float p,
                                unsigned long long seed, void *stream);

FA_API fa_status fa_bwd_dropout(const void *q, const void *k, const void *v, const void *o,
                                const float *lse, const void *dout, void *dq, void *dk,
                                void *dv, int B, int H, int N, int d, float scale, int causal,
                                const int32_t *kv_len, const uint8_t *block_mask, float p,
                                unsigned long long seed, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Split-KV forward for a short query block against a long key/value cache
 * (decoding).  The key tiles of every row are cut into num_splits contiguous
 * ranges processed by separate CTAs; each range leaves its own normalised
 * partial output O_s and lse_s (the online-softmax state of [EXPL] "Method",
 * steps 2-4, over that range), and a merge kernel combines them exactly:
 *     lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s
 * ([MATH] section 4: the softmax-weighted sum splits into independent key
 * ranges whose states combine by rescaling).  The result is the fa_fwd
 * result with Nq query rows and Nk key rows, no causal mask and no block
 * mask (kv_len as in fa_fwd, clamped to [0, Nk]).  d = 64 or 128.
 *   q              in : bf16 [B, H, Nq, d]
 *   k, v           in : bf16 [B, H, Nk, d]
 *   o              out: bf16 [B, H, Nq, d]
 *   lse            out: fp32 [B, H, Nq]
 *   num_splits     in : 0 = about two CTAs per SM of a 152-SM GB300, else the
 *                       count (at most 1024); capped at ceil(Nk / 128)
 *   workspace      in : device scratch of >= fa_fwd_splitkv_workspace_size()
 *                       bytes (same num_splits), 16-byte aligned, caller-owned:
 *                       fp32 partial outputs and lse, S * B * H * ceil(Nq/128)
 *                       * 128 * (4 d + 4) bytes, each part rounded up to 256.
 */
FA_API size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int Nk, int d, int num_splits);

FA_API fa_status fa_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                                int B, int H, int Nq, int Nk, int d, float scale,
                                const int32_t *kv_len, int num_splits, void *workspace,
                                size_t workspace_bytes, void *stream);

/*
 * Host-buffer entry points: the forward (fa_fwd_host) or the forward and the
 * backward (fa_fwd_bwd_host) of the tensors above held in HOST memory.  Every
 * (b, h) is an independent N x d problem ([EXPL] "Method"), so the heads are
 * cut into contiguous groups and the host-to-device copies of one group, the
 * kernels of the previous one and the device-to-host copies of the one before
 * overlap on the GPU (two copy streams of the library plus `stream`, joined
 * by events).  Each group runs fa_fwd (and fa_bwd) on its heads, so the
 * results are those entry points' results for the same inputs.
 *   q, k, v, dout  in : HOST bf16 [B, H, N, d]; page-locked (pinned) memory
 *                       is needed for the copies to overlap anything
 *   o              out: HOST bf16 [B, H, N, d]
 *   lse            out: HOST fp32 [B, H, N]
 *   dq, dk, dv     out: HOST bf16 [B, H, N, d] (fa_fwd_bwd_host only)
 *   kv_len         in : NULL or HOST int32 [B]
 *   block_mask     in : NULL or HOST uint8 [nb * nb], as in fa_fwd
 *   n_chunks       in : head groups; 0 = about 256 query tiles per group,
 *                       2 to 8 groups; at most 64; capped at B * H
 *   arena          in : DEVICE scratch of >= fa_host_arena_size() bytes,
 *                       256-byte aligned, caller-owned: device copies of the
 *                       tensors, the backward's workspace and small slack
 *   stream         in : the kernels run on it, and it completes only after the
 *                       last copy back: synchronise it (or fa_check) before
 *                       reading the outputs or reusing the inputs
 * No dropout: the keep mask depends on the head's index in the whole problem;
 * use fa_fwd_dropout / fa_bwd_dropout on device tensors.  Errors: fa_fwd's
 * and fa_bwd's codes for the same arguments; FA_ERR_WORKSPACE for a missing,
 * misaligned or short arena; FA_ERR_INVALID_ARG for n_chunks outside
 * [0, 64]; FA_ERR_CUDA when a copy or a stream / event call fails.  Every
 * argument is checked before anything is enqueued; a CUDA failure part-way
 * leaves the groups enqueued before it running, so after FA_ERR_CUDA the
 * outputs are undefined until the device has been synchronised.  The
 * library cannot tell host from device pointers here: pass host memory.
 * Calls on one device share
 * the copy streams: they are enqueued one at a time and their copies run in
 * call order.
 */
FA_API size_t fa_host_arena_size(int B, int H, int N, int d);

FA_API fa_status fa_fwd_host(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int N, int d, float scale, int causal,
                             const int32_t *kv_len, const uint8_t *block_mask, int n_chunks,
                             void *arena, size_t arena_bytes, void *stream);

FA_API fa_status fa_fwd_bwd_host(const void *q, const void *k, const void *v, const void *dout,
                                 void *o, float *lse, void *dq, void *dk, void *dv, int B, int H,
                                 int N, int d, float scale, int causal, const int32_t *kv_len,
                                 const uint8_t *block_mask, int n_chunks, void *arena,
                                 size_t arena_bytes, void *stream);

/*
 * fa_bwd without a workspace argument, for callers that cannot allocate
 * device memory when they run the backward pass (for instance a plugin whose
 * host application owns every device allocation, or a latency-critical loop
 * that must not allocate).  The paper has no counterpart: this is a
 * deployment variant of fa_bwd with identical arguments, results and status
 * codes apart from the workspace (it runs fa_bwd's own argument checks
 * first, so an argument fa_bwd rejects is rejected here with the same code).
 *   Scratch comes from a fixed array inside the library's device image of
 *   fa_bwd_noalloc_max_scratch_bytes() bytes (64 MiB).  A problem whose
 *   fa_bwd_workspace_size() exceeds it is rejected with FA_ERR_WORKSPACE
 *   before anything is launched.
 *   The array is reserved in device memory when the module holding it is
 *   loaded into a context: under CUDA's default lazy module loading that is
 *   the first call on each device, which therefore allocates those 64 MiB
 *   implicitly, can fail with FA_ERR_CUDA when the device lacks the memory,
 *   and may synchronise; it stays reserved until the context is destroyed.
 *   Make the first call on a device outside latency-critical code and before
 *   any stream capture.  The array's device address is cached per device and
 *   per context (a call in another context, or after a device reset, looks
 *   it up again).
 *   All calls share the one array: calls that overlap on the GPU race and
 *   must be ordered by the caller.  Nothing needs clearing between calls;
 *   each call rewrites the scratch it reads.
 *   After its first call on a device it allocates nothing: no cudaMalloc,
 *   cudaFree or allocating library call.
 */
FA_API fa_status fa_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                const float *lse, const void *dout, void *dq, void *dk,
                                void *dv, int B, int H, int N, int d, float scale, int causal,
                                const int32_t *kv_len, const uint8_t *block_mask, void *stream);

/* Size in bytes of fa_bwd_noalloc's fixed scratch array (its maximum workspace). */
FA_API size_t fa_bwd_noalloc_max_scratch_bytes(void);

/*
 * fa_fwd that also writes the two row statistics the pages keep in HBM
 * ([EXPL] "Method" and "Key ideas": the running max m and the exponential
 * sum l of every query row, from which the backward can rebuild P):
 *   row_max  out: fp32 [B, H, N], m_i = max over the allowed keys of s_ij,
 *                 s = scale * Q K^T (natural units, not base 2)
 *   row_sum  out: fp32 [B, H, N], l_i = sum over the allowed keys of
 *                 exp(s_ij - m_i)
 * so that lse_i = m_i + ln l_i; a row with no allowed key gets m = -inf,
 * l = 0.  Both pointers are required and 16-byte aligned.  Everything else
 * as fa_fwd.
 */
FA_API fa_status fa_fwd_stats(const void *q, const void *k, const void *v, void *o, float *lse,
                              float *row_max, float *row_sum, int B, int H, int N, int d,
                              float scale, int causal, const int32_t *kv_len,
                              const uint8_t *block_mask, void *stream);

/*
 * fa_fwd with the block-sparse mask given in compressed-row form instead of
 * the dense nb x nb bytes ([EXPL] "Extension: Block-Sparse FlashAttention":
 * only the nonzero blocks of the mask are evaluated; a CSR list of them is
 * the same mask):
 *   row_ptr  in : DEVICE int32 [nb + 1], nb = ceil(N / 128); row_ptr[0] = 0,
 *                 non-decreasing, row_ptr[nb] = nnz
 *   col_idx  in : DEVICE int32 [nnz]; the key tiles of query tile I are
 *                 col_idx[row_ptr[I] .. row_ptr[I + 1]), in any order;
 *                 repeated entries count once.  May be NULL when nnz = 0.
 * A row range or tile index out of range is skipped and reported by
 * fa_check as FA_ERR_INVALID_ARG (the values live on the device, so they are
 * checked by the kernel, not before the launch).  N <= 1024 * 128.
 */
FA_API fa_status fa_fwd_csr(const void *q, const void *k, const void *v, void *o, float *lse,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t *kv_len, const int32_t *row_ptr,
                            const int32_t *col_idx, int nnz, void *stream);

/*
 * Backward of fa_fwd_csr: the CSR mask is expanded into the dense form in
 * the workspace, then fa_bwd runs with it.  The workspace is
 * fa_bwd_csr_workspace_size() bytes: fa_bwd_workspace_size() plus nb * nb
 * rounded up to 256.  Same errors as fa_fwd_csr and fa_bwd.
 */
FA_API size_t fa_bwd_csr_workspace_size(int B, int H, int N, int d);

FA_API fa_status fa_bwd_csr(const void *q, const void *k, const void *v, const void *o,
                            const float *lse, const void *dout, void *dq, void *dk, void *dv,
                            int B, int H, int N, int d, float scale, int causal,
                            const int32_t *kv_len, const int32_t *row_ptr,
                            const int32_t *col_idx, int nnz, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * Forward of Nq query rows against Nk key rows (a query block that continues
 * a longer key sequence, such as the new tokens of a decoder attending to
 * their cache).  The pages fix only the square case; causal is aligned to
 * the bottom right: query i keeps key j iff j <= i + (Nk - Nq), so the last
 * query sees every key and Nq == Nk is fa_fwd's rule; query rows with
 * i < Nq - Nk have no key and get O = 0, lse = -inf.  No block mask, no
 * dropout; kv_len as in fa_fwd, clamped to [0, Nk].
 *   q, o  : bf16 [B, H, Nq, d];  k, v : bf16 [B, H, Nk, d];  lse : fp32 [B, H, Nq]
 */
FA_API fa_status fa_fwd_qk(const void *q, const void *k, const void *v, void *o, float *lse,
                           int B, int H, int Nq, int Nk, int d, float scale, int causal,
                           const int32_t *kv_len, void *stream);

/*
 * Backward of fa_fwd_qk, by the same recomputation as fa_bwd with the same
 * bottom-right causal rule; the gradient definitions are fa_bwd's with Nq
 * query rows and Nk key rows.
 *   q, o, dO in : bf16 [B, H, Nq, d];  k, v in : bf16 [B, H, Nk, d]
 *   lse      in : fp32 [B, H, Nq], fa_fwd_qk's output for the same inputs
 *   dq      out : bf16 [B, H, Nq, d];  dk, dv out : bf16 [B, H, Nk, d]
 *   workspace   : >= fa_bwd_workspace_size(B, H, Nq, d) bytes (it scales
 *                 with the query rows only)
 * Query rows with no key give dQ = 0; keys that no query sees (past kv_len)
 * give dK = dV = 0.  Errors as fa_bwd (FA_ERR_INVALID_ARG also for Nk < 1).
 */
FA_API fa_status fa_bwd_qk(const void *q, const void *k, const void *v, const void *o,
                           const float *lse, const void *dout, void *dq, void *dk, void *dv,
                           int B, int H, int Nq, int Nk, int d, float scale, int causal,
                           const int32_t *kv_len, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * Synchronises stream and reports the first device-side error recorded since
 * the previous fa_check: FA_ERR_TIMEOUT when a bounded wait inside a kernel
 * ran out (the kernel then returned early and its outputs are invalid),
 * FA_ERR_INVALID_ARG when a kernel found a device-side argument out of range
 * (a CSR block mask), FA_ERR_CUDA for an asynchronous CUDA error, FA_OK
 * otherwise.  Clears the recorded error.
 */
FA_API fa_status fa_check(void *stream);

/* Human-readable name of a status code (static storage; never NULL). */
FA_API const char *fa_status_string(int status);

/*
 * Upper bound, in nanoseconds, on every spin-wait inside the kernels
 * (default 2e9).  Values <= 0 restore the default.  Affects launches issued
 * after the call.  Intended for tests of the timeout path.
 */
FA_API void fa_set_wait_timeout_ns(long long ns);

/*
 * Test hook for the failure-detection path: when enabled (nonzero), the next
 * fa_fwd launches its kernel with the key/value producer told never to
 * issue its loads, so that the consumers' bounded waits run out and the
 * kernel returns FA_ERR_TIMEOUT through fa_check.  No GPU fault is raised.
 * The flag clears itself after one launch.
 */
FA_API void fa_debug_starve_next_fwd(int enable);

/*
 * Measurement hook: when both are non-NULL, subsequent fa_bwd calls record
 * the two cudaEvent_t handles on their stream immediately before and after
 * the main backward kernel (the dK/dV/dQ kernel), so a caller can time that
 * kernel alone with cudaEventElapsedTime.  Pass NULLs to stop.  The events
 * are owned by the caller.
 */
FA_API void fa_set_bwd_main_events(void *start_event, void *stop_event);

#ifdef __cplusplus
}
#endif
#endif /* FA_H */
