/*
 * fa.h - C ABI of the GB300 (sm_103a) exact-attention library (libfa.so).
 *
 * Operations
 *   fa_fwd             FlashAttention-2 forward over dense [B,H,S,D] tensors.
 *   fa_fwd_varlen      the same forward over packed variable-length sequences.
 *   fa_decode_splitkv  split-KV decoding, phase 1: per-partition partials.
 *   fa_splitkv_merge   split-KV decoding, phase 2: log-sum-exp merge.
 *   fa_decode_splitkv_fused, fa_decode_paged_splitkv_fused
 *                      both phases in one launch (last partition merges).
 *   fa_bwd             backward pass: dQ, dK, dV from dO and the forward LSE.
 *
 * Common rules
 *   - Every tensor pointer is a DEVICE pointer owned by the caller. The library
 *     allocates no memory and keeps no state between calls, apart from one
 *     device-resident error word per GPU (see fa_check_device_error) and the
 *     test setting of fa_test_withhold_load (off unless a test turns it on).
 *   - Calls are asynchronous: work is enqueued on `stream` (a cudaStream_t
 *     passed as void*, NULL = the legacy default stream) and the call returns
 *     after the launch. Inputs must stay valid until the work completes.
 *   - Arguments are validated on the host before anything is launched; a
 *     failed check returns a negative status and enqueues nothing. Contents of
 *     device arrays (cu_seqlens) are not read on the host.
 *   - 16-bit tensors are contiguous, row-major, 16-byte aligned; fp32 arrays
 *     are contiguous and 4-byte aligned. D is 64 or 128 (the forward also
 *     takes 256, 512 and 1024).
 *   - `scale` multiplies Q K^T before the softmax and must be finite and > 0
 *     (1/sqrt(D) is the usual value).
 *   - LSE outputs are natural-log sums over the scaled, masked scores:
 *     LSE_i = ln sum_j exp(scale * q_i . k_j).
 *   - No C++ exception crosses this boundary.
 *
 * The kernels are compiled for sm_103a only; on another GPU every launch fails
 * with FA_ERR_CUDA.
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

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = -1,           /* a required pointer is NULL */
    FA_ERR_SHAPE = -2,          /* a size is <= 0, or too large for 32-bit indexing */
    FA_ERR_HEADDIM = -3,        /* D not supported: forward 64/128/256/512/1024, decode and backward 64/128 */
    FA_ERR_DTYPE = -4,          /* dtype is not FA_FP16 or FA_BF16 */
    FA_ERR_ALIGN = -5,          /* a 16-bit tensor is not 16-byte aligned (fp32: 4-byte) */
    FA_ERR_SPLITS = -6,         /* num_splits < 1 or > Sk (or > FA_MAX_SPLITS) */
    FA_ERR_SCALE = -7,          /* scale is not finite and > 0 */
    FA_ERR_CUDA = -8,           /* the CUDA runtime reported an error (launch, tensor map) */
    FA_ERR_DEVICE_TIMEOUT = -9, /* a kernel gave up waiting on an on-chip barrier */
    FA_ERR_SCRATCH = -10,       /* fa_decode_noalloc: problem larger than its built-in scratch */
    FA_ERR_DEVICE_INDEX = -11,  /* a kernel met an out-of-range block-table entry */
    FA_ERR_WORKSPACE = -12,     /* caller workspace smaller than required */
    FA_ERR_DEVICE_SEQLENS = -13 /* fa_fwd_varlen: cu_seqlens inconsistent with the sizes (see there) */
} fa_status_t;

typedef enum { FA_FP16 = 0, FA_BF16 = 1 } fa_dtype_t;

/* Upper bound on the number of KV partitions of the split-KV decode. */
#define FA_MAX_SPLITS 1024

/*
 * fa_fwd - exact attention forward pass, O = softmax(scale * Q K^T [+ mask]) V.
 *
 * Defined by "FlashAttention-2 MMA" (Usage Example: [B,H,S,D] tensors and a
 * causal flag; Technical Details: online softmax with running max and sum,
 * causal rule k_idx <= q_idx) and "Adaptive High-Performance Attention Kernels
 * in CUDA" (Architectural Progression, stages 3-4: outer loop over query
 * tiles, on-chip output accumulator, upper-triangular tiles skipped).
 *
 *   q    [B,H,Sq,D]  fp16/bf16          k, v [B,H,Sk,D]  same dtype
 *   o    [B,H,Sq,D]  output, dtype of q
 *   lse  [B,H,Sq]    fp32 output
 *   causal  0 or 1. When 1, query i sees keys j <= i (top-left alignment,
 *           also when Sq != Sk).
 *   D       64, 128, 256, 512 or 1024. D = 256 covers the pages' large-head
 *           ("GPT-4 style", head_dim 256) configuration and runs a kernel with
 *           one query tile per CTA and 64-key K/V tiles. D = 512 and 1024 (the
 *           pages' "Large Head" and "Massive Head" rows) take the Split-D
 *           strategy ("FlashAttention-2 MMA", Supported Dispatch
 *           Strategies 3: head_dim > 256 partitions the
 *           head dimension across thread blocks): each CTA forms the full
 *           scores and writes one 256-column slice of O. Same results
 *           contract for every D.
 * Errors: FA_ERR_NULL, FA_ERR_SHAPE (B,H,Sq,Sk < 1), FA_ERR_HEADDIM,
 * FA_ERR_DTYPE, FA_ERR_ALIGN, FA_ERR_SCALE, FA_ERR_CUDA.
 */
FA_API fa_status_t fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                   int B, int H, int Sq, int Sk, int D, int causal, float scale,
                   fa_dtype_t dtype, void *stream);

/*
 * fa_fwd_varlen - the forward pass over packed sequences of different lengths.
 *
 * Defined by "Adaptive High-Performance Attention Kernels in CUDA" (Advanced
 * Production Features 3: tokens flattened to [total_tokens, H, d], sequence
 * boundaries from cumulative lengths, no padding computed).
 *
 *   q, o          [total_q,H,D]      k, v [total_k,H,D]
 *   lse           [H,total_q] fp32   (per-head contiguous)
 *   cu_seqlens_q  device int32[num_seqs+1], 0 = cu[0] <= cu[1] <= ... = total_q
 *   cu_seqlens_k  device int32[num_seqs+1], same rules with total_k
 *   max_seqlen_q  >= every query length (sizes the launch)
 * Sequence i attends its own keys only; causal positions are counted from the
 * start of each sequence. Zero-length sequences are allowed.
 * The offsets are checked on the device (the host cannot read them without a
 * synchronisation): if cu_seqlens_q or cu_seqlens_k is negative, decreasing or
 * beyond total_q / total_k, or a query sequence is longer than max_seqlen_q,
 * the launch computes nothing (o and lse are neither read nor written) and
 * the next fa_check_device_error returns FA_ERR_DEVICE_SEQLENS.
 * Errors: as fa_fwd, plus FA_ERR_SHAPE for num_seqs < 1 or total_* < 1.
 */
FA_API fa_status_t fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                          int num_seqs, int total_q, int total_k, int max_seqlen_q,
                          int H, int D, int causal, float scale, fa_dtype_t dtype,
                          void *stream);

/*
 * fa_decode_splitkv - split-KV decoding, phase 1 (one query per head).
 *
 * Defined by "Adaptive High-Performance Attention Kernels in CUDA" (Advanced
 * Production Features 1: the KV cache is split into S partitions that run
 * partial attention concurrently) and "FlashAttention-2 MMA" (Split-KV
 * strategy for S_q = 1).
 *
 * Partition s covers keys [s*P, min((s+1)*P, Sk)) with P = ceil(Sk/S); the
 * last partitions may be short or empty. For each (b,h,s):
 *   m_part[b,h,s] = max_j scale * q . k_j                  (-inf if empty)
 *   l_part[b,h,s] = sum_j exp(scale * q . k_j - m)         (0 if empty)
 *   o_part[b,h,s,:] = sum_j exp(scale * q . k_j - m) v_j   (unnormalised)
 *
 *   q [B,H,1,D] (= [B,H,D])   k, v [B,H,Sk,D]   fp16/bf16
 *   o_part [B,H,S,D] fp32, m_part and l_part [B,H,S] fp32: caller workspace.
 * Errors: FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEADDIM, FA_ERR_DTYPE,
 * FA_ERR_ALIGN, FA_ERR_SPLITS, FA_ERR_SCALE, FA_ERR_CUDA.
 */
FA_API fa_status_t fa_decode_splitkv(const void *q, const void *k, const void *v, float *o_part,
                              float *m_part, float *l_part, int B, int H, int Sk, int D,
                              int num_splits, float scale, fa_dtype_t dtype, void *stream);

/*
 * fa_decode_paged_splitkv - split-KV decoding, phase 1, over a paged KV cache.
 *
 * Defined by "Adaptive High-Performance Attention Kernels in CUDA" (Advanced
 * Production Features 4: the KV cache is kept as physical pages
 * [num_blocks, H, block_size, d] and a per-sequence block table translates a
 * logical key position into a page) combined with the split-KV phase 1 above.
 *
 *   q            [B,H,1,D] fp16/bf16
 *   k_cache, v_cache [num_blocks,H,block_size,D], same dtype
 *   block_table  device int32 [B, max_blocks_per_seq]: page of each logical
 *                block; entries past a sequence's length are never read
 *   seq_lens     device int32 [B]: keys of each sequence (clamped to
 *                [0, max_blocks_per_seq * block_size])
 *   o_part [B,H,S,D], m_part and l_part [B,H,S] fp32 outputs, as in
 *                fa_decode_splitkv, with partition size ceil(seq_lens[b]/S)
 *                per sequence (a length-0 sequence has only empty partitions).
 *   block_size   a power of two, 1..1024.
 * Page numbers outside [0, num_blocks) are never dereferenced: their keys are
 * skipped and fa_check_device_error later returns FA_ERR_DEVICE_INDEX.
 * Phase 2 is fa_splitkv_merge, unchanged.
 * Errors: FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEADDIM, FA_ERR_DTYPE,
 * FA_ERR_ALIGN, FA_ERR_SPLITS, FA_ERR_SCALE, FA_ERR_CUDA.
 */
FA_API fa_status_t fa_decode_paged_splitkv(const void *q, const void *k_cache, const void *v_cache,
                                           const int32_t *block_table, const int32_t *seq_lens,
                                           float *o_part, float *m_part, float *l_part, int B, int H,
                                           int D, int num_blocks, int block_size,
                                           int max_blocks_per_seq, int num_splits, float scale,
                                           fa_dtype_t dtype, void *stream);

/*
 * fa_splitkv_merge - split-KV decoding, phase 2 (log-sum-exp reduction).
 *
 * Defined by "Adaptive High-Performance Attention Kernels in CUDA" (Advanced
 * Production Features 1: O = sum_s e^{m_s - m_global} / l_global * O_s), read
 * with m_global = max_s m_s and l_global = sum_s e^{m_s - m_global} l_s.
 *
 *   inputs as written by fa_decode_splitkv with the same B, H, D, num_splits
 *   o   [B,H,1,D] output (dtype)     lse [B,H] fp32 output = m_global + ln l_global
 * Errors: FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEADDIM, FA_ERR_DTYPE,
 * FA_ERR_ALIGN, FA_ERR_SPLITS, FA_ERR_CUDA.
 */
FA_API fa_status_t fa_splitkv_merge(const float *o_part, const float *m_part, const float *l_part,
                             void *o, float *lse, int B, int H, int D, int num_splits,
                             fa_dtype_t dtype, void *stream);

/*
 * fa_decode_splitkv_fused - split-KV decoding, phase 1 and phase 2 in one
 * launch.
 *
 * Computes what fa_decode_splitkv followed by fa_splitkv_merge computes
 * ("Adaptive High-Performance Attention Kernels in CUDA", Advanced Production
 * Features 1: partial attention per partition, then the log-sum-exp merge),
 * without the second launch: each partition's CTA writes its partials to
 * o_part, m_part, l_part (same layout and values as fa_decode_splitkv), then
 * counts itself done on the head's counter; the CTA that finishes last merges
 * the head into o and lse and sets the counter back to zero.
 *
 *   q, k, v, o_part, m_part, l_part, B, H, Sk, D, num_splits, scale, dtype:
 *             as fa_decode_splitkv
 *   o         [B,H,1,D] output (dtype), lse [B,H] fp32: as fa_splitkv_merge
 *   counters  device int32 [B*H], caller-owned. All zero before the first
 *             call; a call that completes leaves it all zero again, so it can
 *             be reused without clearing. If a call fails to launch, clear it.
 * Calls that share counters or partial buffers must not overlap on the GPU.
 * Errors: as fa_decode_splitkv, plus FA_ERR_NULL when o, lse or counters is
 * NULL and FA_ERR_ALIGN when o is not 16-byte or lse/counters not 4-byte
 * aligned.
 */
FA_API fa_status_t fa_decode_splitkv_fused(const void *q, const void *k, const void *v, void *o, float *lse,
                                           float *o_part, float *m_part, float *l_part, int32_t *counters,
                                           int B, int H, int Sk, int D, int num_splits, float scale,
                                           fa_dtype_t dtype, void *stream);

/*
 * fa_decode_paged_splitkv_fused - fa_decode_paged_splitkv and
 * fa_splitkv_merge in one launch, over a paged KV cache ("Adaptive ...",
 * Advanced Production Features 4 and 1).
 *
 *   arguments as fa_decode_paged_splitkv, plus o, lse and counters as
 *   fa_decode_splitkv_fused (same rules for counters).
 * A length-0 sequence gives o = 0 and lse = -inf. Out-of-range page numbers
 * are skipped and reported as by fa_decode_paged_splitkv.
 * Errors: as fa_decode_paged_splitkv, plus those of fa_decode_splitkv_fused
 * for o, lse and counters.
 */
FA_API fa_status_t fa_decode_paged_splitkv_fused(const void *q, const void *k_cache, const void *v_cache,
                                                 const int32_t *block_table, const int32_t *seq_lens, void *o,
                                                 float *lse, float *o_part, float *m_part, float *l_part,
                                                 int32_t *counters, int B, int H, int D, int num_blocks,
                                                 int block_size, int max_blocks_per_seq, int num_splits,
                                                 float scale, fa_dtype_t dtype, void *stream);

/*
 * fa_bwd_workspace_bytes - bytes of workspace fa_bwd needs:
 * 4 * (B*H*Sq*D + 2*B*H*ceil(Sq/128)*128) + 16 (an fp32 dQ accumulator, the
 * per-row statistics and the work counter of the D = 128 kernel); 0 for an
 * invalid shape.
 */
FA_API size_t fa_bwd_workspace_bytes(int B, int H, int Sq, int D);

/*
 * fa_bwd - exact attention backward pass.
 *
 * Defined by "Adaptive High-Performance Attention Kernels in CUDA" (Advanced
 * Production Features 2, Custom CUDA Backward Pass): S = scale Q K^T and
 * P = exp(S - LSE) are recomputed on chip from the forward's LSE (P is never
 * stored), D_i = sum_k dO_ik O_ik, dS = P (dP - D_i) with dP = dO V^T; then
 * dV = P^T dO, dK = scale dS^T Q, dQ = scale dS K (chain rule of the same
 * definition), with the causal rule of fa_fwd.
 *
 *   q, o, dout  [B,H,Sq,D]  fp16/bf16   k, v [B,H,Sk,D]  same dtype
 *   lse         [B,H,Sq] fp32, as written by fa_fwd for these q, k, v
 *   dq [B,H,Sq,D], dk and dv [B,H,Sk,D]: outputs in the input dtype
 *   workspace   caller-owned device memory of at least
 *               fa_bwd_workspace_bytes(B, H, Sq, D) bytes, 16-byte aligned
 *               (fp32 dQ accumulator, per-row statistics, work counter); its
 *               contents on entry do not matter. Calls sharing a workspace
 *               must not overlap on the GPU.
 *   D           64 or 128.
 * Three launches on `stream`. dQ sums contributions of all key tiles with
 * fp32 atomic additions, so its rounding can differ between runs; dK and dV
 * are deterministic.
 * Errors: FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEADDIM, FA_ERR_DTYPE,
 * FA_ERR_ALIGN, FA_ERR_SCALE, FA_ERR_WORKSPACE, FA_ERR_CUDA.
 */
FA_API fa_status_t fa_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                          const float *lse, void *dq, void *dk, void *dv, float *workspace,
                          size_t workspace_bytes, int B, int H, int Sq, int Sk, int D, int causal,
                          float scale, fa_dtype_t dtype, void *stream);

/*
 * fa_bwd_varlen_workspace_bytes - bytes of workspace fa_bwd_varlen needs:
 * 4 * (total_q*H*D + 2*H*total_q) + 16; 0 for an invalid shape.
 */
FA_API size_t fa_bwd_varlen_workspace_bytes(int total_q, int H, int D);

/*
 * fa_bwd_varlen - the backward pass over packed sequences of different lengths.
 *
 * Defined by "Adaptive High-Performance Attention Kernels in CUDA" (Advanced
 * Production Features 2, Custom CUDA Backward Pass, and 3, Ragged / Variable-
 * Length Sequences): the gradients of fa_fwd_varlen. Each sequence is an
 * independent attention over its own keys, so its gradients are those of
 * fa_bwd on that sequence alone; causal positions count from each sequence's
 * start (top-left, as in fa_fwd_varlen).
 *
 *   q, o, dout    [total_q,H,D]  fp16/bf16   k, v [total_k,H,D]  same dtype
 *   lse           [H,total_q] fp32, as written by fa_fwd_varlen
 *   dq [total_q,H,D], dk and dv [total_k,H,D]: outputs in the input dtype;
 *                 rows of tokens outside every sequence are left unwritten in
 *                 dk and dv, and dq rows outside every sequence are zero
 *   cu_seqlens_q, cu_seqlens_k   device int32[num_seqs+1], as in fa_fwd_varlen
 *   max_seqlen_q, max_seqlen_k   >= every query / key length (size the launch)
 *   workspace     caller-owned device memory of at least
 *                 fa_bwd_varlen_workspace_bytes(total_q, H, D) bytes, 16-byte
 *                 aligned; its contents on entry do not matter. Calls sharing
 *                 a workspace must not overlap on the GPU.
 *   D             64 or 128.
 * Keys of a sequence without queries get dK = dV = 0. Three launches on
 * `stream`; dQ's fp32 additions make its rounding run-dependent, dK and dV are
 * deterministic. The offsets are checked on the device: a sequence whose
 * offsets lie outside the tensors, or that is longer than max_seqlen_q /
 * max_seqlen_k, is skipped (its gradients are not written) and the next
 * fa_check_device_error returns FA_ERR_DEVICE_SEQLENS.
 * Errors: FA_ERR_NULL, FA_ERR_SHAPE, FA_ERR_HEADDIM, FA_ERR_DTYPE,
 * FA_ERR_ALIGN, FA_ERR_SCALE, FA_ERR_WORKSPACE, FA_ERR_CUDA.
 */
FA_API fa_status_t fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const void *dout,
                                 const float *lse, void *dq, void *dk, void *dv, float *workspace,
                                 size_t workspace_bytes, const int32_t *cu_seqlens_q,
                                 const int32_t *cu_seqlens_k, int num_seqs, int total_q, int total_k,
                                 int max_seqlen_q, int max_seqlen_k, int H, int D, int causal, float scale,
                                 fa_dtype_t dtype, void *stream);

/*
 * fa_check_device_error - synchronise `stream`, then read and clear the
 * current device's error word. Kernels bound every wait on an on-chip barrier;
 * a wait that runs out sets the word, releases what the CTA holds and returns.
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_INDEX (an out-of-range
 * block-table entry was skipped), FA_ERR_DEVICE_SEQLENS (a packed-sequence
 * launch found inconsistent cu_seqlens: see fa_fwd_varlen, fa_bwd_varlen), or FA_ERR_CUDA
 * when the runtime itself reports an error.
 */
FA_API fa_status_t fa_check_device_error(void *stream);

/*
 * fa_test_withhold_load - test support for the failure path of the prefill
 * kernels (fa_fwd, fa_fwd_varlen, fa_bwd, fa_bwd_varlen). With load = n > 0,
 * CTA 0 of every later launch of those kernels never issues one of its tile
 * loads (the forward's V tile n - 1, the backward's Q/dO step n - 1), so the
 * wait for it cannot complete: the kernel's bounded wait runs out after
 * `wait_limit_ns`, its CTAs drain the copies they issued, release tensor
 * memory and stop, and fa_check_device_error returns FA_ERR_DEVICE_TIMEOUT.
 * Outputs of such a launch are undefined. `wait_limit_ns` (0 = the default,
 * one second) bounds every on-chip wait of every launch of those kernels.
 * load = 0 and wait_limit_ns = 0 restore normal operation. The setting is
 * process-wide; it is not meant to be changed while other threads launch.
 * Returns FA_OK, or FA_ERR_SHAPE for a negative load.
 */
FA_API fa_status_t fa_test_withhold_load(int load, unsigned long long wait_limit_ns);

/*
 * fa_decode_noalloc - split-KV decoding (phase 1 and phase 2 in one call) that
 * allocates nothing and needs no caller workspace. The pages have no
 * counterpart: this entry point exists for callers that cannot allocate
 * device memory when they call in (an engine hook that must not allocate, a
 * latency-critical loop that cannot take the device-wide synchronisation an
 * allocation may bring, a process whose memory a pool has fully reserved).
 *
 * The partials live in a fixed device array built into the library, of
 * FA_NOALLOC_SCRATCH_FLOATS floats (8 MiB), which every GPU that loads the
 * library holds until the process exits. A call needs
 * B*H*num_splits*D + 2*B*H*num_splits floats (each part rounded up to 4);
 * larger problems return FA_ERR_SCRATCH before anything is enqueued. The
 * first call on a device looks up the array's device address (with that
 * device current); make it before any stream capture. All calls share the
 * array: calls whose work overlaps on the GPU race and must be serialised by
 * the caller. Nothing needs clearing between calls.
 *
 *   q [B,H,1,D], k and v [B,H,Sk,D], o [B,H,1,D] (dtype), lse [B,H] fp32.
 *   Results equal fa_decode_splitkv followed by fa_splitkv_merge.
 * Errors: as fa_decode_splitkv, plus FA_ERR_SCRATCH.
 */
#define FA_NOALLOC_SCRATCH_FLOATS (2 * 1024 * 1024)
FA_API fa_status_t fa_decode_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                                     int B, int H, int Sk, int D, int num_splits, float scale,
                                     fa_dtype_t dtype, void *stream);

/* Static, NUL-terminated description of a status code (never NULL). */
FA_API const char *fa_status_string(fa_status_t status);

/* Library version as major*10000 + minor*100 + patch. */
FA_API int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
