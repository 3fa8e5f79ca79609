/*
 * fa_gb300.h -- C ABI of the GB300 (sm_103a) variable-length attention
 * forward library (libfa_gb300.so).
 *
 * The library computes, for packed variable-length sequences,
 *
 *     O = softmax(scale * Q Kᵀ + mask) V        (online softmax, fp32 state)
 *     LSE = log-sum-exp of the masked, scaled scores (natural log)
 *
 * and the sparse-MLA decode variant that attends over per-token top-k rows
 * gathered from a paged 576-wide latent cache.
 *
 * Conventions shared by every entry point
 *   - All tensors are caller-owned device buffers, C-contiguous (except the
 *     q/k/v views fa_varlen_fwd_strided takes), 16-byte aligned.  bf16 means
 *     IEEE bfloat16 bit patterns (2 bytes).
 *   - Calls are asynchronous on `stream` (NULL = legacy default stream).  The
 *     library performs no host<->device copy and never synchronises; it only
 *     encodes TMA descriptors on the host and launches.  It allocates no
 *     device memory per call.  The one exception is a one-time allocation:
 *     fa_sparse_mla_decode allocates a partial-result workspace for a
 *     (device, stream) on the first call there that needs one (see that
 *     entry point).  fa_sparse_mla_decode_noalloc never allocates.
 *     The first call on a device queries device attributes once; make it
 *     before any stream capture that is to contain a call.
 *   - Errors detected on the host (argument checks) are returned before any
 *     launch and leave every output untouched.  A launch failure returns
 *     FA_ERR_LAUNCH.  Problems found on the device (a pipeline wait that ran
 *     out of time) set a device status word that fa_get_device_status()
 *     reports; outputs of that call are then undefined.
 *   - Results are bitwise deterministic run to run for identical inputs.
 *
 * Sources of the semantics (web pages the interface is taken from):
 *   [flash_attn]   vLLM API docs, "vllm.v1.attention.backends.mla.prefill.
 *                  flash_attn": FA4MLAPrefillKernel (CompileKey fields: q/k/v
 *                  shapes, cu_seqlens, max_seqlen, softmax_scale, causal,
 *                  window_size, return_softmax_lse), FlashAttnPrefillBackend
 *                  (run_prefill_new_tokens: causal, cu_seqlens_q ==
 *                  cu_seqlens_k; run_prefill_context_chunk: non-causal,
 *                  returns the LSE), FA4SplitKVCombineKernel (LSE laid out
 *                  [num_heads, total_q]).
 *   [sglang-fa4]   sglang PR #41344, "fill gaps in FA4 path on Blackwell":
 *                  "Motivation" and "Modifications" (row max, exp2, rescale
 *                  threshold, masking only boundary tiles), "Accuracy Tests"
 *                  (chunked prefill with q shorter than k; head dims
 *                  64/96/128/(192,128); sliding window), "Speed Tests and
 *                  Profiling" (ViT head dims 64/72/80/128).
 *   [mla_sparse]   vLLM API docs, "vllm.v1.attention.backends.mla.
 *                  flashattn_mla_sparse": FlashAttnMLASparseFA4Backend (BF16
 *                  cache only, head size 576 = 512 latent + 64 rope, block
 *                  size a multiple of 64, index_topk % 128 == 0, 8..128
 *                  query heads) and _fa4_varlen_scalars (one query row per
 *                  token).
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st* fa_stream_t;

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer */
  FA_ERR_UNSUPPORTED = 2,   /* valid request outside what is compiled in */
  FA_ERR_ARCH = 3,          /* current device is not sm_103 (GB300) */
  FA_ERR_LAUNCH = 4,        /* CUDA launch or driver call failed */
  FA_ERR_DEVICE_TIMEOUT = 5, /* reported by fa_get_device_status only */
  FA_ERR_SCRATCH = 6        /* fa_sparse_mla_decode_noalloc: the call needs more
                               scratch than its fixed buffer holds */
} fa_status;

/*
 * fa_varlen_fwd -- attention forward over packed variable-length sequences.
 * Defined by [flash_attn] (flash_attn_varlen_func keyword arguments as used
 * by run_prefill_new_tokens / run_prefill_context_chunk) and [sglang-fa4].
 *
 *   q             bf16 [total_q, num_heads,   d_qk]
 *   k             bf16 [total_k, num_heads_k, d_qk]
 *   v             bf16 [total_k, num_heads_k, d_v]
 *   cu_seqlens_q  int32 [batch + 1] device, non-decreasing, cu[0] = 0,
 *                 cu[batch] = total_q.  Sequence b owns query tokens
 *                 [cu_seqlens_q[b], cu_seqlens_q[b+1]).  The kernel
 *                 clamps each entry to [0, total_q] and each end to at least
 *                 its start, so a malformed array gives empty or shortened
 *                 sequences and no access outside the tensors (rows that
 *                 two such sequences share get either's values).
 *   cu_seqlens_k  int32 [batch + 1] device, same for keys/values.
 *   batch         >= 1.  Up to 2048 sequences run as one launch (the
 *                 kernel sorts their work list in shared memory); a larger
 *                 batch runs as consecutive launches of up to 2048
 *                 sequences each, on `stream`.
 *   num_heads, num_heads_k  num_heads % num_heads_k == 0; query head h reads
 *                 key/value head h / (num_heads / num_heads_k).  When the
 *                 query sequences are short (by the max_seqlen_q hint, else
 *                 total_q / batch), P query heads of one group share each
 *                 128-row query tile (head-group packing, [sglang-fa4]
 *                 "Accuracy Tests": pack_gqa), so that each K/V tile is
 *                 loaded once for P heads; P is the largest power of two up
 *                 to 16 that divides the group and leaves each work item
 *                 (256 / P tokens) at least the expected query length.
 *   (d_qk, d_v)   one of (64,64) (72,72) (80,80) (96,96) (128,128) (192,128).
 *   max_seqlen_q, max_seqlen_k  host hints only (never used for
 *                 correctness; may be 0): they steer head-group packing
 *                 and split-KV.
 *   softmax_scale scale applied to Q Kᵀ before the softmax (> 0).
 *   causal        nonzero: key j is visible to query row i of a sequence iff
 *                 j <= i + (Lk - Lq), i.e. the diagonal is aligned to the
 *                 bottom-right corner (chunked prefill with Lq < Lk).
 *   window_left, window_right  sliding window, inclusive, in the same
 *                 bottom-right frame: j >= i + (Lk-Lq) - window_left and
 *                 j <= i + (Lk-Lq) + window_right; -1 = unbounded.
 *   out           bf16 [total_q, num_heads, d_v]  (written)
 *   lse           fp32 [num_heads, total_q] natural-log LSE, or NULL.
 *
 * A query row with no visible key gets O = 0 and LSE = -inf.  With
 * total_q = 0 nothing is launched (q, out and lse may then be NULL); with
 * total_k = 0 every row has no visible key (k and v may then be NULL).
 *
 * Split-KV ([flash_attn] FA4SplitKVCombineKernel): when the work items
 * (query head x 256 query rows of a sequence) cannot fill half of the SMs
 * and the keys are long, each item's key tiles are split over a thread-block
 * cluster of up to 16 CTAs (8 where larger clusters are unavailable).  Each
 * CTA computes a partial result over its part, and the cluster merges the
 * partials by their log-sum-exp through distributed shared memory, in a
 * fixed order: no workspace, and the same result on every run.  The split
 * is chosen on the host from the sizes and the max_seqlen_k hint (see
 * fa_varlen_fwd_plan); it changes rounding, never the result beyond it.
 *
 * Host errors: FA_ERR_INVALID_ARG (null required pointer, negative sizes,
 * batch < 1, head counts, window < -1, scale <= 0, unaligned pointers),
 * FA_ERR_UNSUPPORTED (head dims), FA_ERR_ARCH.
 */
fa_status fa_varlen_fwd(const void* q, const void* k, const void* v,
                        const int* cu_seqlens_q, const int* cu_seqlens_k,
                        int batch, int total_q, int total_k, int num_heads,
                        int num_heads_k, int d_qk, int d_v, int max_seqlen_q,
                        int max_seqlen_k, float softmax_scale, int causal,
                        int window_left, int window_right, void* out,
                        float* lse, fa_stream_t stream);

/*
 * fa_varlen_fwd_plan -- the launch shape fa_varlen_fwd (and
 * fa_varlen_fwd_strided) would use for a call with these sizes on the
 * current device, without launching anything.  Arguments as fa_varlen_fwd.
 *
 *   *grid   CTAs of the launch (0 when total_q = 0); with more than 2048
 *           sequences, of each launch of 2048
 *   *split  CTAs per work item: 1 = persistent grid of at most one CTA per
 *           SM walking the work list; > 1 = split-KV, one cluster of
 *           *split CTAs per work item
 *   *heads_per_tile  query heads packed into one 128-row query tile (GQA
 *           head-group packing): 1, or P in {2, 4, 8, 16}
 *
 * Host errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (head dims),
 * FA_ERR_ARCH, FA_ERR_LAUNCH (a device query failed).
 */
fa_status fa_varlen_fwd_plan(int batch, int total_q, int total_k, int num_heads,
                             int num_heads_k, int d_qk, int d_v, int max_seqlen_q,
                             int max_seqlen_k, int causal, int window_left, int window_right,
                             int* grid, int* split, int* heads_per_tile);

/*
 * fa_varlen_fwd_strided -- fa_varlen_fwd with q, k and v given as strided
 * views: element (t, h, c) of q is at q + t * q_row_stride + h *
 * q_head_stride + c, likewise for k and v; strides are in elements.  This is
 * the v_stride of [flash_attn] (FA4MLAPrefillKernel.dispatch, the CompileKey's
 * v_stride when V needs no padding): V read straight out of a combined
 * [tokens, heads, nope + v] buffer, its rows num_heads * (nope + v_dim) and
 * its heads nope + v_dim elements apart.
 *
 *   *_row_stride, *_head_stride  multiples of 8 (16 bytes), head stride >=
 *                 the tensor's last dimension, row stride >= (heads - 1) *
 *                 head stride + last dimension (views do not overlap
 *                 themselves); the innermost dimension is contiguous.
 *   all other arguments and errors as fa_varlen_fwd; a stride that breaks
 *   these rules is FA_ERR_INVALID_ARG.  out and lse stay contiguous.
 *   fa_varlen_fwd is this call with the contiguous strides
 *   (num_heads * d, d).
 */
fa_status fa_varlen_fwd_strided(const void* q, long long q_row_stride, long long q_head_stride,
                                const void* k, long long k_row_stride, long long k_head_stride,
                                const void* v, long long v_row_stride, long long v_head_stride,
                                const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                                int total_q, int total_k, int num_heads, int num_heads_k,
                                int d_qk, int d_v, int max_seqlen_q, int max_seqlen_k,
                                float softmax_scale, int causal, int window_left,
                                int window_right, void* out, float* lse, fa_stream_t stream);

/*
 * fa_sparse_mla_decode -- one query row per token attending over top-k rows
 * gathered from a paged latent cache shared by all heads.  Defined by
 * [mla_sparse] (FlashAttnMLASparseFA4Backend, _fa4_varlen_scalars).
 *
 *   q             bf16 [num_tokens, num_heads, 576]
 *   kv_cache      bf16 [num_pages, 64, 576]: 512 latent + 64 rope columns
 *   page_table    int32 [num_tokens, max_pages_per_tok]: physical page of
 *                 each logical page of the token's context
 *   topk_idx      int32 [num_tokens, topk]: logical positions p in the
 *                 token's context; row = page_table[t, p/64]*64 + p%64.
 *                 A slot with p < 0, p >= 64*max_pages_per_tok or a page id
 *                 outside [0, num_pages) is skipped (contributes nothing).
 *   num_heads     one of 8, 16, 32, 64, 128
 *   topk          multiple of 128, 128 .. 64*max_pages_per_tok.  A CTA
 *                 takes at most 2048 key slots (its row table is held in
 *                 shared memory), so a token with a larger top-k is always
 *                 cut between CTAs and merged.
 *   softmax_scale scale of the 576-wide dot product (> 0)
 *   out           bf16 [num_tokens, num_heads, 512]: sum_j p_j * row_j[0:512]
 *   lse           fp32 [num_heads, num_tokens] or NULL
 *   With num_tokens = 0 nothing is launched (q, page_table, topk_idx, out
 *   and lse may then be NULL).
 *
 * The (token, head group, 64-key tile) work is spread evenly over the SMs.
 * When a token's keys end up on several CTAs, their partial results go to a
 * workspace, and a second kernel on `stream` merges them by their
 * log-sum-exp [flash_attn] (FA4SplitKVCombineKernel).
 *
 * Workspace ownership: the library keeps one workspace per (device, stream)
 * for the life of the process.  The first call on a stream whose split needs
 * one allocates it with cudaMalloc; later calls reuse it and allocate
 * nothing.  A call that needs more than the stream's workspace holds
 * allocates a larger one and keeps the old one allocated, so a CUDA graph
 * captured earlier stays valid.  fa_sparse_mla_decode_plan gives the size a
 * call needs.  Make the first call on a stream before any stream capture
 * that is to contain a call.  Calls on one stream share its workspace in
 * stream order.  Per-thread default streams of different host threads share
 * one workspace per device, so they must not run decode calls at the same
 * time.  Up to top-k 2048 the split is used for at most two waves of CTAs
 * (a workspace of about 80 MB on 152 SMs); a larger top-k always splits,
 * and its workspace is 2 x CTAs x 131 KB (fa_sparse_mla_decode_plan).
 *
 * Host errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED (heads, topk),
 * FA_ERR_ARCH, FA_ERR_LAUNCH (launch or workspace allocation failed).
 */
fa_status fa_sparse_mla_decode(const void* q, const void* kv_cache,
                               const int* page_table, const int* topk_idx,
                               int num_tokens, int num_heads, int topk,
                               int num_pages, int max_pages_per_tok,
                               float softmax_scale, void* out, float* lse,
                               fa_stream_t stream);

/*
 * fa_sparse_mla_decode_plan -- the work split fa_sparse_mla_decode (and
 * fa_sparse_mla_decode_noalloc) would use for a call of this size on the
 * current device, without launching anything.
 *
 *   *launches         kernel launches of the call: 0 (no tokens), 1, or 2
 *                     (the split cuts tokens between CTAs and a merge
 *                     kernel combines them)
 *   *workspace_bytes  partial-result workspace the call needs (0 with one
 *                     launch)
 *
 * Host errors: FA_ERR_INVALID_ARG (null outputs, negative sizes),
 * FA_ERR_UNSUPPORTED (heads, topk as fa_sparse_mla_decode), FA_ERR_ARCH.
 */
fa_status fa_sparse_mla_decode_plan(int num_tokens, int num_heads, int topk, int* launches,
                                    size_t* workspace_bytes);

/*
 * fa_sparse_mla_decode_noalloc -- fa_sparse_mla_decode without any device
 * memory allocation.  The method's pages have no counterpart to this entry
 * point: it serves callers that must not allocate (a fixed memory budget, or
 * their own memory management).  Arguments, layouts, results and the other
 * errors are those of fa_sparse_mla_decode; the same kernels run.
 *
 * When the work split cuts a token's keys between CTAs, the partial results
 * go to one scratch buffer of fixed size (FA_NOALLOC_SCRATCH_BYTES) that the
 * library holds in device memory (one per device) instead of a workspace
 * allocation.  Nothing in it has to start at zero: every partial result is
 * written before it is read, within the same call.
 *
 *   - A call whose split needs more scratch returns FA_ERR_SCRATCH and
 *     launches nothing (fa_sparse_mla_decode handles it).
 *   - Calls that can overlap in time on one device (different streams, or
 *     different host threads) race on the shared scratch: the caller must
 *     order them.
 *   - The first call on each device does one-time setup (scratch address
 *     lookup, kernel attributes, and, under CUDA's lazy module loading, the
 *     load of the module that holds the scratch); make that first call
 *     before any stream capture.
 *   - The scratch's device address is looked up once per device and kept;
 *     after a cudaDeviceReset it no longer holds, so no call may follow a
 *     cudaDeviceReset in the same process.
 *   - With lazy module loading (CUDA_MODULE_LOADING=LAZY, the default since
 *     CUDA 12.2) the scratch is committed on a device only by the first call
 *     there; with eager loading, every process that loads the library
 *     commits it on every device it uses.
 *
 * Host errors: those of fa_sparse_mla_decode, and FA_ERR_SCRATCH.
 */
#define FA_NOALLOC_SCRATCH_BYTES (48u << 20)
fa_status fa_sparse_mla_decode_noalloc(const void* q, const void* kv_cache,
                                       const int* page_table, const int* topk_idx,
                                       int num_tokens, int num_heads, int topk,
                                       int num_pages, int max_pages_per_tok,
                                       float softmax_scale, void* out, float* lse,
                                       fa_stream_t stream);

/*
 * fa_merge_attn_states -- merges two partial attention results of the same
 * query rows computed over disjoint key sets, weighted by their LSEs:
 *     L = ln(e^{L_prefix} + e^{L_suffix}),
 *     O = e^{L_prefix - L} O_prefix + e^{L_suffix - L} O_suffix.
 * Defined by [flash_attn] (merge_attn_states, used by FlashAttnPrefillBackend
 * to combine the non-causal context-chunk partial with the causal
 * new-token partial; both come from fa_varlen_fwd with an lse buffer).
 *
 *   out, prefix_out, suffix_out   bf16 [total_q, num_heads, head_dim]
 *   out_lse (nullable), prefix_lse, suffix_lse   fp32 [num_heads, total_q]
 *   head_dim      multiple of 8
 * An LSE of -inf marks an empty part (weight 0); both empty gives O = 0 and
 * LSE = -inf.  out may alias neither input.
 * Host errors: FA_ERR_INVALID_ARG (null pointer, sizes, alignment),
 * FA_ERR_UNSUPPORTED (more than 2^31 rows), FA_ERR_ARCH.
 */
fa_status fa_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                               const float* prefix_lse, const void* suffix_out,
                               const float* suffix_lse, int total_q, int num_heads,
                               int head_dim, fa_stream_t stream);

/*
 * fa_get_device_status -- reads and clears the library's device status word
 * on the current device.  Synchronises the device (not for the hot path).
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT if a kernel abandoned a pipeline wait
 * since the last call, or FA_ERR_LAUNCH if the read itself failed.
 */
fa_status fa_get_device_status(void);

/*
 * fa_set_wait_limit_ns -- sets the time limit of the kernels' pipeline
 * waits for every later launch of the library in this process (all
 * devices); 0 restores the default of 4 s.  The method's pages have no
 * counterpart: it is a diagnostic and test hook.  Every wait inside the
 * kernels is bounded; when one runs out, the kernel records
 * FA_ERR_DEVICE_TIMEOUT in the device status word, the other warps of its
 * CTA give up their waits too, and the CTA lets the copies and tensor-core
 * operations it started complete, frees its tensor memory and exits (the
 * outputs of that call are undefined).  Normal waits last microseconds; a
 * limit of a few microseconds makes a long call run out on purpose, which
 * exercises that path without any fault.  Limits below 1 ms poll the
 * barriers without suspending the thread.  Always FA_OK.
 */
fa_status fa_set_wait_limit_ns(unsigned long long ns);

/* Human-readable name of a status code (static string). */
const char* fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
