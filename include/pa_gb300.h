/*
 * pa_gb300.h - C ABI of the GB300 (sm_103a) paged KV-cache attention library
 * (libpa_gb300.so).
 *
 * Three operations, each on one GPU and asynchronous on the caller's stream:
 *
 *   pa_store_kvcache   write new K/V rows into the paged cache through slot_mapping
 *   pa_decode          one query per sequence over its paged K/V (split-K + combine)
 *   pa_varlen_prefill  packed variable-length causal / chunked / sliding-window prefill
 *
 * Common conventions
 *   - Element type: every q / k / v / cache / out buffer is bf16, row-major as stated.
 *   - Cache layout: k_cache and v_cache are the two halves of the
 *     [2, num_blocks, block_size, num_kv_heads, head_dim] cache ("05 Attention
 *     Backends", section 3, get_kv_cache_shape; "MinivLLM API docs - Attention",
 *     paged_attention_decode), i.e. each is [num_blocks, block_size, num_kv_heads,
 *     head_dim] with head_dim contiguous.  They may be two separate allocations.
 *   - block_table: [num_seqs, max_num_blocks] int32, row-contiguous; entry (i, j) is
 *     the physical block of logical block j of sequence i; entries past
 *     ceil(seq_len / block_size) are never read and may be -1.
 *   - seq_lens[i]: keys of sequence i in the cache, INCLUDING the tokens of this step
 *     (seq_len = context_len + query_len, "05 Attention Backends", section 4).
 *   - GQA: query head h uses kv head h / (num_heads / num_kv_heads)
 *     ("vllm-npu 0.4.2, torch_sdpa.py", TorchSDPABackendImpl, num_queries_per_kv).
 *   - Mask: the query_len queries of a sequence are its LAST query_len positions
 *     (bottom-right causal alignment); with sliding_window = w > 0 a query at
 *     position p sees keys p-w+1 .. p (w keys, its own included); w <= 0 means no
 *     window ("transformers continuous_batching/input_ouputs.py",
 *     build_attention_mask, and "vllm-npu 0.4.2, torch_sdpa.py",
 *     _make_sliding_window_bias).
 *   - scale is the final logit scale (normally 1/sqrt(head_dim)).
 *   - Arithmetic: bf16 operands, fp32 accumulation, bf16 output (round to nearest).
 *   - Ownership: the caller owns every buffer (inputs, outputs, the cache and any
 *     workspace).  The library allocates no device memory on these calls and keeps
 *     no pointer after a call returns.
 *   - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work; inputs must stay valid until it finishes.
 *   - Errors: argument errors are found on the host before anything is launched and
 *     return PA_ERR_INVALID_ARG / PA_ERR_UNSUPPORTED; a failed launch returns
 *     PA_ERR_CUDA.  Conditions only visible on the device (a slot or block index out
 *     of range, seq_len larger than the declared maximum, query_len > seq_len) never
 *     make a kernel touch memory outside its buffers: the offending row is skipped or
 *     zero-filled and a bit is OR-ed into a per-device error word that
 *     pa_read_device_error returns.  Nothing throws across this ABI.
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shapes, misalignment */
    PA_ERR_UNSUPPORTED = 2, /* valid but not built: head_dim, block_size, group size */
    PA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    PA_ERR_DEVICE_CHECK = 4 /* pa_read_device_error found device-side check bits set */
} pa_status;

/* Bits of the device error word (see pa_read_device_error). */
#define PA_DEVERR_SLOT_RANGE 0x1u  /* store: slot >= num_blocks * block_size (row skipped) */
#define PA_DEVERR_BLOCK_RANGE 0x2u /* block_table entry outside [0, num_blocks) (zero-filled) */
#define PA_DEVERR_SEQ_RANGE 0x4u   /* seq_len > max_num_blocks*block_size or > max_seq_len */
#define PA_DEVERR_QUERY_LEN 0x8u   /* prefill: query_len > seq_len, or > max_seqlen_q */
#define PA_DEVERR_SEQLENS_K 0x10u  /* prefill: cu_seqlens_k differences disagree with seq_lens */
#define PA_DEVERR_TIMEOUT 0x20u    /* a pipeline wait gave up (internal error; output undefined) */
#define PA_DEVERR_SLOT_MISMATCH 0x40u /* fused store: slot_mapping[t] >= 0 is not the cache row
                                         of token t's own position (row still written) */

/* Human-readable name of a status code (static storage). */
const char *pa_status_string(pa_status status);

/* Library version, e.g. "pa_gb300 0.1 sm_103a". */
const char *pa_version(void);

/*
 * CUDA error text behind the most recent PA_ERR_CUDA returned on the calling host
 * thread ("no error" if there was none).  Static storage owned by the CUDA runtime;
 * reading it clears nothing.
 */
const char *pa_last_cuda_error_string(void);

/*
 * pa_store_kvcache - "MinivLLM API docs - Attention", section store_kvcache, and
 * "05 Attention Backends", Q&A 2 (slot -> block, offset).
 *
 * For every token t in [0, num_tokens) with s = slot_mapping[t] >= 0:
 *     k_cache[s / block_size][s % block_size][:][:] = key[t][:][:]
 *     v_cache[s / block_size][s % block_size][:][:] = value[t][:][:]
 * Negative slots (padding, -1 on the page) are skipped.  Bit-exact copy.
 *
 *   key, value    [num_tokens, num_kv_heads, head_dim] bf16, device, 16-byte aligned
 *   k_cache/v_cache [num_blocks, block_size, num_kv_heads, head_dim] bf16, device,
 *                 16-byte aligned
 *   slot_mapping  [num_tokens] int32, device
 * Requires num_kv_heads * head_dim to be a multiple of 8.  Slots >= num_blocks *
 * block_size are skipped and flagged PA_DEVERR_SLOT_RANGE.  Two tokens mapped to the
 * same slot in one call leave either one's row (undefined which).
 */
pa_status pa_store_kvcache(const void *key, const void *value, void *k_cache, void *v_cache,
                           const int32_t *slot_mapping, int64_t num_tokens,
                           int64_t num_blocks, int block_size, int num_kv_heads,
                           int head_dim, void *stream);

/*
 * Split-K planning for pa_decode.  The KV range of each (sequence, kv-head group)
 * is cut into at most `num_splits` slices processed by separate CTAs and merged by
 * a log-sum-exp combine.  pa_decode_num_splits returns the slice count pa_decode
 * will use for these arguments (num_splits <= 0 asks for the automatic choice);
 * pa_decode_workspace_size returns the workspace bytes pa_decode needs for them
 * (0 when one slice suffices).  Both return 0 for invalid arguments.
 */
int pa_decode_num_splits(int batch, int num_heads, int num_kv_heads, int head_dim,
                         int max_seq_len, int sliding_window, int num_splits);
size_t pa_decode_workspace_size(int batch, int num_heads, int num_kv_heads, int head_dim,
                                int max_seq_len, int sliding_window, int num_splits);

/*
 * pa_decode - paged attention for one new query per sequence.  "MinivLLM API docs
 * - Attention", section paged_attention_decode; "vllm-npu 0.4.2, xformers.py",
 * XFormersImpl.forward (decode branch, PagedAttention.forward_decode); the split-KV
 * merge follows "05 Attention Backends", section 7.1 (split-KV for long decode).
 *
 * For each sequence b (L = seq_lens[b]) and query head h:
 *     out[b][h] = sum_j softmax_j(scale * q[b][h] . K_j) V_j
 * over keys j in [max(0, L - w), L - 1] (all j < L without a window), K_j/V_j read
 * from kv head h / (num_heads / num_kv_heads) through block_table.  L == 0 gives a
 * zero row.
 *
 *   out           [batch, num_heads, head_dim] bf16, device (written)
 *   q             [batch, num_heads, head_dim] bf16, device, 16-byte aligned
 *   key, value, slot_mapping   optional (all NULL or all set): [batch, num_kv_heads,
 *                 head_dim] bf16 and [batch] int32, the new token of each sequence.
 *                 When set, the same launch stores them into the cache as
 *                 pa_store_kvcache would (slot < 0: skipped) before reading it: each
 *                 block that reads key L - 1 writes that row first.  This requires
 *                 slot_mapping[b] to be the cache row of position L - 1 of sequence b
 *                 (or negative), as it is when derived from block_table; another slot
 *                 is still written but raises PA_DEVERR_SLOT_MISMATCH, and the
 *                 attention then reads whatever the row of L - 1 holds.
 *   k_cache, v_cache  the paged cache (written only by that optional store)
 *   block_table   [batch, max_num_blocks] int32, device
 *   seq_lens      [batch] int32, device
 *   max_seq_len   host-side upper bound of seq_lens (sizes the split-K grid); a larger
 *                 seq_len is flagged PA_DEVERR_SEQ_RANGE and truncated
 *   num_splits    <= 0: automatic; otherwise an upper bound on the slice count
 *   workspace     device scratch of at least pa_decode_workspace_size(...) bytes,
 *                 256-byte aligned (may be NULL when that size is 0); its contents
 *                 on entry do not matter
 * Supported: head_dim in {64, 128}; block_size a power of two in [1, 1024];
 * num_heads / num_kv_heads in [1, 64]; batch <= 65535.
 */
pa_status pa_decode(void *out, const void *q, const void *key, const void *value,
                    const int32_t *slot_mapping, void *k_cache, void *v_cache,
                    const int32_t *block_table, int max_num_blocks, const int32_t *seq_lens,
                    int batch, int max_seq_len, int64_t num_blocks, int block_size,
                    int num_heads, int num_kv_heads, int head_dim, int sliding_window,
                    float scale, int num_splits, void *workspace, size_t workspace_bytes,
                    void *stream);

/*
 * pa_decode_noalloc - pa_decode for callers that cannot allocate device memory.  No page
 * the library follows defines it: this is a calling convention of this library only.
 *
 * Some callers have no way to call cudaMalloc: a plugin whose host framework hands it
 * just the tensors of the call and owns every other byte of the GPU, a binding from a
 * language without a device allocator, or a latency-critical loop that cannot pay for
 * cudaMalloc/cudaFree's implicit device-wide synchronisation.  This entry point takes
 * the same arguments as pa_decode minus the workspace and computes the same result;
 * its split-K scratch is a fixed PA_NOALLOC_SCRATCH_BYTES array compiled into the
 * library, which every GPU that loads the library holds until the process exits.
 *
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   - Set-up: the first call on a device (with that device current) looks up the
 *     array's device address once; make that first call before any stream capture.
 *   - Limit: returns PA_ERR_UNSUPPORTED, launching nothing, when the split-K
 *     workspace these arguments need (pa_decode_workspace_size) exceeds
 *     PA_NOALLOC_SCRATCH_BYTES; lower num_splits or the batch to fit.
 *   - Sharing: all calls on a device share the one array and it keeps the last call's
 *     partials.  Nothing in it needs to start at zero, but two calls that can overlap
 *     on the GPU (different streams without ordering between them) race on it: order
 *     them, or use pa_decode with a workspace per stream.
 */
#define PA_NOALLOC_SCRATCH_BYTES (16u << 20)
pa_status pa_decode_noalloc(void *out, const void *q, const void *key, const void *value,
                            const int32_t *slot_mapping, void *k_cache, void *v_cache,
                            const int32_t *block_table, int max_num_blocks,
                            const int32_t *seq_lens, int batch, int max_seq_len,
                            int64_t num_blocks, int block_size, int num_heads,
                            int num_kv_heads, int head_dim, int sliding_window, float scale,
                            int num_splits, void *stream);

/*
 * FP8 E4M3 KV cache.  "vllm-npu 0.4.2 wheel diff", torch_sdpa.py / xformers.py: with an
 * fp8 cache the cache write (write_to_paged_cache) and paged attention
 * (forward_decode) take one kv_scale.  Reading taken: the cache holds E4M3 codes
 * ("fn": no infinities, largest 448) of x / kv_scale -- the division in fp32, then
 * round to nearest even, finite values beyond 448 saturating -- and attention reads
 * code * kv_scale.  The caches are [num_blocks, block_size, num_kv_heads, head_dim]
 * bytes; everything else is as pa_store_kvcache / pa_decode (bf16 q, key, value, out).
 *
 * pa_store_kvcache_fp8: the store; num_kv_heads * head_dim must be a multiple of 16.
 * pa_decode_fp8: the decode (the new tokens, when given, are stored the same way inside
 *     the launch); workspace as pa_decode_workspace_size.  kv_scale > 0.
 */
pa_status pa_store_kvcache_fp8(const void *key, const void *value, void *k_cache,
                               void *v_cache, const int32_t *slot_mapping, int64_t num_tokens,
                               int64_t num_blocks, int block_size, int num_kv_heads,
                               int head_dim, float kv_scale, void *stream);
pa_status pa_decode_fp8(void *out, const void *q, const void *key, const void *value,
                        const int32_t *slot_mapping, void *k_cache, void *v_cache,
                        const int32_t *block_table, int max_num_blocks, const int32_t *seq_lens,
                        int batch, int max_seq_len, int64_t num_blocks, int block_size,
                        int num_heads, int num_kv_heads, int head_dim, int sliding_window,
                        float scale, float kv_scale, int num_splits, void *workspace,
                        size_t workspace_bytes, void *stream);

/*
 * pa_decode_state - the partial result of pa_decode over a part of each sequence's keys.
 * "05 Attention Backends", section 7.1 (split-KV: each slice of a long context gives a
 * partial result that is merged afterwards) and section 8 (cascade attention: a shared
 * prefix and each request's suffix are attended separately and combined).
 *
 * Same keys as pa_decode (window included), restricted to j >= key_begin[b].  For each
 * (b, h) it writes the normalised row
 *     state[b][h] = sum_j e^{s_j} V_j / sum_j e^{s_j},   s_j = scale * q[b][h] . K_j,
 * and lse[b][h] = ln sum_j e^{s_j}; with no key left: a zero row and lse = -inf.
 * Partial results of disjoint key sets merge with pa_merge_states.
 *
 *   state      [batch, num_heads, head_dim] fp32, device, 16-byte aligned (written)
 *   lse        [batch, num_heads] fp32, device (written)
 *   key_begin  [batch] int32, device, or NULL (0): first key position to attend
 *   workspace  at least pa_decode_state_workspace_size(...) bytes, 256-byte aligned
 * Other arguments, limits and errors as pa_decode (no new-token store here).
 */
size_t pa_decode_state_workspace_size(int batch, int num_heads, int num_kv_heads, int head_dim,
                                      int max_seq_len, int sliding_window, int num_splits);
pa_status pa_decode_state(float *state, float *lse, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_table, int max_num_blocks,
                          const int32_t *seq_lens, const int32_t *key_begin, int batch,
                          int max_seq_len, int64_t num_blocks, int block_size, int num_heads,
                          int num_kv_heads, int head_dim, int sliding_window, float scale,
                          int num_splits, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * pa_merge_states - merge partial results of the same rows ("05 Attention Backends",
 * sections 7.1 and 8; the split-KV combine of pa_decode, exposed).  For each row i:
 *     lse_i = ln sum_r e^{lses[r][i]},   o_i = sum_r e^{lses[r][i] - lse_i} states[r][i]
 * Parts with lse = -inf are absent; a row with no part gives zeros and lse = -inf.
 *
 *   out        [rows, head_dim] bf16, device, 16-byte aligned, or NULL
 *   out_state  [rows, head_dim] fp32, device, 16-byte aligned, or NULL
 *   out_lse    [rows] fp32, device, or NULL (at least one of the three is set)
 *   states     [num_states, rows, head_dim] fp32, device, 16-byte aligned
 *   lses       [num_states, rows] fp32, device
 * A row is one (token, head) pair: rows = tokens * num_heads.  head_dim in {64, 128}.
 * Asynchronous on `stream`; no allocation.
 */
pa_status pa_merge_states(void *out, float *out_state, float *out_lse, const float *states,
                          const float *lses, int num_states, int64_t rows, int head_dim,
                          void *stream);

/*
 * pa_cascade_decode - decode for a batch whose requests share a cached prefix: the
 * shared keys are attended once for all requests, each request's own keys apart, and
 * the two merged.  "05 Attention Backends", section 8 and Q&A 4 (cascade attention:
 * when the requests of a batch share a long prefix, every query attends the one copy
 * of the prefix K/V, each request attends its own suffix, and the results combine;
 * mathematically equivalent, the prefix read once).
 *
 * Same result as pa_decode (same arguments, window included, no new-token store) when
 * the first prefix_len / block_size entries of every row of block_table are equal.
 * The prefix runs on the tensor cores with the requests' query heads as the rows (one
 * read of each prefix page per 2 x 128 query rows), the suffix as pa_decode_state from
 * key prefix_len, and pa_merge_states combines them.
 *
 *   prefix_len  shared keys, a multiple of block_size, <= every seq_len (use
 *               pa_common_prefix_blocks(...) * block_size); 0 gives plain decode
 *   workspace   at least pa_cascade_decode_workspace_size(...) bytes, 256-byte aligned
 * Supported: head_dim in {64, 128}; block_size a power of two in [16, 256];
 * num_heads / num_kv_heads <= 64; scale > 0.
 */
size_t pa_cascade_decode_workspace_size(int batch, int num_heads, int num_kv_heads,
                                        int head_dim, int max_seq_len, int prefix_len,
                                        int sliding_window);
pa_status pa_cascade_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_table, int max_num_blocks,
                            const int32_t *seq_lens, int batch, int max_seq_len, int prefix_len,
                            int64_t num_blocks, int block_size, int num_heads, int num_kv_heads,
                            int head_dim, int sliding_window, float scale, void *workspace,
                            size_t workspace_bytes, void *stream);

/*
 * pa_common_prefix_blocks - host-side scan ("05 Attention Backends", Q&A 4: after the
 * scheduler has fixed the batch it scans the requests' block tables for the longest
 * common prefix of blocks).  Returns the largest n such that entries 0 .. n-1 are equal
 * in every row of block_table and n * block_size <= every seq_len; -1 on invalid
 * arguments.  block_table [batch, max_num_blocks] and seq_lens [batch] are HOST
 * pointers.
 */
int pa_common_prefix_blocks(const int32_t *block_table, int batch, int max_num_blocks,
                            const int32_t *seq_lens, int block_size);

/*
 * pa_varlen_prefill - packed variable-length causal / chunked prefill over the
 * paged cache.  "MinivLLM API docs - Attention", section flash_attention_prefill
 * (varlen packing by cu_seqlens, causal, GQA); "vllm-npu 0.4.2, xformers.py",
 * XFormersImpl.forward (forward_prefix with a cached context, sliding window);
 * "05 Attention Backends", section 5 (flash_attn_varlen_func with cu_seqlens_q,
 * seqused_k, block_table); mask as build_attention_mask.
 *
 * Sequence i owns query rows [cu_seqlens_q[i], cu_seqlens_q[i+1]) of q and out
 * (sq_i rows) and sk_i keys in the cache (sk_i = seq_lens[i], or
 * cu_seqlens_k[i+1] - cu_seqlens_k[i] when seq_lens is NULL); sq_i <= sk_i.  Row r
 * is the query at absolute position p = sk_i - sq_i + r and attends keys
 * [max(0, p - w + 1), p] (all keys <= p without a window).  sq_i == 1 rows are
 * legal, so a mixed prefill + decode batch may be passed as one call; when seq_lens is
 * given, those sequences run on the decode kernel within the call (no workspace needed)
 * while the tensor-core kernel takes the rest.  The decode kernel then runs at the same
 * time, on the SMs the tensor-core kernel's items leave free; the call's work completes
 * (in stream order) only after both kernels have finished.
 *
 *   out           [total_q, num_heads, head_dim] bf16, device (written)
 *   q             [total_q, num_heads, head_dim] bf16, device, 16-byte aligned
 *   key, value, slot_mapping   optional (all NULL or all set): [total_q, num_kv_heads,
 *                 head_dim] bf16 and [total_q] int32; stored first, as pa_store_kvcache
 *   cu_seqlens_q  [num_seqs + 1] int32, device, non-decreasing, cu_seqlens_q[0] == 0,
 *                 cu_seqlens_q[num_seqs] == total_q
 *   cu_seqlens_k  [num_seqs + 1] int32 or NULL; when both it and seq_lens are given,
 *                 seq_lens is used and a disagreement is flagged PA_DEVERR_SEQLENS_K
 *   seq_lens      [num_seqs] int32 or NULL (not both NULL)
 *   block_table   [num_seqs, max_num_blocks] int32, device
 *   max_seqlen_q  host-side upper bound of sq_i (sizes the grid); larger is flagged
 *   max_seqlen_k  host-side upper bound of sk_i; larger is flagged
 * scale must be positive and finite (PA_ERR_INVALID_ARG otherwise).
 * Supported: head_dim in {64, 128}; block_size a power of two in [16, 256];
 * num_heads / num_kv_heads in [1, 128]; num_seqs <= 65535; num_blocks * block_size and
 * total_q below 2^31.
 */
pa_status pa_varlen_prefill(void *out, const void *q, const void *key, const void *value,
                            const int32_t *slot_mapping, void *k_cache, void *v_cache,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            const int32_t *seq_lens, const int32_t *block_table,
                            int max_num_blocks, int num_seqs, int total_q, int max_seqlen_q,
                            int max_seqlen_k, int64_t num_blocks, int block_size,
                            int num_heads, int num_kv_heads, int head_dim,
                            int sliding_window, float scale, void *stream);

/*
 * pa_varlen_prefill_fp8 - pa_varlen_prefill over an FP8 E4M3 cache (the reading of the
 * FP8 block above: the caches hold codes of x / kv_scale, attention reads code *
 * kv_scale).  "05 Attention Backends", section 5: the backend views the cache as FP8 and
 * hands that view to the one varlen call that serves prefill and decode rows.
 * Arguments as pa_varlen_prefill, with k_cache / v_cache [num_blocks, block_size,
 * num_kv_heads, head_dim] bytes, key / value (optional) stored as pa_store_kvcache_fp8,
 * and kv_scale > 0 finite.  The products run in f16 (every E4M3 value is an f16; q is
 * rounded to f16 once, exactly for |q| in [2^-14, 65504], clamped beyond 65504; the
 * softmax weights are f16).  Supported: head_dim 128 (others: PA_ERR_UNSUPPORTED);
 * single-row sequences go to the FP8 decode kernel as in pa_varlen_prefill.
 */
pa_status pa_varlen_prefill_fp8(void *out, const void *q, const void *key, const void *value,
                                const int32_t *slot_mapping, void *k_cache, void *v_cache,
                                const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                const int32_t *seq_lens, const int32_t *block_table,
                                int max_num_blocks, int num_seqs, int total_q, int max_seqlen_q,
                                int max_seqlen_k, int64_t num_blocks, int block_size,
                                int num_heads, int num_kv_heads, int head_dim,
                                int sliding_window, float scale, float kv_scale, void *stream);

/*
 * pa_read_device_error - synchronise `stream`, then return in *flags the device
 * error word of the current device (PA_DEVERR_* bits OR-ed by every launch since it
 * was last cleared) and clear it when `clear` is non-zero.  Returns PA_OK when no
 * bit is set, PA_ERR_DEVICE_CHECK when some bit is set, PA_ERR_CUDA on a CUDA
 * failure.  flags may be NULL.
 */
pa_status pa_read_device_error(void *stream, uint32_t *flags, int clear);

/*
 * pa_debug_prefill_stall - testing aid for the device-side failure detection; the
 * pages have no counterpart.  Every wait inside the prefill kernel (pa_varlen_prefill,
 * the prefix part of pa_cascade_decode) gives up after a time limit, raises
 * PA_DEVERR_TIMEOUT, lets the copies and products it issued land, frees its tensor
 * memory and returns, so the context stays usable.
 *   stall != 0: later prefill launches of this process hand out no work item, so the
 *               first wait of every role runs out while nothing is in flight.
 *   wait_limit_ns: the limit of every wait of later launches (0: the default 2 s).
 * pa_debug_prefill_stall(0, 0) restores normal launches.  The setting is process-wide
 * and read when a launch is made (not synchronised with launches on other threads).
 * Returns PA_OK.
 */
pa_status pa_debug_prefill_stall(int stall, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_H */
