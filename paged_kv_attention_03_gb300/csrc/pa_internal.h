// pa_internal.h - launcher interface between the C ABI (pa_api.cu) and the kernels.
// Arguments reaching these launchers have already been validated on the host.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <cstdint>

#include "pa_gb300.h"

namespace pa {

// ------------------------------------------------------------------ store ---
struct StoreArgs {
    const void *key;
    const void *value;
    void *k_cache;
    void *v_cache;
    const int32_t *slot_mapping;
    int64_t num_tokens;
    int64_t num_slots;  // num_blocks * block_size
    int row_elems;      // num_kv_heads * head_dim (multiple of 8)
    unsigned *err;
};
cudaError_t launch_store_kvcache(const StoreArgs &a, cudaStream_t stream);
// FP8 E4M3 cache: k_cache / v_cache are [num_slots, row_elems] bytes (row_elems % 16 == 0).
cudaError_t launch_store_kvcache_fp8(const StoreArgs &a, float kv_scale, cudaStream_t stream);

// ----------------------------------------------------------------- decode ---
// SM count the decode split plan is made for.  The plan does not query the device, so
// pa_decode_workspace_size stays a pure function of its arguments (callers size the
// workspace before any device is chosen); it is also the fallback of sm_count() when
// the device cannot be asked.
constexpr int kPlanSms = 152;

struct DecodePlan {
    int group;        // query heads per kv head
    int head_tiles;   // ceil(group / 16): 16-row MMA tiles per kv head
    int span;         // longest key range one sequence can need (tokens)
    int chunk;        // tokens per split (multiple of 16)
    int num_splits;   // ceil(span / chunk)
};
// Returns false on invalid arguments.
bool plan_decode(int batch, int num_heads, int num_kv_heads, int head_dim, int max_seq_len,
                 int sliding_window, int num_splits_request, DecodePlan *plan);
// state: the call returns partial states (always through the workspace and combine).
size_t decode_workspace_bytes(int batch, int num_heads, int head_dim, const DecodePlan &p,
                              bool state = false);

struct DecodeArgs {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_table;
    int max_num_blocks;
    const int32_t *seq_lens;
    int batch;
    int max_seq_len;
    int64_t num_blocks;
    int block_size;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int sliding_window;
    float scale;
    void *workspace;
    // Fused store of each sequence's new token (all null when not fused).
    const void *key;               // [batch, num_kv_heads, head_dim]
    const void *value;
    const int32_t *slot_mapping;   // [batch]
    void *k_cache_w;               // the caches, writable
    void *v_cache_w;
    // Partial-state output (all null for the normal bf16 output).
    const int32_t *key_begin;      // [batch] first key to attend, or null (key_begin_all)
    int key_begin_all;
    // FP8 E4M3 cache: k_cache / v_cache hold codes of x / kv_scale (one byte each).
    int fp8;
    float kv_scale;
    float *state_o;                // [batch, num_heads, head_dim]
    float *state_lse;              // [batch, num_heads]
    // Extra partial states merged into the output by the combine (the cascade's prefix
    // parts): pre_parts x [batch * num_heads] rows, normalised fp32 rows pre_o and
    // natural-log denominators pre_lse (-inf: empty).  0 parts: none.
    const float *pre_o;
    const float *pre_lse;
    int pre_parts;
    // Varlen layout (null: q / out rows are the sequences): sequence b is processed only
    // if q_rows[b + 1] - q_rows[b] == 1, with q / out row q_rows[b].
    const int32_t *q_rows;
    int total_q;                   // number of q / out rows (bounds q_rows)
    // With q_rows and no prefill launch over the batch: check every sequence's query
    // length (0..max_seqlen_q, <= seq_lens) and cu_seqlens_k against seq_lens.
    bool check_rows;
    int max_seqlen_q;
    const int32_t *cu_seqlens_k;   // may be null
    // Launch the split kernel as a programmatic dependent of the kernel before it (set
    // only right after the prefill kernel of the same call, which triggers its dependents
    // once all its CTAs are resident).  The split CTAs run beside the prefill; the grid's
    // last CTA waits for the prefill grid before it exits.
    bool after_prefill;
    unsigned *err;
};
cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream);

// ---------------------------------------------------------------- prefill ---
struct PrefillArgs {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *cu_seqlens_q;
    const int32_t *cu_seqlens_k;  // may be null
    const int32_t *seq_lens;      // may be null (then cu_seqlens_k is used)
    const int32_t *block_table;
    int max_num_blocks;
    int num_seqs;
    int total_q;
    int max_seqlen_q;
    int max_seqlen_k;
    int64_t num_blocks;
    int block_size;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int sliding_window;
    float scale;
    // FP8 E4M3 cache (head_dim 128): k_cache / v_cache hold codes of x / kv_scale.
    int fp8;
    float kv_scale;
    unsigned *err;
};
cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream);
// Testing aid behind pa_debug_prefill_stall (process-wide; read at each prefill launch).
void debug_prefill_stall(int stall, uint64_t wait_ns);

// Shared-prefix (cascade) partial states: every request's decode query against the
// prefix_len keys in the first prefix_len / block_size entries of block_table, split
// into n_splits parts of chunk_tiles 128-key tiles.
struct PrefixArgs {
    const void *q;             // [num_req, num_heads, head_dim] bf16
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_table;  // the prefix blocks (a row of the table)
    const int32_t *req_lens;     // [num_req] seq_lens (window bound)
    int num_req;
    int prefix_len;              // multiple of block_size
    int64_t num_blocks;
    int block_size;
    int num_heads;
    int num_kv_heads;
    int head_dim;
    int sliding_window;
    float scale;
    float *st_o;                 // [n_splits, num_req * num_heads, head_dim]
    float *st_lse;               // [n_splits, num_req * num_heads]
    int n_splits;
    int chunk_tiles;
    unsigned *err;
};
void plan_prefix_splits(int num_req, int num_heads, int num_kv_heads, int prefix_len,
                        int *n_splits, int *chunk_tiles);
cudaError_t launch_prefix_states(const PrefixArgs &a, cudaStream_t stream);

// ------------------------------------------------------------ merge_states ---
struct MergeArgs {
    void *out;               // [rows, head_dim] bf16, or null
    float *out_state;        // [rows, head_dim] fp32, or null
    float *out_lse;          // [rows] fp32, or null
    const float *states;     // [num_states, rows, head_dim] fp32
    const float *lses;       // [num_states, rows] fp32
    int num_states;
    int64_t rows;
    int head_dim;
};
cudaError_t launch_merge_states(const MergeArgs &a, cudaStream_t stream);

// Map a CUDA error to a pa_status, remembering it for pa_last_cuda_error_string().
pa_status cuda_status(cudaError_t e);

// Raises kernel f's dynamic shared-memory limit to `bytes` once per device (done: one bit
// per device ordinal, owned by the caller for that kernel), so launches after the first
// make no attribute call.
template <typename Kernel>
inline cudaError_t smem_limit_once(Kernel f, int bytes, std::atomic<uint64_t> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

}  // namespace pa
