// pa_api.cu - the extern "C" boundary of libpa_gb300.so (declared in pa_gb300.h).
//
// Host-side argument validation, the per-device error word, and dispatch to the
// launchers.  Nothing here allocates device memory.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "pa_gb300.h"
#include "pa_internal.h"

namespace pa {
// Last CUDA error behind a PA_ERR_CUDA, per host thread.
static thread_local cudaError_t t_last_cuda_error = cudaSuccess;

pa_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return PA_OK;
    t_last_cuda_error = e;
    return PA_ERR_CUDA;
}

const char *last_cuda_error_string() { return cudaGetErrorString(t_last_cuda_error); }
}  // namespace pa

namespace {

// One error word per device: kernels OR PA_DEVERR_* bits into it.
__device__ unsigned int g_pa_device_error;

constexpr int kMaxDevices = 64;
std::atomic<unsigned *> g_err_ptr[kMaxDevices];
std::mutex g_err_mutex;

// Device address of this device's error word (looked up once per device).
unsigned *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned *p = g_err_ptr[dev].load(std::memory_order_acquire);
    if (p != nullptr) return p;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    p = g_err_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_pa_device_error) != cudaSuccess) return nullptr;
        p = static_cast<unsigned *>(addr);
        g_err_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
bool supported_head_dim(int d) { return d == 64 || d == 128; }

pa_status from_cuda(cudaError_t e) { return pa::cuda_status(e); }

// Store-argument checks shared by the three entry points.
pa_status check_store(const void *key, const void *value, const void *k_cache,
                      const void *v_cache, const int32_t *slot_mapping, int64_t num_tokens,
                      int64_t num_blocks, int block_size, int num_kv_heads, int head_dim) {
    if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if ((static_cast<int64_t>(num_kv_heads) * head_dim) % 8 != 0) return PA_ERR_UNSUPPORTED;
    if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

pa_status run_store(const void *key, const void *value, void *k_cache, void *v_cache,
                    const int32_t *slot_mapping, int64_t num_tokens, int64_t num_blocks,
                    int block_size, int num_kv_heads, int head_dim, cudaStream_t stream) {
    pa::StoreArgs a{};
    a.key = key;
    a.value = value;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.slot_mapping = slot_mapping;
    a.num_tokens = num_tokens;
    a.num_slots = num_blocks * block_size;
    a.row_elems = num_kv_heads * head_dim;
    a.err = device_error_word();
    return from_cuda(pa::launch_store_kvcache(a, stream));
}

}  // namespace

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE_CHECK: return "PA_ERR_DEVICE_CHECK";
    }
    return "PA_ERR_UNKNOWN";
}

const char *pa_version(void) { return "pa_gb300 0.1 sm_103a"; }

const char *pa_last_cuda_error_string(void) { return pa::last_cuda_error_string(); }

pa_status pa_store_kvcache(const void *key, const void *value, void *k_cache, void *v_cache,
                           const int32_t *slot_mapping, int64_t num_tokens,
                           int64_t num_blocks, int block_size, int num_kv_heads,
                           int head_dim, void *stream) {
    const pa_status st = check_store(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                     num_blocks, block_size, num_kv_heads, head_dim);
    if (st != PA_OK || num_tokens == 0) return st;
    return run_store(key, value, k_cache, v_cache, slot_mapping, num_tokens, num_blocks,
                     block_size, num_kv_heads, head_dim, static_cast<cudaStream_t>(stream));
}

int pa_decode_num_splits(int batch, int num_heads, int num_kv_heads, int head_dim,
                         int max_seq_len, int sliding_window, int num_splits) {
    pa::DecodePlan plan;
    if (!pa::plan_decode(batch, num_heads, num_kv_heads, head_dim, max_seq_len, sliding_window,
                         num_splits, &plan))
        return 0;
    return plan.num_splits;
}

size_t pa_decode_workspace_size(int batch, int num_heads, int num_kv_heads, int head_dim,
                                int max_seq_len, int sliding_window, int num_splits) {
    pa::DecodePlan plan;
    if (!pa::plan_decode(batch, num_heads, num_kv_heads, head_dim, max_seq_len, sliding_window,
                         num_splits, &plan))
        return 0;
    return pa::decode_workspace_bytes(batch, num_heads, head_dim, plan);
}

// pa_decode and pa_decode_state: out (bf16) or state_o / state_lse (partial state).
static pa_status decode_impl(void *out, float *state_o, float *state_lse,
                             const int32_t *key_begin, const void *q, const void *key,
                             const void *value, const int32_t *slot_mapping, void *k_cache,
                             void *v_cache, const int32_t *block_table, int max_num_blocks,
                             const int32_t *seq_lens, int batch, int max_seq_len,
                             int64_t num_blocks, int block_size, int num_heads,
                             int num_kv_heads, int head_dim, int sliding_window, float scale,
                             int num_splits, void *workspace, size_t workspace_bytes,
                             void *stream, int fp8 = 0, float kv_scale = 1.f) {
    const bool state = state_o != nullptr || state_lse != nullptr;
    if (fp8 && (!(kv_scale > 0.f) || !(kv_scale < 3.0e38f))) return PA_ERR_INVALID_ARG;
    if (batch < 0 || max_seq_len < 0 || num_blocks < 0 || max_num_blocks < 0 ||
        num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
    if (!is_pow2(block_size) || block_size > 1024) return PA_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 64) return PA_ERR_UNSUPPORTED;
    if (batch > 65535) return PA_ERR_UNSUPPORTED;  // one grid row per sequence
    const bool has_new = key || value || slot_mapping;
    if (has_new && !(key && value && slot_mapping)) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (state ? !(state_o && state_lse) : !out) return PA_ERR_INVALID_ARG;
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
    if ((out && !aligned16(out)) || (state_o && !aligned16(state_o)) || !aligned16(q) ||
        !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    if (max_seq_len > 0 && max_num_blocks == 0) return PA_ERR_INVALID_ARG;
    pa::DecodePlan plan;
    if (!pa::plan_decode(batch, num_heads, num_kv_heads, head_dim, max_seq_len, sliding_window,
                         num_splits, &plan))
        return PA_ERR_INVALID_ARG;
    const size_t need = pa::decode_workspace_bytes(batch, num_heads, head_dim, plan, state);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need ||
                     (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
        return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (has_new) {
        const pa_status st = check_store(key, value, k_cache, v_cache, slot_mapping, batch,
                                         num_blocks, block_size, num_kv_heads, head_dim);
        if (st != PA_OK) return st;
    }
    pa::DecodeArgs a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.max_num_blocks = max_num_blocks;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.max_seq_len = max_seq_len;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.sliding_window = sliding_window;
    a.scale = scale;
    a.workspace = workspace;
    // The new tokens are stored by the decode launch itself.
    a.key = has_new ? key : nullptr;
    a.value = has_new ? value : nullptr;
    a.slot_mapping = has_new ? slot_mapping : nullptr;
    a.k_cache_w = k_cache;
    a.v_cache_w = v_cache;
    a.key_begin = key_begin;
    a.state_o = state_o;
    a.state_lse = state_lse;
    a.fp8 = fp8;
    a.kv_scale = kv_scale;
    a.err = device_error_word();
    return from_cuda(pa::launch_decode(a, plan, s));
}

pa_status pa_decode(void *out, const void *q, const void *key, const void *value,
                    const int32_t *slot_mapping, void *k_cache, void *v_cache,
                    const int32_t *block_table, int max_num_blocks, const int32_t *seq_lens,
                    int batch, int max_seq_len, int64_t num_blocks, int block_size,
                    int num_heads, int num_kv_heads, int head_dim, int sliding_window,
                    float scale, int num_splits, void *workspace, size_t workspace_bytes,
                    void *stream) {
    if (out == nullptr && batch > 0) return PA_ERR_INVALID_ARG;
    return decode_impl(out, nullptr, nullptr, nullptr, q, key, value, slot_mapping, k_cache,
                       v_cache, block_table, max_num_blocks, seq_lens, batch, max_seq_len,
                       num_blocks, block_size, num_heads, num_kv_heads, head_dim,
                       sliding_window, scale, num_splits, workspace, workspace_bytes, stream);
}

pa_status pa_decode_fp8(void *out, const void *q, const void *key, const void *value,
                        const int32_t *slot_mapping, void *k_cache, void *v_cache,
                        const int32_t *block_table, int max_num_blocks, const int32_t *seq_lens,
                        int batch, int max_seq_len, int64_t num_blocks, int block_size,
                        int num_heads, int num_kv_heads, int head_dim, int sliding_window,
                        float scale, float kv_scale, int num_splits, void *workspace,
                        size_t workspace_bytes, void *stream) {
    if (out == nullptr && batch > 0) return PA_ERR_INVALID_ARG;
    return decode_impl(out, nullptr, nullptr, nullptr, q, key, value, slot_mapping, k_cache,
                       v_cache, block_table, max_num_blocks, seq_lens, batch, max_seq_len,
                       num_blocks, block_size, num_heads, num_kv_heads, head_dim,
                       sliding_window, scale, num_splits, workspace, workspace_bytes, stream,
                       1, kv_scale);
}

pa_status pa_store_kvcache_fp8(const void *key, const void *value, void *k_cache,
                               void *v_cache, const int32_t *slot_mapping, int64_t num_tokens,
                               int64_t num_blocks, int block_size, int num_kv_heads,
                               int head_dim, float kv_scale, void *stream) {
    if (!(kv_scale > 0.f) || !(kv_scale < 3.0e38f)) return PA_ERR_INVALID_ARG;
    const pa_status st = check_store(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                     num_blocks, block_size, num_kv_heads, head_dim);
    if (st != PA_OK || num_tokens == 0) return st;
    if ((static_cast<int64_t>(num_kv_heads) * head_dim) % 16 != 0) return PA_ERR_UNSUPPORTED;
    pa::StoreArgs a{};
    a.key = key;
    a.value = value;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.slot_mapping = slot_mapping;
    a.num_tokens = num_tokens;
    a.num_slots = num_blocks * block_size;
    a.row_elems = num_kv_heads * head_dim;
    a.err = device_error_word();
    return from_cuda(pa::launch_store_kvcache_fp8(a, kv_scale, static_cast<cudaStream_t>(stream)));
}

size_t pa_decode_state_workspace_size(int batch, int num_heads, int num_kv_heads, int head_dim,
                                      int max_seq_len, int sliding_window, int num_splits) {
    pa::DecodePlan plan;
    if (!pa::plan_decode(batch, num_heads, num_kv_heads, head_dim, max_seq_len, sliding_window,
                         num_splits, &plan))
        return 0;
    return pa::decode_workspace_bytes(batch, num_heads, head_dim, plan, true);
}

pa_status pa_decode_state(float *state, float *lse, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_table, int max_num_blocks,
                          const int32_t *seq_lens, const int32_t *key_begin, int batch,
                          int max_seq_len, int64_t num_blocks, int block_size, int num_heads,
                          int num_kv_heads, int head_dim, int sliding_window, float scale,
                          int num_splits, void *workspace, size_t workspace_bytes,
                          void *stream) {
    if (batch > 0 && (state == nullptr || lse == nullptr)) return PA_ERR_INVALID_ARG;
    return decode_impl(nullptr, state, lse, key_begin, q, nullptr, nullptr, nullptr,
                       const_cast<void *>(k_cache), const_cast<void *>(v_cache), block_table,
                       max_num_blocks, seq_lens, batch, max_seq_len, num_blocks, block_size,
                       num_heads, num_kv_heads, head_dim, sliding_window, scale, num_splits,
                       workspace, workspace_bytes, stream);
}

// Split-K plan of the cascade's suffix part: its keys start at prefix_len, so the splits
// only have to cover the longest suffix.
static bool suffix_plan(int batch, int num_heads, int num_kv_heads, int head_dim,
                        int max_seq_len, int prefix_len, int sliding_window,
                        pa::DecodePlan *plan) {
    const int span = max_seq_len - prefix_len > 1 ? max_seq_len - prefix_len : 1;
    return pa::plan_decode(batch, num_heads, num_kv_heads, head_dim, span, sliding_window, 0,
                           plan);
}

// Cascade workspace: the prefix splits' parts ([rows, head_dim] fp32 and [rows] lse each),
// then the suffix decode's own split-K workspace (its combine merges the prefix parts).
struct CascadeLayout {
    int n_splits = 0, chunk_tiles = 1;
    size_t states = 0, lses = 0, decode_ws = 0, decode_need = 0, total = 0;
};

static bool cascade_layout(int batch, int num_heads, int num_kv_heads, int head_dim,
                           int max_seq_len, int prefix_len, int sliding_window,
                           CascadeLayout *c) {
    pa::plan_prefix_splits(batch, num_heads, num_kv_heads, prefix_len, &c->n_splits,
                           &c->chunk_tiles);
    pa::DecodePlan plan;
    if (!suffix_plan(batch, num_heads, num_kv_heads, head_dim, max_seq_len, prefix_len,
                     sliding_window, &plan))
        return false;
    const size_t rows = static_cast<size_t>(batch) * num_heads;
    const size_t parts = static_cast<size_t>(c->n_splits) > 0 ? c->n_splits : 1;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    c->states = 0;
    c->lses = up(parts * rows * head_dim * sizeof(float));
    c->decode_ws = c->lses + up(parts * rows * sizeof(float));
    c->decode_need = pa::decode_workspace_bytes(batch, num_heads, head_dim, plan, true);
    c->total = c->decode_ws + up(c->decode_need);
    return true;
}

size_t pa_cascade_decode_workspace_size(int batch, int num_heads, int num_kv_heads,
                                        int head_dim, int max_seq_len, int prefix_len,
                                        int sliding_window) {
    if (batch <= 0 || num_heads <= 0 || num_kv_heads <= 0 || prefix_len < 0 ||
        num_heads % num_kv_heads != 0)
        return 0;
    CascadeLayout c;
    if (!cascade_layout(batch, num_heads, num_kv_heads, head_dim, max_seq_len, prefix_len,
                        sliding_window, &c))
        return 0;
    return c.total;
}

pa_status pa_cascade_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_table, int max_num_blocks,
                            const int32_t *seq_lens, int batch, int max_seq_len, int prefix_len,
                            int64_t num_blocks, int block_size, int num_heads, int num_kv_heads,
                            int head_dim, int sliding_window, float scale, void *workspace,
                            size_t workspace_bytes, void *stream) {
    if (batch < 0 || max_seq_len < 0 || num_blocks < 0 || max_num_blocks < 0 ||
        num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
        prefix_len < 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
    if (!is_pow2(block_size) || block_size < 16 || block_size > 256) return PA_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 64) return PA_ERR_UNSUPPORTED;
    if (batch > 65535) return PA_ERR_UNSUPPORTED;
    if (prefix_len % block_size != 0 || prefix_len > max_seq_len ||
        prefix_len / block_size > max_num_blocks)
        return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    CascadeLayout c;
    if (!cascade_layout(batch, num_heads, num_kv_heads, head_dim, max_seq_len, prefix_len,
                        sliding_window, &c))
        return PA_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < c.total ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    float *states = reinterpret_cast<float *>(ws + c.states);
    float *lses = reinterpret_cast<float *>(ws + c.lses);
    unsigned *err = device_error_word();
    // 1. The prefix, attended once for every request: parts 0 .. n_splits - 1.
    if (c.n_splits > 0) {
        pa::PrefixArgs pr{};
        pr.q = q;
        pr.k_cache = k_cache;
        pr.v_cache = v_cache;
        pr.block_table = block_table;  // row 0 holds the shared prefix blocks
        pr.req_lens = seq_lens;
        pr.num_req = batch;
        pr.prefix_len = prefix_len;
        pr.num_blocks = num_blocks;
        pr.block_size = block_size;
        pr.num_heads = num_heads;
        pr.num_kv_heads = num_kv_heads;
        pr.head_dim = head_dim;
        pr.sliding_window = sliding_window;
        pr.scale = scale;
        pr.st_o = states;
        pr.st_lse = lses;
        pr.n_splits = c.n_splits;
        pr.chunk_tiles = c.chunk_tiles;
        pr.err = err;
        const pa_status st = from_cuda(pa::launch_prefix_states(pr, s));
        if (st != PA_OK) return st;
    }
    // 2. Each request's suffix (keys from prefix_len on): the last part.
    pa::DecodePlan plan;
    if (!suffix_plan(batch, num_heads, num_kv_heads, head_dim, max_seq_len, prefix_len,
                     sliding_window, &plan))
        return PA_ERR_INVALID_ARG;
    pa::DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.max_num_blocks = max_num_blocks;
    a.seq_lens = seq_lens;
    a.batch = batch;
    a.max_seq_len = max_seq_len;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.sliding_window = sliding_window;
    a.scale = scale;
    a.workspace = ws + c.decode_ws;
    a.key_begin_all = prefix_len;
    // The suffix's split combine also merges the prefix parts and writes the bf16 rows.
    a.out = out;
    a.pre_o = states;
    a.pre_lse = lses;
    a.pre_parts = c.n_splits;
    // The suffix runs beside the prefix kernel, on the SMs its items leave free.
    a.after_prefill = c.n_splits > 0;
    a.err = err;
    return from_cuda(pa::launch_decode(a, plan, s));
}

int pa_common_prefix_blocks(const int32_t *block_table, int batch, int max_num_blocks,
                            const int32_t *seq_lens, int block_size) {
    if (batch < 0 || max_num_blocks < 0 || block_size <= 0) return -1;
    if (batch == 0 || block_table == nullptr || seq_lens == nullptr) return 0;
    int64_t n = max_num_blocks;
    for (int b = 0; b < batch; ++b) {
        const int64_t covered = seq_lens[b] > 0 ? seq_lens[b] / block_size : 0;  // whole blocks
        if (covered < n) n = covered;
    }
    for (int64_t i = 0; i < n; ++i) {
        const int32_t blk = block_table[i];
        for (int b = 1; b < batch; ++b) {
            if (block_table[static_cast<int64_t>(b) * max_num_blocks + i] != blk) return static_cast<int>(i);
        }
    }
    return static_cast<int>(n);
}

pa_status pa_merge_states(void *out, float *out_state, float *out_lse, const float *states,
                          const float *lses, int num_states, int64_t rows, int head_dim,
                          void *stream) {
    if (num_states <= 0 || rows < 0 || head_dim <= 0) return PA_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim)) return PA_ERR_UNSUPPORTED;
    if (rows == 0) return PA_OK;
    if (!states || !lses || (!out && !out_state && !out_lse)) return PA_ERR_INVALID_ARG;
    if (!aligned16(states) || (out && !aligned16(out)) || (out_state && !aligned16(out_state)))
        return PA_ERR_INVALID_ARG;
    pa::MergeArgs a{};
    a.out = out;
    a.out_state = out_state;
    a.out_lse = out_lse;
    a.states = states;
    a.lses = lses;
    a.num_states = num_states;
    a.rows = rows;
    a.head_dim = head_dim;
    return from_cuda(pa::launch_merge_states(a, static_cast<cudaStream_t>(stream)));
}

namespace {

// pa_varlen_prefill and pa_varlen_prefill_fp8: argument checks, the optional store of the
// new tokens, then the launch.
pa_status varlen_prefill(void *out, const void *q, const void *key, const void *value,
                         const int32_t *slot_mapping, void *k_cache, void *v_cache,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                         const int32_t *seq_lens, const int32_t *block_table, int max_num_blocks,
                         int num_seqs, int total_q, int max_seqlen_q, int max_seqlen_k,
                         int64_t num_blocks, int block_size, int num_heads, int num_kv_heads,
                         int head_dim, int sliding_window, float scale, void *stream, bool fp8,
                         float kv_scale) {
    if (num_seqs < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
        num_blocks < 0 || max_num_blocks < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (max_seqlen_q > max_seqlen_k) return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !(scale < 3.0e38f)) return PA_ERR_INVALID_ARG;  // folded into exp2
    if (fp8 && (!(kv_scale > 0.f) || !(kv_scale < 3.0e38f))) return PA_ERR_INVALID_ARG;
    if (!supported_head_dim(head_dim) || (fp8 && head_dim != 128)) return PA_ERR_UNSUPPORTED;
    if (!is_pow2(block_size) || block_size < 16 || block_size > 256) return PA_ERR_UNSUPPORTED;
    if (num_heads / num_kv_heads > 128) return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535) return PA_ERR_UNSUPPORTED;  // one grid row per sequence
    if (num_blocks * block_size > 0x7fffff00LL || total_q > 0x7fffff00) return PA_ERR_UNSUPPORTED;
    const bool has_new = key || value || slot_mapping;
    if (has_new && !(key && value && slot_mapping)) return PA_ERR_INVALID_ARG;
    if (total_q == 0) return PA_OK;
    // With no sequence there is nothing to attend, but the new tokens are still stored.
    auto store = [&]() -> pa_status {
        return fp8 ? pa_store_kvcache_fp8(key, value, k_cache, v_cache, slot_mapping, total_q,
                                          num_blocks, block_size, num_kv_heads, head_dim, kv_scale,
                                          stream)
                   : pa_store_kvcache(key, value, k_cache, v_cache, slot_mapping, total_q,
                                      num_blocks, block_size, num_kv_heads, head_dim, stream);
    };
    if (num_seqs == 0) return has_new ? store() : PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !cu_seqlens_q) return PA_ERR_INVALID_ARG;
    if (!seq_lens && !cu_seqlens_k) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    if (max_seqlen_k > 0 && max_num_blocks == 0) return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (has_new) {
        const pa_status st = store();
        if (st != PA_OK) return st;
    }
    pa::PrefillArgs a{};
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.cu_seqlens_q = cu_seqlens_q;
    a.cu_seqlens_k = cu_seqlens_k;
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.max_num_blocks = max_num_blocks;
    a.num_seqs = num_seqs;
    a.total_q = total_q;
    a.max_seqlen_q = max_seqlen_q;
    a.max_seqlen_k = max_seqlen_k;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.sliding_window = sliding_window;
    a.scale = scale;
    a.fp8 = fp8 ? 1 : 0;
    a.kv_scale = kv_scale;
    a.err = device_error_word();
    return from_cuda(pa::launch_prefill(a, s));
}

}  // namespace

pa_status pa_varlen_prefill(void *out, const void *q, const void *key, const void *value,
                            const int32_t *slot_mapping, void *k_cache, void *v_cache,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                            const int32_t *seq_lens, const int32_t *block_table,
                            int max_num_blocks, int num_seqs, int total_q, int max_seqlen_q,
                            int max_seqlen_k, int64_t num_blocks, int block_size,
                            int num_heads, int num_kv_heads, int head_dim,
                            int sliding_window, float scale, void *stream) {
    return varlen_prefill(out, q, key, value, slot_mapping, k_cache, v_cache, cu_seqlens_q,
                          cu_seqlens_k, seq_lens, block_table, max_num_blocks, num_seqs, total_q,
                          max_seqlen_q, max_seqlen_k, num_blocks, block_size, num_heads,
                          num_kv_heads, head_dim, sliding_window, scale, stream, false, 1.f);
}

pa_status pa_varlen_prefill_fp8(void *out, const void *q, const void *key, const void *value,
                                const int32_t *slot_mapping, void *k_cache, void *v_cache,
                                const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                                const int32_t *seq_lens, const int32_t *block_table,
                                int max_num_blocks, int num_seqs, int total_q, int max_seqlen_q,
                                int max_seqlen_k, int64_t num_blocks, int block_size,
                                int num_heads, int num_kv_heads, int head_dim,
                                int sliding_window, float scale, float kv_scale, void *stream) {
    return varlen_prefill(out, q, key, value, slot_mapping, k_cache, v_cache, cu_seqlens_q,
                          cu_seqlens_k, seq_lens, block_table, max_num_blocks, num_seqs, total_q,
                          max_seqlen_q, max_seqlen_k, num_blocks, block_size, num_heads,
                          num_kv_heads, head_dim, sliding_window, scale, stream, true, kv_scale);
}

pa_status pa_debug_prefill_stall(int stall, uint64_t wait_limit_ns) {
    pa::debug_prefill_stall(stall, wait_limit_ns);
    return PA_OK;
}

pa_status pa_read_device_error(void *stream, uint32_t *flags, int clear) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return from_cuda(e);
    unsigned *word = device_error_word();
    if (word == nullptr) return PA_ERR_CUDA;
    unsigned host = 0;
    e = cudaMemcpy(&host, word, sizeof host, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (clear && host != 0) {
        e = cudaMemset(word, 0, sizeof host);
        if (e != cudaSuccess) return from_cuda(e);
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return from_cuda(e);
    }
    if (flags) *flags = host;
    return host == 0 ? PA_OK : PA_ERR_DEVICE_CHECK;
}

}  // extern "C"
