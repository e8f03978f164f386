// decode_noalloc.cu - pa_decode_noalloc: paged decode whose split-K scratch lives in a
// fixed array inside this library instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory: a plugin whose host framework hands it
// only the tensors of the call and owns every other byte of the GPU, a binding from a
// language with no device allocator, or a latency-critical loop that cannot afford the
// implicit device-wide synchronisation of cudaMalloc/cudaFree.  For them this entry
// point needs nothing beyond inputs and outputs: the split-K partials go to the
// file-scope array below, which every GPU that loads the library holds until the
// process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "pa_gb300.h"
#include "pa_internal.h"

namespace {

// The shared split-K scratch: PA_NOALLOC_SCRATCH_BYTES per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mutex;

// Device address of this device's scratch array, looked up once per device with that
// device current.  The host-side symbol is only a stand-in and must never reach a kernel.
void *scratch_address(cudaError_t *err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p != nullptr) return p;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
        void *addr = nullptr;
        *err = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (*err != cudaSuccess || addr == nullptr) return nullptr;
        p = addr;
        g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void *out, const void *q, const void *key,
                                       const void *value, const int32_t *slot_mapping,
                                       void *k_cache, void *v_cache,
                                       const int32_t *block_table, int max_num_blocks,
                                       const int32_t *seq_lens, int batch, int max_seq_len,
                                       int64_t num_blocks, int block_size, int num_heads,
                                       int num_kv_heads, int head_dim, int sliding_window,
                                       float scale, int num_splits, void *stream) {
    if (batch < 0 || max_seq_len < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        head_dim <= 0 || num_heads % num_kv_heads != 0)
        return PA_ERR_INVALID_ARG;
    const size_t need = pa_decode_workspace_size(batch, num_heads, num_kv_heads, head_dim,
                                                 max_seq_len, sliding_window, num_splits);
    if (need > static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES)) return PA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (need > 0) {
        cudaError_t err = cudaSuccess;
        scratch = scratch_address(&err);
        if (scratch == nullptr) return pa::cuda_status(err != cudaSuccess ? err : cudaErrorUnknown);
    }
    // Nothing in the scratch has to start at zero: every split the combine reads is
    // written first by the same call.
    return pa_decode(out, q, key, value, slot_mapping, k_cache, v_cache, block_table,
                     max_num_blocks, seq_lens, batch, max_seq_len, num_blocks, block_size,
                     num_heads, num_kv_heads, head_dim, sliding_window, scale, num_splits,
                     scratch, need > 0 ? static_cast<size_t>(PA_NOALLOC_SCRATCH_BYTES) : 0,
                     stream);
}
