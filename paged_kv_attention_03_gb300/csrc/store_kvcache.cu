// store_kvcache.cu - scatter of new K/V rows into the paged cache.
//
// "MinivLLM API docs - Attention", section store_kvcache: token t with slot
// s = slot_mapping[t] >= 0 lands in block s / block_size, row s % block_size; -1 is
// padding and is skipped.  With the [num_blocks, block_size, num_kv_heads, head_dim]
// layout the destination row of slot s is simply row s of a [num_slots,
// num_kv_heads * head_dim] matrix, so the whole store is a row gather->scatter.
//
// GB300 design: the page's Triton kernel runs one program per (token, kv head); here
// one thread moves one 16-byte chunk of K and the matching chunk of V (two loads in
// flight per thread, 128 consecutive threads cover one 2 KB token row), so every
// warp reads and writes 512 contiguous bytes per tensor.  Pure HBM copy: 2 x
// num_tokens x row bytes read and the same written.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

__global__ void __launch_bounds__(256)
store_kvcache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const int32_t *__restrict__ slot_mapping, int64_t num_tokens,
                     int64_t num_slots, int chunks_per_row, unsigned *err) {
    const int64_t total = num_tokens * chunks_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += stride) {
        const int64_t t = i / chunks_per_row;
        const int c = static_cast<int>(i - t * chunks_per_row);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;  // padding token
        if (slot >= num_slots) {
            if (c == 0) flag_error(err, kErrSlotRange);
            continue;
        }
        const uint4 k = __ldcs(key + i);
        const uint4 v = __ldcs(value + i);
        const int64_t dst = slot * chunks_per_row + c;
        k_cache[dst] = k;
        v_cache[dst] = v;
    }
}

cudaError_t launch_store_kvcache(const StoreArgs &a, cudaStream_t stream) {
    if (a.num_tokens == 0) return cudaSuccess;
    const int chunks_per_row = a.row_elems / 8;
    const int64_t total = a.num_tokens * chunks_per_row;
    constexpr int kThreads = 256;
    int64_t blocks = (total + kThreads - 1) / kThreads;
    const int64_t max_blocks = 152LL * 64;  // grid-stride beyond ~8 waves of 8 CTAs/SM
    if (blocks > max_blocks) blocks = max_blocks;
    store_kvcache_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        static_cast<const uint4 *>(a.key), static_cast<const uint4 *>(a.value),
        static_cast<uint4 *>(a.k_cache), static_cast<uint4 *>(a.v_cache), a.slot_mapping,
        a.num_tokens, a.num_slots, chunks_per_row, a.err);
    return cudaGetLastError();
}

}  // namespace pa
