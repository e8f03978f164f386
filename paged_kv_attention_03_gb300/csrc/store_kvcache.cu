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

// FP8 E4M3 cache (the vllm-npu torch_sdpa / xformers paths pass one kv_scale to the
// cache write): each element is stored as E4M3(x / kv_scale), the division in fp32
// (correctly rounded), then round to nearest even with saturation at 448.  One thread
// turns 16 bf16 elements (32 B) of K and of V into 16 codes (16 B) each.
namespace {

__device__ __forceinline__ uint32_t quant2(uint32_t bf16x2, float kv_scale) {
    const float lo = __fdiv_rn(__uint_as_float(bf16x2 << 16), kv_scale);
    const float hi = __fdiv_rn(__uint_as_float(bf16x2 & 0xffff0000u), kv_scale);
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint4 quant16(const uint4 *src, float kv_scale) {
    const uint4 a = __ldcs(src), b = __ldcs(src + 1);
    uint4 o;
    o.x = quant2(a.x, kv_scale) | (quant2(a.y, kv_scale) << 16);
    o.y = quant2(a.z, kv_scale) | (quant2(a.w, kv_scale) << 16);
    o.z = quant2(b.x, kv_scale) | (quant2(b.y, kv_scale) << 16);
    o.w = quant2(b.z, kv_scale) | (quant2(b.w, kv_scale) << 16);
    return o;
}

}  // namespace

__global__ void __launch_bounds__(256)
store_kvcache_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                         uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                         const int32_t *__restrict__ slot_mapping, int64_t num_tokens,
                         int64_t num_slots, int chunks_per_row, float kv_scale, unsigned *err) {
    // chunks_per_row: 16-element groups per token row (one 16-byte fp8 chunk each).
    const int64_t total = num_tokens * chunks_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += stride) {
        const int64_t t = i / chunks_per_row;
        const int c = static_cast<int>(i - t * chunks_per_row);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (c == 0) flag_error(err, kErrSlotRange);
            continue;
        }
        const int64_t dst = slot * chunks_per_row + c;
        k_cache[dst] = quant16(key + 2 * i, kv_scale);
        v_cache[dst] = quant16(value + 2 * i, kv_scale);
    }
}

cudaError_t launch_store_kvcache_fp8(const StoreArgs &a, float kv_scale, cudaStream_t stream) {
    if (a.num_tokens == 0) return cudaSuccess;
    const int chunks_per_row = a.row_elems / 16;
    const int64_t total = a.num_tokens * chunks_per_row;
    constexpr int kThreads = 256;
    int64_t blocks = (total + kThreads - 1) / kThreads;
    const int64_t max_blocks = 152LL * 64;
    if (blocks > max_blocks) blocks = max_blocks;
    store_kvcache_fp8_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(
        static_cast<const uint4 *>(a.key), static_cast<const uint4 *>(a.value),
        static_cast<uint4 *>(a.k_cache), static_cast<uint4 *>(a.v_cache), a.slot_mapping,
        a.num_tokens, a.num_slots, chunks_per_row, kv_scale, a.err);
    return cudaGetLastError();
}

}  // namespace pa
