// merge_states.cu - merge partial attention results of the same rows.
//
// "vLLM learning book, 05 Attention Backends", section 7.1 (split-KV: each slice of a
// long context gives a partial result, merged afterwards) and section 8 (cascade
// attention: a shared prefix is attended once, each request's suffix separately, then
// the two are combined; mathematically equivalent).  A partial result over a key subset
// J is a normalised row o_J and lse_J = ln sum_{j in J} exp(s_j); for disjoint parts
//     lse = ln sum_r exp(lse_r),   o = sum_r exp(lse_r - lse) o_r.
// An empty part has lse = -inf and contributes nothing.
//
// One warp per row: lanes split the head dimension (float4 / float2 per lane), and the
// weights of 32 parts at a time are read in one round trip.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

template <int D>
__global__ void __launch_bounds__(128) merge_states_kernel(MergeArgs a) {
    constexpr int PER_LANE = D / 32;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= a.rows) return;
    const int R = a.num_states;
    float M = -INFINITY;
    for (int r0 = 0; r0 < R; r0 += 32) {
        const int r = r0 + lane;
        if (r < R) M = fmaxf(M, a.lses[static_cast<int64_t>(r) * a.rows + row]);
    }
    M = warp_max(M);
    float acc[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        for (int r0 = 0; r0 < R; r0 += 32) {
            const int r = r0 + lane;
            // exp(lse_r - M) as 2^((lse_r - M) log2 e); an empty part gives 0.
            const float wl =
                r < R ? exp2f((a.lses[static_cast<int64_t>(r) * a.rows + row] - M) * kLog2e)
                      : 0.f;
            wsum += wl;
            const int n = min(32, R - r0);
            for (int k = 0; k < n; ++k) {
                const float w = __shfl_sync(0xffffffffu, wl, k);
                const float *src =
                    a.states + (static_cast<int64_t>(r0 + k) * a.rows + row) * D + lane * PER_LANE;
                if constexpr (PER_LANE == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    acc[0] += w * v.x;
                    acc[1] += w * v.y;
                    acc[2] += w * v.z;
                    acc[3] += w * v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    acc[0] += w * v.x;
                    acc[1] += w * v.y;
                }
            }
        }
        wsum = warp_sum(wsum);
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] *= inv;
    if (a.out_state != nullptr) {
        float *dst = a.out_state + row * D + lane * PER_LANE;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) dst[i] = acc[i];
    }
    if (a.out_lse != nullptr && lane == 0)
        a.out_lse[row] = M == -INFINITY ? -INFINITY : M + logf(wsum);
    if (a.out != nullptr) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(a.out) + row * D + lane * PER_LANE;
#pragma unroll
        for (int i = 0; i < PER_LANE; i += 2)
            *reinterpret_cast<__nv_bfloat162 *>(dst + i) = __floats2bfloat162_rn(acc[i], acc[i + 1]);
    }
}

}  // namespace

cudaError_t launch_merge_states(const MergeArgs &a, cudaStream_t stream) {
    if (a.rows == 0) return cudaSuccess;
    const int64_t blocks = (a.rows + 3) / 4;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    switch (a.head_dim) {
        case 64: merge_states_kernel<64><<<static_cast<unsigned>(blocks), 128, 0, stream>>>(a); break;
        case 128: merge_states_kernel<128><<<static_cast<unsigned>(blocks), 128, 0, stream>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace pa
