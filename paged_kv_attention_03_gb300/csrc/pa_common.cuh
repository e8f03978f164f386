// pa_common.cuh - small device helpers shared by the kernels of libpa_gb300.so.
// sm_103a only.  Inline PTX for cp.async, ldmatrix and the bf16 warp MMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Device error word bits (mirrors PA_DEVERR_* of the public header).
constexpr unsigned kErrSlotRange = 0x1u;
constexpr unsigned kErrBlockRange = 0x2u;
constexpr unsigned kErrSeqRange = 0x4u;
constexpr unsigned kErrQueryLen = 0x8u;
constexpr unsigned kErrSeqlensK = 0x10u;
constexpr unsigned kErrSlotMismatch = 0x40u;

__device__ __forceinline__ void flag_error(unsigned *err, unsigned bit) {
    if (err != nullptr) atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


__device__ __forceinline__ void cp_async_16_policy(uint32_t dst, const void *src,
                                                   uint32_t src_bytes, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst),
                 "l"(src), "r"(src_bytes), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Four FP8 E4M3 codes (low byte first) -> two f16x2 words, exactly (every E4M3 value, at
// most 4 significant bits with exponents 2^-9 .. 2^8, is an f16): codes 0, 1 into lo and
// codes 2, 3 into hi.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t &lo, uint32_t &hi) {
    asm("{\n"
        ".reg .b16 a, b;\n"
        "mov.b32 {a, b}, %2;\n"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n"
        "}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    uint32_t h;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
    return h;
}

// Two bf16 (low half first) -> two f16: exact for values in the f16 normal range, rounded
// below it, clamped to +-65504 beyond it (one saturating conversion; a NaN stays NaN).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t h;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(h)
        : "f"(__uint_as_float(w & 0xffff0000u)), "f"(__uint_as_float(w << 16)));
    return h;
}

// lo += float(f16 low half of v), hi += float(f16 high half of v) (mixed-precision adds).
__device__ __forceinline__ void add_f16x2_f32(float &lo, float &hi, uint32_t v) {
    asm("{\n"
        ".reg .b16 l, h;\n"
        "mov.b32 {l, h}, %2;\n"
        "add.rn.f32.f16 %0, l, %0;\n"
        "add.rn.f32.f16 %1, h, %1;\n"
        "}\n"
        : "+f"(lo), "+f"(hi)
        : "r"(v));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// log2(e): logits are kept in the base-2 domain so exp() becomes exp2().
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace pa
