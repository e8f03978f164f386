// prefill.cu - packed variable-length causal / chunked / sliding-window prefill over the
// paged KV cache on the sm_103a tensor cores (tcgen05 + TMEM), K/V gathered by TMA.
//
// What it computes ("MinivLLM API docs - Attention", section flash_attention_prefill;
// "vllm-npu 0.4.2, xformers.py", forward_prefix; "05 Attention Backends", section 5):
// sequence i owns query rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1 (sq of them) and
// sk = seq_lens[i] keys in the cache.  Row r is the query at position p = sk - sq + r
// (bottom-right alignment, build_attention_mask) and attends keys [max(0, p-w+1), p]
// (all keys <= p without a window) of kv head h / (H / Hkv).
//
// GB300 design (the page's Triton kernel uses 32x32 or 64x64 tiles sized for ~48 KB of
// shared memory and reads contiguous K/V):
//  * One CTA per (128-row query tile, kv head, sequence).  The 128 MMA rows pack the G
//    query heads of one kv head for T = floor(128 / G) consecutive tokens (row m =
//    token m / G, head m % G), so one K/V tile feeds all heads of the group.
//  * K/V come straight from the paged cache: the TMA producer walks block_table and
//    fetches each 16-key piece of a page as one 3-D box {64 dims, 1 kv head, 16 rows}
//    with 128-byte swizzle; pieces past the sequence are loaded from an out-of-range
//    coordinate, which the TMA unit fills with zeros.
//  * S = Q K^T (M=128, N=128 keys, K=head_dim) and O += P V (M=128, N=head_dim,
//    K=128 keys) run as tcgen05.mma kind::f16 with fp32 accumulators in tensor memory:
//    S double-buffered (2 x 128 columns), O in 128 columns.
//  * Warp roles: warp 0 loads Q and K, warp 6 loads V, warp 1 issues the MMAs (one
//    thread), warps 2-5 own one accumulator row each (thread = TMEM lane) and do the
//    mask, the online softmax in base 2 (the O rescale in TMEM is skipped unless the
//    running max grows by more than 2^8), write P as bf16 to shared memory, and the
//    epilogue.
//  * Every mbarrier wait is bounded: on timeout the CTA raises an error bit, drains, frees
//    its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstring>
#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "sm100_ptx.cuh"

namespace pa {

constexpr unsigned kErrTimeout = 0x20u;

namespace {

using namespace sm100;

constexpr int BM = 128;                       // MMA rows per CTA
constexpr int BN = 128;                       // keys per KV tile
constexpr uint32_t HALF = 128u * 128u;        // [128 rows][64 bf16] = 16 KB (one swizzle span)
constexpr int NSK = 3;                        // K stages
constexpr int NSV = 2;                        // V stages
constexpr int kThreads = 224;                 // 7 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait

struct PrefillKernelParams {
    CUtensorMap tmap_q;
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    __nv_bfloat16 *out;
    const int32_t *cu_q;
    const int32_t *cu_k;
    const int32_t *seq_lens;
    const int32_t *block_table;
    int max_num_blocks;
    int num_seqs;
    int max_seqlen_q;
    int64_t seq_cap;  // max_num_blocks * block_size, capped by max_seqlen_k
    int64_t num_blocks;
    int log2_bs;
    int num_heads;
    int num_kv_heads;
    int group;
    int tok_per_tile;  // floor(128 / group)
    int window;
    float scale_log2;
    unsigned *err;
};

// Barrier indices.
enum : int {
    B_Q = 0,
    B_KFULL = 1,
    B_KEMPTY = B_KFULL + NSK,
    B_VFULL = B_KEMPTY + NSK,
    B_VEMPTY = B_VFULL + NSV,
    B_SFULL = B_VEMPTY + NSV,
    B_SFREE = B_SFULL + 2,
    B_PFULL = B_SFREE + 2,
    B_ODONE = B_PFULL + 1,
    NBARS = B_ODONE + 1
};

template <int HD>
struct Layout {
    static constexpr int NHALF = HD / 64;
    static constexpr uint32_t TILE = NHALF * HALF;  // one [128][HD] bf16 tile
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + TILE;
    static constexpr uint32_t OFF_V = OFF_K + NSK * TILE;
    static constexpr uint32_t OFF_P = OFF_V + NSV * TILE;
    static constexpr uint32_t OFF_BAR = OFF_P + 2 * HALF;  // P is [128][128 keys]
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr uint32_t BYTES = OFF_MISC + 16;
    // Request at least 116 KB so a single CTA owns an SM (and all of its TMEM).
    static constexpr uint32_t SMEM = (BYTES + 1024 > 118784u ? BYTES + 1024 : 118784u);
};

// Bounded wait by one thread.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      unsigned *err) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 31u) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            if (now - t0 > kTimeoutNs) {
                *abort_flag = 1;
                flag_error(err, kErrTimeout);
                return false;
            }
        }
    }
}

// Bounded wait by a whole warp; every lane returns the same answer.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag, unsigned *err) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((it & 31u) == 31u) {
            bool stop = *abort_flag != 0;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            stop = stop || (now - t0 > kTimeoutNs);
            if (__any_sync(0xffffffffu, stop)) {
                if ((threadIdx.x & 31) == 0) {
                    *abort_flag = 1;
                    flag_error(err, kErrTimeout);
                }
                return false;
            }
        }
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillKernelParams p) {
    using L = Layout<HD>;
    constexpr int NHALF = L::NHALF;
    constexpr int KSTEPS_S = HD / 16;   // MMAs per S tile
    constexpr int KSTEPS_O = BN / 16;   // MMAs per PV tile

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const uint32_t sQ = base + L::OFF_Q;
    const uint32_t sK = base + L::OFF_K;
    const uint32_t sV = base + L::OFF_V;
    const uint32_t sP = base + L::OFF_P;
    const uint32_t sBar = base + L::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(sb + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int kvh = blockIdx.y;
    const int qt = gridDim.x - 1 - blockIdx.x;  // longest-running tiles first
    const bool reporter = threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0;

    // ---- sequence geometry (uniform over the CTA) ----
    const int q_start = p.cu_q[seq];
    const int sq = p.cu_q[seq + 1] - q_start;
    int sk;
    if (p.seq_lens != nullptr) {
        sk = p.seq_lens[seq];
        if (p.cu_k != nullptr && reporter && p.cu_k[seq + 1] - p.cu_k[seq] != sk)
            flag_error(p.err, kErrSeqlensK);
    } else {
        sk = p.cu_k[seq + 1] - p.cu_k[seq];
    }
    if (sk < 0 || static_cast<int64_t>(sk) > p.seq_cap) {
        if (reporter) flag_error(p.err, kErrSeqRange);
        sk = sk < 0 ? 0 : static_cast<int>(p.seq_cap);
    }
    if (sq < 0 || sq > sk || sq > p.max_seqlen_q) {
        if (reporter) flag_error(p.err, kErrQueryLen);
        if (sq < 0 || sq > sk) return;
    }
    const int T = p.tok_per_tile;
    const int G = p.group;
    const int q0 = qt * T;
    if (q0 >= sq) return;
    const int rows_tok = min(T, sq - q0);
    const int p_lo = sk - sq + q0;
    const int p_hi = p_lo + rows_tok - 1;
    const int kmin = p.window > 0 ? max(0, p_lo - p.window + 1) : 0;
    const int kt0 = kmin / BN;
    const int kt1 = p_hi / BN;
    const int n_tiles = kt1 - kt0 + 1;

    // ---- set-up: barriers, tensor memory ----
    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_SFULL + s), 1);
            mbar_init(bar(B_SFREE + s), 4);
        }
        mbar_init(bar(B_PFULL), 4);
        mbar_init(bar(B_ODONE), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(base + L::OFF_MISC, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int32_t *bt_row = p.block_table + static_cast<int64_t>(seq) * p.max_num_blocks;
    const int bs_mask = (1 << p.log2_bs) - 1;
    // Cache row (slot) of the 16-key piece starting at key k0, or an out-of-range row
    // (zero fill) when the piece is past the sequence or its block index is invalid.
    auto kv_row = [&](int k0) -> int {
        if (k0 >= sk) return -16;
        const int blk = __ldg(bt_row + (k0 >> p.log2_bs));
        if (blk < 0 || blk >= p.num_blocks) {
            flag_error(p.err, kErrBlockRange);
            return -16;
        }
        return (blk << p.log2_bs) | (k0 & bs_mask);
    };

    if (warp == 0) {
        // ---------------- Q + K producer ----------------
        if (lane == 0) {
            prefetch_tmap(&p.tmap_q);
            prefetch_tmap(&p.tmap_k);
            mbar_arrive_expect_tx(bar(B_Q), static_cast<uint32_t>(G * T) * 128u * NHALF);
#pragma unroll
            for (int h = 0; h < NHALF; ++h)
                tma_load_3d(sQ + h * HALF, &p.tmap_q, h * 64, kvh * G, q_start + q0, bar(B_Q));
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % NSK;
                if (j >= NSK && !wait1(bar(B_KEMPTY + st), ((j / NSK) - 1) & 1, abort_flag, p.err))
                    break;
                const int key0 = (kt0 + j) * BN;
                mbar_arrive_expect_tx(bar(B_KFULL + st), L::TILE);
                const uint32_t dst = sK + st * L::TILE;
#pragma unroll 1
                for (int u = 0; u < BN / 16; ++u) {
                    const int row = kv_row(key0 + u * 16);
#pragma unroll
                    for (int h = 0; h < NHALF; ++h)
                        tma_load_3d(dst + h * HALF + u * 2048, &p.tmap_k, h * 64, kvh, row,
                                    bar(B_KFULL + st));
                }
            }
        }
    } else if (warp == 6) {
        // ---------------- V producer ----------------
        if (lane == 0) {
            prefetch_tmap(&p.tmap_v);
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j % NSV;
                if (j >= NSV && !wait1(bar(B_VEMPTY + st), ((j / NSV) - 1) & 1, abort_flag, p.err))
                    break;
                const int key0 = (kt0 + j) * BN;
                mbar_arrive_expect_tx(bar(B_VFULL + st), L::TILE);
                const uint32_t dst = sV + st * L::TILE;
#pragma unroll 1
                for (int u = 0; u < BN / 16; ++u) {
                    const int row = kv_row(key0 + u * 16);
#pragma unroll
                    for (int h = 0; h < NHALF; ++h)
                        tma_load_3d(dst + h * HALF + u * 2048, &p.tmap_v, h * 64, kvh, row,
                                    bar(B_VFULL + st));
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false);
            constexpr uint32_t idesc_o = idesc_bf16_f32(BM, HD, true);
            auto issue_s = [&](int j) -> bool {
                const int st = j % NSK;
                if (!wait1(bar(B_KFULL + st), (j / NSK) & 1, abort_flag, p.err)) return false;
                const int sbuf = j & 1;
                if (j >= 2 && !wait1(bar(B_SFREE + sbuf), ((j >> 1) - 1) & 1, abort_flag, p.err))
                    return false;
                tc_fence_after();
                const uint32_t kbase = sK + st * L::TILE;
#pragma unroll
                for (int k = 0; k < KSTEPS_S; ++k) {
                    const uint32_t off = (k >> 2) * HALF + (k & 3) * 32;
                    const uint64_t a = smem_desc_sw128(sQ + off, 16, 1024);
                    const uint64_t b = smem_desc_sw128(kbase + off, 16, 1024);
                    mma_bf16_ss(tmem + (sbuf ? kColS1 : kColS0), a, b, idesc_s, k > 0);
                }
                mma_commit(bar(B_SFULL + sbuf));
                mma_commit(bar(B_KEMPTY + st));
                return true;
            };
            bool ok = wait1(bar(B_Q), 0, abort_flag, p.err);
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles && !issue_s(j + 1)) break;
                const int st = j % NSV;
                if (!wait1(bar(B_PFULL), j & 1, abort_flag, p.err)) break;
                if (!wait1(bar(B_VFULL + st), (j / NSV) & 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t vbase = sV + st * L::TILE;
#pragma unroll
                for (int k = 0; k < KSTEPS_O; ++k) {
                    const uint64_t a = smem_desc_sw128(sP + (k >> 2) * HALF + (k & 3) * 32, 16, 1024);
                    const uint64_t b = smem_desc_sw128(vbase + k * 2048, HALF, 1024);
                    mma_bf16_ss(tmem + kColO, a, b, idesc_o, (j > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(bar(B_ODONE));
                mma_commit(bar(B_VEMPTY + st));
            }
        }
    } else {
        // ---------------- softmax / correction / epilogue (warps 2..5) ----------------
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
        const int tok = row / G;
        const int g = row - tok * G;
        const bool valid = tok < rows_tok;
        const int pos = sk - sq + q0 + tok;
        const float sl2 = p.scale_log2;
        const int w = p.window;
        float m_ref = -INFINITY;
        float l_sum = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int sbuf = j & 1;
            if (!wait_warp(bar(B_SFULL + sbuf), (j >> 1) & 1, abort_flag, p.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float s[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) {
                float v[32];
                tmem_ld_32x32b_x32(tmem + t_lane + (sbuf ? kColS1 : kColS0) + c * 32, v);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c * 32 + i] = v[i];
            }
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_SFREE + sbuf));

            const int key0 = (kt0 + j) * BN;
            const bool all_visible = key0 + BN - 1 <= pos && (w <= 0 || key0 >= pos - w + 1);
            float mx = -INFINITY;
            if (all_visible) {
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    s[c] *= sl2;
                    mx = fmaxf(mx, s[c]);
                }
            } else {
                const int lo = w > 0 ? pos - w + 1 : INT_MIN;
#pragma unroll
                for (int c = 0; c < BN; ++c) {
                    const int k = key0 + c;
                    const bool vis = k <= pos && k >= lo;
                    s[c] = vis ? s[c] * sl2 : -INFINITY;
                    mx = fmaxf(mx, s[c]);
                }
            }
            const float m_new = fmaxf(m_ref, mx);
            const bool need = m_new > m_ref + 8.f;
            if (j > 0) {
                // PV(j-1) must be complete: O is stable and the P buffer is free.
                if (!wait_warp(bar(B_ODONE), (j - 1) & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, need)) {
                    const float f = need ? ex2_approx(m_ref - m_new) : 1.f;
#pragma unroll 1
                    for (int c = 0; c < HD / 32; ++c) {
                        float o[32];
                        tmem_ld_32x32b_x32(tmem + t_lane + kColO + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= f;
                        tmem_st_32x32b_x32(tmem + t_lane + kColO + c * 32, o);
                    }
                    tmem_wait_st();
                    l_sum *= f;
                    if (need) m_ref = m_new;
                }
            } else {
                m_ref = m_new;
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;

            // P = 2^(s - m) as bf16 into the swizzled K-major P tile; row sum in fp32.
#pragma unroll
            for (int c8 = 0; c8 < BN / 8; ++c8) {
                float e[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) e[i] = ex2_approx(s[c8 * 8 + i] - m_use);
                uint32_t pk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    pk[i] = pack_bf16x2(e[2 * i], e[2 * i + 1]);
                    // The denominator sums the bf16 weights the MMA actually uses.
                    l_sum += __uint_as_float(pk[i] << 16) + __uint_as_float(pk[i] & 0xffff0000u);
                }
                const uint32_t addr = sP + (c8 >> 3) * HALF + row * 128 +
                                      ((((c8 & 7) ^ (row & 7))) << 4);
                st_shared_v4(addr, pk[0], pk[1], pk[2], pk[3]);
            }
            // Keys of the sequence's last, partly filled 16-key piece that lie past sk
            // are stale cache rows: zero them in the V tile so 0 * V stays 0.
            if (((sk - 1) / BN) == kt0 + j && (sk & 15) != 0) {
                const int st = j % NSV;
                if (!wait_warp(bar(B_VFULL + st), (j / NSV) & 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                const int r0 = sk - key0;               // first stale row in the tile
                const int nrows = 16 - (sk & 15);
                const uint32_t vb = sV + st * L::TILE;
                for (int idx = row; idx < nrows * 8 * NHALF; idx += 128) {
                    const int r = r0 + idx / (8 * NHALF);
                    const int rest = idx % (8 * NHALF);
                    const uint32_t addr = vb + (rest >> 3) * HALF + r * 128 + ((rest & 7) << 4);
                    st_shared_v4(addr, 0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_PFULL));
        }
        // ---- epilogue: O / l -> bf16 rows ----
        if (ok && wait_warp(bar(B_ODONE), (n_tiles - 1) & 1, abort_flag, p.err)) {
            tc_fence_after();
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            __nv_bfloat16 *dst = p.out +
                                 (static_cast<int64_t>(q_start + q0 + tok) * p.num_heads +
                                  kvh * G + g) * HD;
#pragma unroll 1
            for (int c = 0; c < HD / 32; ++c) {
                float o[32];
                tmem_ld_32x32b_x32(tmem + t_lane + kColO + c * 32, o);
                tmem_wait_ld();
                if (valid) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 v;
                        v.x = pack_bf16x2(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
                        v.y = pack_bf16x2(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
                        v.z = pack_bf16x2(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
                        v.w = pack_bf16x2(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
                        d4[i] = v;
                    }
                }
            }
        }
        tc_fence_before();
    }

    // ---- teardown: everyone done, then free tensor memory ----
    __syncthreads();
    if (*abort_flag) {
        // Drain whatever this CTA still has in flight before its shared and tensor memory
        // go away: outstanding tensor-core work (one commit after the last issue) and TMA
        // loads (their full barriers), each wait bounded.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side ---

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult qres;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &qres) == cudaSuccess &&
            qres == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool encode_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
               uint32_t b2) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int HD>
cudaError_t launch_prefill_d(PrefillKernelParams &kp, const PrefillArgs &a, cudaStream_t stream) {
    using L = Layout<HD>;
    const int64_t slots = a.num_blocks * a.block_size;
    if (!encode_3d(&kp.tmap_q, a.q, HD, a.num_heads, a.total_q, HD * 2ull,
                   static_cast<uint64_t>(a.num_heads) * HD * 2ull, 64, kp.group, kp.tok_per_tile))
        return cudaErrorInvalidValue;
    if (!encode_3d(&kp.tmap_k, a.k_cache, HD, a.num_kv_heads, static_cast<uint64_t>(slots),
                   HD * 2ull, static_cast<uint64_t>(a.num_kv_heads) * HD * 2ull, 64, 1, 16))
        return cudaErrorInvalidValue;
    if (!encode_3d(&kp.tmap_v, a.v_cache, HD, a.num_kv_heads, static_cast<uint64_t>(slots),
                   HD * 2ull, static_cast<uint64_t>(a.num_kv_heads) * HD * 2ull, 64, 1, 16))
        return cudaErrorInvalidValue;
    auto kern = prefill_kernel<HD>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    if (e != cudaSuccess) return e;
    const int q_tiles = (a.max_seqlen_q + kp.tok_per_tile - 1) / kp.tok_per_tile;
    dim3 grid(q_tiles, a.num_kv_heads, a.num_seqs);
    kern<<<grid, kThreads, L::SMEM, stream>>>(kp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs &a, cudaStream_t stream) {
    if (a.num_seqs == 0 || a.total_q == 0 || a.max_seqlen_q == 0) return cudaSuccess;
    const int64_t slots = a.num_blocks * a.block_size;
    if (slots > 0x7fffffffLL - 256 || a.total_q > 0x7fffffff - 256) return cudaErrorInvalidValue;
    PrefillKernelParams kp;
    memset(&kp, 0, sizeof kp);
    kp.out = static_cast<__nv_bfloat16 *>(a.out);
    kp.cu_q = a.cu_seqlens_q;
    kp.cu_k = a.cu_seqlens_k;
    kp.seq_lens = a.seq_lens;
    kp.block_table = a.block_table;
    kp.max_num_blocks = a.max_num_blocks;
    kp.num_seqs = a.num_seqs;
    kp.max_seqlen_q = a.max_seqlen_q;
    int log2_bs = 0;
    while ((1 << log2_bs) < a.block_size) ++log2_bs;
    kp.log2_bs = log2_bs;
    const int64_t table_cap = static_cast<int64_t>(a.max_num_blocks) << log2_bs;
    kp.seq_cap = table_cap < a.max_seqlen_k ? table_cap : a.max_seqlen_k;
    kp.num_blocks = a.num_blocks;
    kp.num_heads = a.num_heads;
    kp.num_kv_heads = a.num_kv_heads;
    kp.group = a.num_heads / a.num_kv_heads;
    kp.tok_per_tile = BM / kp.group;
    kp.window = a.sliding_window;
    kp.scale_log2 = a.scale * kLog2e;
    kp.err = a.err;
    switch (a.head_dim) {
        case 64: return launch_prefill_d<64>(kp, a, stream);
        case 128: return launch_prefill_d<128>(kp, a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
