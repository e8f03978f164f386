// decode.cu - split-K flash-decoding over the paged KV cache, plus the LSE combine.
//
// What it computes ("MinivLLM API docs - Attention", section paged_attention_decode;
// "vllm-npu 0.4.2, xformers.py", decode branch): for sequence b with L = seq_lens[b]
// keys and query head h, out[b][h] = softmax(scale * q K^T) V over keys
// [max(0, L - w), L) (w = sliding window, or all keys), K/V of kv head
// h / (num_heads / num_kv_heads), read through block_table.
//
// GB300 design (the page's Triton kernel runs one program per (sequence, query
// head) and streams the whole context once per query head):
//  * One CTA per (sequence, kv head, 16-head tile, split).  All query heads that
//    share a kv head sit in the same CTA, so each K/V byte is read from HBM once per
//    kv head, not once per query head.
//  * The split's key range is cut into 16-key units; warp w takes units w, w + NW,
//    ... and streams them through its own cp.async ring (16-byte copies, XOR-swizzled
//    so ldmatrix is bank-conflict free).  With block_size >= 16 a unit lies in one
//    block: one table lookup and one 64-bit base per unit; smaller power-of-two blocks
//    look up every key row.
//  * S^T = K Q^T and O^T += V^T P^T run on the warp MMA (m16n8k16, fp32 accumulate)
//    with the unit's 16 keys as the M rows and the query heads as N (8 per n-tile):
//    with 4-5 query heads per kv head, heads as the M = 16 rows would leave 3/4 of each
//    MMA and of the softmax as padding.  Decode is HBM bound; the MMA only keeps the
//    issue slots free (a CUDA-core dot product would need about one FFMA per loaded
//    element per query head).
//  * Online softmax in the base-2 domain with a lazily moved reference maximum; the
//    warps of a CTA merge their (m, l, O) through shared memory; a split writes either
//    the final bf16 row (single split) or a normalised fp32 partial plus (m, l) to the
//    workspace for decode_combine_kernel, which is launched with programmatic stream
//    serialization so its launch overlaps the splits' tail.
//  * Three CTAs per SM (2-stage rings, <= 168 registers) hide each other's pipeline
//    fill; the FP8 instantiation keeps the codes fp8 in shared memory (a 3-stage ring,
//    four CTAs per SM with one head n-tile) and runs f16 MMAs on codes converted in
//    registers.
#include <math.h>

#include <cuda_fp16.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "sm100_ptx.cuh"

namespace pa {

namespace {

// Resident split CTAs per SM: 4 warps with a 2-stage ring each (64 KB of shared memory
// at head_dim 128) and at most 168 registers a thread, so three fit.  More resident CTAs
// hide the pipeline fill at each CTA's start behind the other CTAs' streaming.
constexpr int kDecodeCtasPerSm = 3;
// The FP8 cache: a 3-stage ring of fp8 tiles (48 KB at head_dim 128); with one n-tile of
// heads the kernel fits 128 registers, so four CTAs (16 warps) hide more latency.
constexpr int kFp8Stages = 3;
constexpr int kDecodeCtasPerSmFp8 = 4;

template <bool FP8, int NT>
constexpr int decode_ctas_per_sm() {
    return FP8 && NT == 1 ? kDecodeCtasPerSmFp8 : kDecodeCtasPerSm;
}

using sm100::ex2_approx;

struct DecodeKernelParams {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *q;
    const __nv_bfloat16 *k_cache;
    const __nv_bfloat16 *v_cache;
    const int32_t *block_table;
    int max_num_blocks;
    const int32_t *seq_lens;
    int64_t seq_cap;  // min(max_num_blocks * block_size, max_seq_len)
    int64_t num_blocks;
    int log2_bs;
    int num_heads;
    int num_kv_heads;
    int group;
    int head_tiles;
    int window;
    float scale_log2;  // scale * log2(e)
    int chunk;
    int num_splits;
    float *ws_o;   // [batch, num_heads, num_splits, D] normalised partial outputs
    float *ws_ml;  // [batch, num_heads, num_splits, 2] (running max in log2 units, sum)
    // Fused store of the new token of each sequence (null when not fused).
    const __nv_bfloat16 *key;    // [batch, num_kv_heads, D]
    const __nv_bfloat16 *value;
    const int32_t *slot_mapping;  // [batch]
    __nv_bfloat16 *kc_w;          // the caches, writable
    __nv_bfloat16 *vc_w;
    // Partial-state output (null for the normal bf16 output): keys from key_begin[b]
    // on, result as fp32 rows st_o [batch, num_heads, D] and st_lse [batch, num_heads]
    // (natural log of the softmax denominator).
    const int32_t *key_begin;
    int key_begin_all;  // used when key_begin is null
    // FP8 E4M3 cache (the FP8 instantiation): codes, their scale, writable views.
    const uint8_t *k8;
    const uint8_t *v8;
    uint8_t *k8_w;
    uint8_t *v8_w;
    float kv_scale;
    float *st_o;
    float *st_lse;
    // Extra partial states the combine merges in (pre_parts x [batch * num_heads] rows).
    const float *pre_o;
    const float *pre_lse;
    int pre_parts;
    // Varlen layout: sequence b is a decode row only if q_rows[b + 1] - q_rows[b] == 1;
    // its q / out row is q_rows[b] (null: row b).
    const int32_t *q_rows;
    int total_q;        // rows of q / out in the varlen layout (q_rows bound)
    // Varlen layout without a prefill launch in the same call: the split kernel checks
    // the batch's query and key lengths itself (cu_k may be null).
    int check_rows;
    int max_seqlen_q;
    const int32_t *cu_k;
    int after_prefill;  // launched as the prefill kernel's programmatic dependent
    unsigned *err;
};

// Key range of one sequence: keys [start, L); splits tile [base, L) in `chunk`s.
struct SeqRange {
    int L;
    int start;
    int base;
};

__device__ __forceinline__ SeqRange decode_range(int raw_len, int64_t cap, int window,
                                                 int key_begin, unsigned *err, bool report) {
    SeqRange r;
    int L = raw_len;
    if (L < 0 || static_cast<int64_t>(L) > cap) {
        if (report) flag_error(err, kErrSeqRange);
        L = L < 0 ? 0 : static_cast<int>(cap);
    }
    r.L = L;
    r.start = window > 0 ? max(0, L - window) : 0;
    if (key_begin > r.start) r.start = min(key_begin, L);  // partial state from key_begin
    r.base = r.start & ~15;
    return r;
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16 *p) {
    return *reinterpret_cast<const uint32_t *>(p);
}

// Transpose of an 8x8 matrix of 16-bit elements held as the MMA accumulator fragment
// (lane holds row lane/4, columns 2 (lane%4) and + 1): afterwards the lane holds row
// lane/4 of the transpose.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4],
                                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Swizzled 16-byte chunk of an fp8 tile row (D bytes): the 8 rows an ldmatrix reads
// land in 8 different bank groups.
template <int D>
__device__ __forceinline__ int swz8(int c, int r) {
    if constexpr (D >= 128) return c ^ (r & 7);
    else return c ^ ((r >> 1) & 3);
}

// Two fp32 values -> two FP8 E4M3 codes (lo in the low byte): round to nearest even,
// finite values beyond 448 saturate.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// FP8: the cache holds E4M3 codes (x / kv_scale).  The products run as f16 MMAs on the
// codes converted in registers (one cvt per pair): K fragments come from ldmatrix on the
// fp8 rows with the head-dim index permuted alike in Q, V fragments from a transposing
// ldmatrix on byte pairs plus one byte permute (even and odd head dims in separate
// MMAs).  kv_scale is applied to the scores (K) and the results (V); Q and P are f16.
template <int D, int NWARPS, int NSTAGES, bool FP8, int NT>
__device__ __forceinline__ void decode_split_body(const DecodeKernelParams &p) {
    constexpr int ROWB = D * 2;               // bytes of one key row of one kv head
    constexpr int TILE_BYTES = 16 * ROWB;     // 16 keys
    constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K tile then V tile
    constexpr int CPR = D / 8;                // 16-byte chunks per row
    constexpr int KSTEPS = D / 16;
    constexpr int DTILES = D / 8;
    // FP8 ring: 16-key tiles of D bytes per row.
    constexpr int TILE8 = 16 * D;
    constexpr int STAGE8 = 2 * TILE8;
    constexpr int CPR8 = D / 16;  // 16-byte chunks per fp8 row
    constexpr int NST = FP8 ? kFp8Stages : NSTAGES;  // ring depth
    constexpr int SB = FP8 ? STAGE8 : STAGE_BYTES;   // bytes per stage

    extern __shared__ __align__(128) uint8_t smem[];

    const int split = blockIdx.x;
    const int b = blockIdx.z;
    int qrow = b;  // q / out row of sequence b
    if (p.q_rows != nullptr) {
        const int r0 = p.q_rows[b];
        const int sq = p.q_rows[b + 1] - r0;
        if (p.check_rows && split == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
            // No prefill kernel ran over this batch, so its length checks fall to here.
            const int sk = p.seq_lens[b];
            if (sq < 0 || sq > p.max_seqlen_q || sq > sk) flag_error(p.err, kErrQueryLen);
            if (p.cu_k != nullptr && p.cu_k[b + 1] - p.cu_k[b] != sk)
                flag_error(p.err, kErrSeqlensK);
        }
        if (sq != 1) return;  // not a single-row sequence
        if (r0 < 0 || r0 >= p.total_q) {  // malformed cu_seqlens_q: no access out of bounds
            if (split == 0 && blockIdx.y == 0 && threadIdx.x == 0) flag_error(p.err, kErrQueryLen);
            return;
        }
        qrow = r0;
    }
    const int kvh = blockIdx.y / p.head_tiles;
    const int ht = blockIdx.y - kvh * p.head_tiles;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // Speculative block-table entry of this warp's first 16-key unit for a range that
    // starts at key 0 (no window, no key_begin): loaded together with seq_lens, so the
    // first K/V copies need one memory round trip less.  Used only if it is that unit.
    const int spec_unit = ((split * p.chunk) >> 4) + static_cast<int>(threadIdx.x >> 5);
    int spec_blk = 0;
    if (p.log2_bs >= 4 && ((spec_unit << 4) >> p.log2_bs) < p.max_num_blocks)
        spec_blk = __ldg(p.block_table + static_cast<int64_t>(b) * p.max_num_blocks +
                         ((spec_unit << 4) >> p.log2_bs));
    const bool report = split == 0 && blockIdx.y == 0 && threadIdx.x == 0;
    const SeqRange sr = decode_range(p.seq_lens[b], p.seq_cap, p.window,
                                     p.key_begin ? p.key_begin[b] : p.key_begin_all, p.err,
                                     report);
    const int lo = max(sr.start, sr.base + split * p.chunk);
    const int hi = min(sr.L, sr.base + (split + 1) * p.chunk);
    const int h0 = kvh * p.group + ht * 16;
    const int rows_valid = min(16, p.group - ht * 16);

    // Fused store: a block that reads key L - 1 first writes this kv head's new token
    // (its row of the cache) itself, so no other launch has to run before it.  Every
    // such block writes the same bytes.  A sequence with no keys still gets its row
    // written, by split 0 of head tile 0.
    if (p.slot_mapping != nullptr &&
        ((lo < hi && hi == sr.L) || (sr.L == 0 && split == 0 && ht == 0))) {
        const int slot = p.slot_mapping[b];
        const int64_t num_slots = p.num_blocks << p.log2_bs;
        if (slot >= 0 && slot < num_slots) {
            const int64_t src_row = static_cast<int64_t>(b) * p.num_kv_heads + kvh;
            const int64_t dst_row = static_cast<int64_t>(slot) * p.num_kv_heads + kvh;
            if constexpr (FP8) {
                // 16 elements per thread: code = E4M3(x / kv_scale), the division in fp32.
                if (threadIdx.x < 2 * CPR8) {
                    const int which = threadIdx.x / CPR8;
                    const int c = threadIdx.x - which * CPR8;
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        (which ? p.value : p.key) + src_row * D + c * 16);
                    uint32_t w[8];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 v = src[h];
                        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float lo = __fdiv_rn(__uint_as_float(u[k] << 16), p.kv_scale);
                            const float hi =
                                __fdiv_rn(__uint_as_float(u[k] & 0xffff0000u), p.kv_scale);
                            w[h * 4 + k] = f32x2_to_e4m3x2(lo, hi);
                        }
                    }
                    uint4 o;
                    o.x = w[0] | (w[1] << 16);
                    o.y = w[2] | (w[3] << 16);
                    o.z = w[4] | (w[5] << 16);
                    o.w = w[6] | (w[7] << 16);
                    *reinterpret_cast<uint4 *>((which ? p.v8_w : p.k8_w) + dst_row * D + c * 16) = o;
                }
            } else if (threadIdx.x < 2 * CPR) {
                const int which = threadIdx.x / CPR;
                const int c = threadIdx.x - which * CPR;
                const uint4 v = reinterpret_cast<const uint4 *>((which ? p.value : p.key) +
                                                                src_row * D)[c];
                reinterpret_cast<uint4 *>((which ? p.vc_w : p.kc_w) + dst_row * D)[c] = v;
            }
            if (threadIdx.x == 0 && sr.L > 0 && ht == 0) {
                // The attention reads key L - 1 through block_table: the slot must be there.
                const int pos = sr.L - 1;
                const int blk = p.block_table[static_cast<int64_t>(b) * p.max_num_blocks +
                                              (pos >> p.log2_bs)];
                const int64_t want =
                    (static_cast<int64_t>(blk) << p.log2_bs) | (pos & ((1 << p.log2_bs) - 1));
                if (want != slot) flag_error(p.err, kErrSlotMismatch);
            }
            if (threadIdx.x == 0 && sr.L == 0) flag_error(p.err, kErrSlotMismatch);
        } else if (slot >= num_slots && threadIdx.x == 0) {
            flag_error(p.err, kErrSlotRange);
        }
        // The block's own loads of the row (cp.async, after this barrier) see the write.
        __syncthreads();
    }

    if (lo >= hi) {
        // Empty split.  A sequence with no keys at all gets a zero row; with several
        // splits the combine kernel writes it.
        if (p.ws_o == nullptr && sr.L == 0) {
            for (int i = threadIdx.x; i < rows_valid * D; i += NWARPS * 32)
                p.out[(static_cast<int64_t>(qrow) * p.num_heads + h0) * D + i] =
                    __float2bfloat16_rn(0.f);
        }
        return;
    }

    // Q^T fragments: the B operand (k = head dims, n = heads) of S^T = K Q^T, per n-tile j
    // of 8 heads (head 8 j + lane / 4) and 16-dim k-step ks: two 32-bit words.  Heads past
    // the group are zero.
    uint32_t qf[NT][KSTEPS][2];
    {
        const __nv_bfloat16 *qb = p.q + (static_cast<int64_t>(qrow) * p.num_heads + h0) * D;
        const int g = lane >> 2;
        if constexpr (FP8) {
            // f16, with the k order of the K fragments: k 2t, 2t+1 are dims 4t, 4t+1 and
            // k 2t+8, 2t+9 dims 4t+2, 4t+3 of the step (t = lane % 4).  |q| is clamped
            // to the f16 range.
            const int c0 = (lane & 3) * 4;
            auto f16pair = [](uint32_t w) -> uint32_t { return bf16x2_to_f16x2(w); };
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    uint2 x = make_uint2(0u, 0u);
                    if (8 * j + g < rows_valid)
                        x = *reinterpret_cast<const uint2 *>(qb + (8 * j + g) * D + ks * 16 + c0);
                    qf[j][ks][0] = f16pair(x.x);
                    qf[j][ks][1] = f16pair(x.y);
                }
        } else {
            const int c0 = (lane & 3) * 2;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int ks = 0; ks < KSTEPS; ++ks) {
                    const bool ok = 8 * j + g < rows_valid;
                    qf[j][ks][0] = ok ? ld_u32(qb + (8 * j + g) * D + ks * 16 + c0) : 0u;
                    qf[j][ks][1] = ok ? ld_u32(qb + (8 * j + g) * D + ks * 16 + c0 + 8) : 0u;
                }
        }
    }

    const int u_first = lo >> 4;
    const int u_last = (hi - 1) >> 4;
    const int32_t *bt_row = p.block_table + static_cast<int64_t>(b) * p.max_num_blocks;
    const int bs_mask = (1 << p.log2_bs) - 1;
    uint8_t *my_stages = smem + warp * NST * SB;  // NST stages of SB bytes
    const uint32_t stage_base = smem_u32(my_stages);
    const uint64_t policy = l2_policy_evict_first();

    // With block_size >= 16 a 16-key unit never straddles two blocks: one table lookup
    // per unit and fixed row strides.  Smaller blocks take the per-row path.
    const bool page_units = p.log2_bs >= 4;

    // The block of 16-key unit u (block_size >= 16: one lookup per unit).
    auto unit_block = [&](int u) -> int {
        return u == spec_unit ? spec_blk : __ldg(bt_row + ((u << 4) >> p.log2_bs));
    };
    // Copy geometry of one 16-key unit: rows of RB bytes (one kv head), 16-byte chunks,
    // RPP rows per pass of the warp.  Lane (c, rsub) copies chunk c of rows
    // i * RPP + rsub; its byte offset within the unit is fixed, so each unit needs one
    // 64-bit base and each pass one 32-bit add.
    constexpr int RB = FP8 ? D : ROWB;
    constexpr int CPRU = RB / 16;
    constexpr int RPP = 32 / CPRU;
    constexpr int NPASS = 16 / RPP;
    constexpr int UT = 16 * RB;  // bytes of a K (or V) tile of one unit in shared memory
    const uint8_t *kc8 = FP8 ? p.k8 : reinterpret_cast<const uint8_t *>(p.k_cache);
    const uint8_t *vc8 = FP8 ? p.v8 : reinterpret_cast<const uint8_t *>(p.v_cache);
    const int u_c = lane % CPRU;
    const int u_rsub = lane / CPRU;
    const int row_bytes = p.num_kv_heads * RB;
    const int lane_off = u_rsub * row_bytes + kvh * RB + u_c * 16;
    auto swz = [&](int c, int r) -> int {
        if constexpr (FP8) return swz8<D>(c, r);
        else return c ^ (r & 7);
    };
    auto issue = [&](int u, int st) {
        const uint32_t sb = stage_base + st * SB;
        const int j0 = u * 16;
        if (page_units) {
            const int blk = unit_block(u);
            const bool blk_ok = blk >= 0 && blk < p.num_blocks;
            if (!blk_ok && lane == 0) flag_error(p.err, kErrBlockRange);
            const int64_t uoff =
                blk_ok ? ((static_cast<int64_t>(blk) << p.log2_bs) + (j0 & bs_mask)) * row_bytes +
                             lane_off
                       : 0;
            const uint8_t *ks = kc8 + uoff;
            const uint8_t *vs = vc8 + uoff;
            if (blk_ok && j0 >= lo && j0 + 16 <= hi) {  // a full unit: no row checks
#pragma unroll
                for (int i = 0; i < NPASS; ++i) {
                    const int r = i * RPP + u_rsub;
                    const uint32_t so = r * RB + (swz(u_c, r) << 4);
                    cp_async_16_policy(sb + so, ks + i * RPP * row_bytes, 16u, policy);
                    cp_async_16_policy(sb + UT + so, vs + i * RPP * row_bytes, 16u, policy);
                }
            } else {
#pragma unroll
                for (int i = 0; i < NPASS; ++i) {
                    const int r = i * RPP + u_rsub;
                    const bool ok = blk_ok && j0 + r >= lo && j0 + r < hi;
                    const int o = ok ? i * RPP * row_bytes : 0;
                    const uint32_t so = r * RB + (swz(u_c, r) << 4);
                    cp_async_16_policy(sb + so, ok ? ks + o : kc8, ok ? 16u : 0u, policy);
                    cp_async_16_policy(sb + UT + so, ok ? vs + o : vc8, ok ? 16u : 0u, policy);
                }
            }
            return;
        }
        // block_size < 16: one table lookup per row.
#pragma unroll
        for (int i = 0; i < NPASS; ++i) {
            const int r = i * RPP + u_rsub;
            const int j = j0 + r;
            int64_t off = 0;
            uint32_t nbytes = 0;
            if (j >= lo && j < hi) {
                const int blk = __ldg(bt_row + (j >> p.log2_bs));
                if (blk < 0 || blk >= p.num_blocks) {
                    flag_error(p.err, kErrBlockRange);
                } else {
                    off = ((static_cast<int64_t>(blk) << p.log2_bs) + (j & bs_mask)) * row_bytes +
                          lane_off - u_rsub * row_bytes;
                    nbytes = 16;
                }
            }
            const uint32_t so = r * RB + (swz(u_c, r) << 4);
            cp_async_16_policy(sb + so, kc8 + off, nbytes, policy);
            cp_async_16_policy(sb + UT + so, vc8 + off, nbytes, policy);
        }
    };

    // O^T accumulators: m-tile mt of 16 head dims x n-tile j of 8 heads.  bf16: rows are
    // dims 16 mt + lane / 4 (+ 8); FP8 (mt = 2 dq + e): dims 32 dq + 2 (lane / 4) + e (+ 16).
    // Columns (heads) 8 j + 2 (lane % 4) and + 1.
    float o[NT][DTILES / 2][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int i = 0; i < DTILES / 2; ++i) o[j][i][0] = o[j][i][1] = o[j][i][2] = o[j][i][3] = 0.f;
    // Per head (8 j + 2 (lane % 4) + e): m_run is the reference maximum the weights are
    // taken against; it only moves when the true maximum exceeds it by more than 2^8, so O
    // is rarely rescaled.  l_run sums this lane's keys; lanes are summed at the end.
    float m_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        m_run[j][0] = m_run[j][1] = -INFINITY;
        l_run[j][0] = l_run[j][1] = 0.f;
    }

    const int my_first = u_first + warp;
    // Prologue: NST - 1 units in flight.
#pragma unroll
    for (int st = 0; st < NST - 1; ++st) {
        const int u = my_first + st * NWARPS;
        if (u <= u_last) issue(u, st);
        cp_async_commit();
    }

    const int g = lane >> 2;
    // ldmatrix row addresses.  K (A operand, non-transposed): matrices (keys 0-7, chunk c),
    // (keys 8-15, c), (keys 0-7, c + 1), (keys 8-15, c + 1).  V (A operand of O^T,
    // transposed): (keys 0-7, c), (keys 0-7, c + 1), (keys 8-15, c), (keys 8-15, c + 1).
    const int rk = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int ck = lane >> 4;
    const int rv = (lane >> 4) * 8 + (lane & 7);
    const int cv = (lane >> 3) & 1;

    int it = 0;
    for (int u = my_first; u <= u_last; u += NWARPS, ++it) {
        {
            const int un = u + (NST - 1) * NWARPS;
            if (un <= u_last) issue(un, (it + NST - 1) % NST);
            cp_async_commit();
        }
        cp_async_wait<NST - 1>();
        __syncwarp();

        const uint32_t kb = stage_base + (it % NST) * SB;
        const uint32_t vb = kb + UT;

        // S^T = K Q^T for 16 keys (M) and 8 heads per n-tile (N); even and odd k-steps in
        // separate accumulators to halve the dependent MMA chain.
        float s[NT][4], s2[NT][4];
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] = s2[j][e] = 0.f;
        if constexpr (FP8) {
            // One ldmatrix.x4 covers 16 keys x 32 dims (two k-steps); a word holds 4
            // consecutive dims of one key: its low f16 pair is k 2t, 2t+1 and its high pair
            // k 2t+8, 2t+9 of the step.
#pragma unroll
            for (int kq = 0; kq < D / 32; ++kq) {
                uint32_t kw[4];
                ldmatrix_x4(kw, kb + rk * D + (swz8<D>(2 * kq + ck, rk) << 4));
                uint32_t f[4][2];
#pragma unroll
                for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(kw[i], f[i][0], f[i][1]);
                const uint32_t a0[4] = {f[0][0], f[1][0], f[0][1], f[1][1]};
                const uint32_t a1[4] = {f[2][0], f[3][0], f[2][1], f[3][1]};
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    mma_f16_16816(s[j], a0, qf[j][2 * kq][0], qf[j][2 * kq][1]);
                    mma_f16_16816(s2[j], a1, qf[j][2 * kq + 1][0], qf[j][2 * kq + 1][1]);
                }
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                uint32_t ka[4];
                ldmatrix_x4(ka, kb + rk * ROWB + (((2 * ks + ck) ^ (rk & 7)) << 4));
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    mma_bf16_16816((ks & 1) ? s2[j] : s[j], ka, qf[j][ks][0], qf[j][ks][1]);
            }
        }

        // Scale, mask (edge units only), online softmax per head column: elements 0, 1 are
        // key u*16 + lane/4, elements 2, 3 key + 8; elements 0, 2 head 2t, 1, 3 head 2t+1.
        const bool edge = u * 16 < lo || u * 16 + 16 > hi;
        // The reference maximum only moves when a score exceeds it by more than 8, so the
        // column maxima (three dependent shuffles per head) are formed only when some
        // score of the warp does; otherwise nothing changes.
        bool over = false;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float v = (s[j][e] + s2[j][e]) * p.scale_log2;
                if (edge) {
                    const int key = u * 16 + g + (e >> 1) * 8;
                    if (key < lo || key >= hi) v = -INFINITY;
                }
                s[j][e] = v;
                over |= v > m_run[j][e & 1] + 8.f;
            }
        }
        if (__any_sync(0xffffffffu, over)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                float f[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float m = fmaxf(s[j][e], s[j][e + 2]);
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                    const float m_new = fmaxf(m_run[j][e], m);
                    const bool nd = m_new > m_run[j][e] + 8.f;
                    f[e] = nd ? ex2_approx(m_run[j][e] - m_new) : 1.f;
                    l_run[j][e] *= f[e];
                    if (nd) m_run[j][e] = m_new;
                }
#pragma unroll
                for (int mt = 0; mt < DTILES / 2; ++mt) {
                    o[j][mt][0] *= f[0];
                    o[j][mt][1] *= f[1];
                    o[j][mt][2] *= f[0];
                    o[j][mt][3] *= f[1];
                }
            }
        }
        // P^T (B operand of O^T = V^T P^T): the weights packed per key row (heads 2t, 2t+1)
        // and transposed by movmatrix into (head lane/4; keys 2t, 2t+1) words.  The
        // denominator sums the rounded weights the MMA actually uses.
        uint32_t pb[NT][2];
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const float m0 = m_run[j][0] == -INFINITY ? 0.f : m_run[j][0];
            const float m1 = m_run[j][1] == -INFINITY ? 0.f : m_run[j][1];
            const float e0 = ex2_approx(s[j][0] - m0), e1 = ex2_approx(s[j][1] - m1);
            const float e2 = ex2_approx(s[j][2] - m0), e3 = ex2_approx(s[j][3] - m1);
            uint32_t w0, w1;
            if constexpr (FP8) {
                w0 = pack_f16x2(e0, e1);
                w1 = pack_f16x2(e2, e3);
                add_f16x2_f32(l_run[j][0], l_run[j][1], w0);
                add_f16x2_f32(l_run[j][0], l_run[j][1], w1);
            } else {
                w0 = pack_bf16x2(e0, e1);
                w1 = pack_bf16x2(e2, e3);
                sm100::add_bf16x2_f32(l_run[j][0], l_run[j][1], w0);
                sm100::add_bf16x2_f32(l_run[j][0], l_run[j][1], w1);
            }
            pb[j][0] = movmatrix_trans(w0);  // keys 0-7
            pb[j][1] = movmatrix_trans(w1);  // keys 8-15
        }

        // O^T += V^T P^T.
        if constexpr (FP8) {
            // ldmatrix.trans on byte pairs: a word holds (key 2t, dims 2c', 2c'+1) and
            // (key 2t+1, same dims); one byte permute makes the key pairs of dim 2c' (low
            // half) and of dim 2c'+1 (high half): even and odd dims are separate m-tiles.
#pragma unroll
            for (int dq = 0; dq < D / 32; ++dq) {
                uint32_t vw[4];
                ldmatrix_x4_trans(vw, vb + rv * D + (swz8<D>(2 * dq + cv, rv) << 4));
                uint32_t f[4][2];
#pragma unroll
                for (int i = 0; i < 4; ++i) e4m3x4_to_f16x2x2(__byte_perm(vw[i], 0u, 0x3120), f[i][0], f[i][1]);
                const uint32_t ae[4] = {f[0][0], f[1][0], f[2][0], f[3][0]};
                const uint32_t ao[4] = {f[0][1], f[1][1], f[2][1], f[3][1]};
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    mma_f16_16816(o[j][2 * dq], ae, pb[j][0], pb[j][1]);
                    mma_f16_16816(o[j][2 * dq + 1], ao, pb[j][0], pb[j][1]);
                }
            }
        } else {
#pragma unroll
            for (int dp = 0; dp < D / 16; ++dp) {
                uint32_t va[4];
                ldmatrix_x4_trans(va, vb + rv * ROWB + (((2 * dp + cv) ^ (rv & 7)) << 4));
#pragma unroll
                for (int j = 0; j < NT; ++j) mma_bf16_16816(o[j][dp], va, pb[j][0], pb[j][1]);
            }
        }
        __syncwarp();
    }
    cp_async_wait<0>();
    // The combine kernel may start launching now (it waits for this grid to finish).
    sm100::griddep_launch_dependents();

#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            l_run[j][e] += __shfl_xor_sync(0xffffffffu, l_run[j][e], 4);
            l_run[j][e] += __shfl_xor_sync(0xffffffffu, l_run[j][e], 8);
            l_run[j][e] += __shfl_xor_sync(0xffffffffu, l_run[j][e], 16);
        }

    // Merge the warps of the CTA through shared memory (the stage ring is free now).
    __syncthreads();
    constexpr int OSTRIDE = D + 4;
    float *m_s = reinterpret_cast<float *>(smem);
    float *l_s = m_s + NWARPS * 16;
    float *o_s = l_s + NWARPS * 16;
    {
        const int t = lane & 3;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (g == 0) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    m_s[warp * 16 + 8 * j + 2 * t + e] = m_run[j][e];
                    l_s[warp * 16 + 8 * j + 2 * t + e] = l_run[j][e];
                }
            }
            float *ow = o_s + (warp * 16 + 8 * j + 2 * t) * OSTRIDE;
#pragma unroll
            for (int mt = 0; mt < DTILES / 2; ++mt) {
                int d0, d1;
                if constexpr (FP8) {
                    d0 = (mt >> 1) * 32 + 2 * g + (mt & 1);
                    d1 = d0 + 16;
                } else {
                    d0 = mt * 16 + g;
                    d1 = d0 + 8;
                }
                ow[d0] = o[j][mt][0];
                ow[OSTRIDE + d0] = o[j][mt][1];
                ow[d1] = o[j][mt][2];
                ow[OSTRIDE + d1] = o[j][mt][3];
            }
        }
    }
    __syncthreads();

    for (int idx = threadIdx.x; idx < rows_valid * D; idx += NWARPS * 32) {
        const int row = idx / D;
        const int d = idx - row * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) M = fmaxf(M, m_s[w * 16 + row]);
        float L = 0.f, acc = 0.f;
#pragma unroll
        for (int w = 0; w < NWARPS; ++w) {
            const float mw = m_s[w * 16 + row];
            const float f = mw == -INFINITY ? 0.f : ex2_approx(mw - M);
            L += f * l_s[w * 16 + row];
            acc += f * o_s[(w * 16 + row) * OSTRIDE + d];
        }
        float res = acc / L;
        if constexpr (FP8) res *= p.kv_scale;  // V elements read code * kv_scale
        const int64_t bh = static_cast<int64_t>(b) * p.num_heads + h0 + row;
        if (p.ws_o == nullptr) {
            p.out[(static_cast<int64_t>(qrow) * p.num_heads + h0 + row) * D + d] =
                __float2bfloat16_rn(res);
        } else {
            p.ws_o[(bh * p.num_splits + split) * D + d] = res;
            if (d == 0) {
                p.ws_ml[(bh * p.num_splits + split) * 2] = M;
                p.ws_ml[(bh * p.num_splits + split) * 2 + 1] = L;
            }
        }
    }
}

template <int D, int NWARPS, int NSTAGES, bool FP8, int NT>
__global__ void __launch_bounds__(NWARPS * 32, (decode_ctas_per_sm<FP8, NT>())) decode_split_kernel(const DecodeKernelParams p) {
    decode_split_body<D, NWARPS, NSTAGES, FP8, NT>(p);
    // As a programmatic dependent of the prefill kernel of the same call (single-row
    // sequences of a varlen batch, or a cascade's suffix) the CTAs run beside the prefill
    // on the SMs it leaves free.  The grid's last CTA waits for the prefill grid, so this
    // grid, the combine that waits for it and work queued later on the stream all
    // complete after the prefill.
    // (The CTA index is read again here, not kept live across the body.)
    if (p.after_prefill) {
        uint32_t x, y, z;
        asm volatile("mov.u32 %0, %%ctaid.x;\n\tmov.u32 %1, %%ctaid.y;\n\tmov.u32 %2, %%ctaid.z;"
                     : "=r"(x), "=r"(y), "=r"(z));
        if (x == gridDim.x - 1 && y == gridDim.y - 1 && z == gridDim.z - 1) sm100::griddep_wait();
    }
}

// acc += w * (one lane's 16- or 8-byte slice of a partial fp32 row).
template <int N>
__device__ __forceinline__ void add_row_slice(float (&acc)[N], const float *src, float w) {
    if constexpr (N == 4) {
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

// Log-sum-exp merge of the splits of one (sequence, head) per warp:
//   M = max_s m_s,  w_s = l_s * 2^(m_s - M),  out = sum_s w_s O_s / sum_s w_s
// where O_s are the normalised split outputs.
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeKernelParams p,
                                                             int batch) {
    constexpr int PER_LANE = D / 32;
    static_assert(PER_LANE == 4 || PER_LANE == 2, "16- or 8-byte row slices");
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int b = gw / p.num_heads;
    const int h = gw - b * p.num_heads;
    if (b >= batch) {
        sm100::griddep_wait();
        return;
    }
    // The call's own inputs (not written by the split grid) are read before the wait.
    const SeqRange sr = decode_range(p.seq_lens[b], p.seq_cap, p.window,
                                     p.key_begin ? p.key_begin[b] : p.key_begin_all, p.err, false);
    sm100::griddep_wait();  // launched early (programmatic serialization): the splits must be done
    const int nsplit = sr.L > sr.start ? (sr.L - sr.base + p.chunk - 1) / p.chunk : 0;
    const int64_t bh = static_cast<int64_t>(b) * p.num_heads + h;
    __nv_bfloat16 *dst = p.out + bh * D + lane * PER_LANE;
    const int npre = p.pre_parts;
    const int64_t pre_rows = static_cast<int64_t>(batch) * p.num_heads;
    if (nsplit == 0 && npre == 0) {
        if (p.st_o != nullptr) {
#pragma unroll
            for (int i = 0; i < PER_LANE; ++i) p.st_o[bh * D + lane * PER_LANE + i] = 0.f;
            if (lane == 0) p.st_lse[bh] = -INFINITY;
        } else {
#pragma unroll
            for (int i = 0; i < PER_LANE; ++i) dst[i] = __float2bfloat16_rn(0.f);
        }
        return;
    }
    const float *ml = p.ws_ml + bh * p.num_splits * 2;
    const float *os = p.ws_o + bh * p.num_splits * D + lane * PER_LANE;
    // Split s's (m, l) and extra part r's lse (log2 of its softmax mass is lse / ln 2) live in
    // lanes s % 32 and r % 32; both are loaded in one round trip when there are at most 32.
    float M = -INFINITY;
    for (int s0 = 0; s0 < nsplit || s0 < npre; s0 += 32) {
        const int s = s0 + lane;
        const float m = s < nsplit ? ml[2 * s] : -INFINITY;
        const float e = s < npre ? p.pre_lse[s * pre_rows + bh] * kLog2e : -INFINITY;
        M = fmaxf(M, fmaxf(m, e));
    }
    M = warp_max(M);
    if (M == -INFINITY) M = 0.f;  // every part empty: all weights are 0
    float wsum = 0.f;
    float acc[PER_LANE];
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) acc[i] = 0.f;
    for (int s0 = 0; s0 < nsplit; s0 += 32) {
        const int s = s0 + lane;
        const float wl = s < nsplit ? ml[2 * s + 1] * ex2_approx(ml[2 * s] - M) : 0.f;
        wsum += wl;
        const int n = min(32, nsplit - s0);
        // The partial rows of these splits, four loads in flight per lane.
#pragma unroll 4
        for (int k = 0; k < n; ++k)
            add_row_slice<PER_LANE>(acc, os + static_cast<int64_t>(s0 + k) * D,
                                    __shfl_sync(0xffffffffu, wl, k));
    }
    for (int r0 = 0; r0 < npre; r0 += 32) {
        const int r = r0 + lane;
        const float wl = r < npre ? ex2_approx(p.pre_lse[r * pre_rows + bh] * kLog2e - M) : 0.f;
        wsum += wl;
        const int n = min(32, npre - r0);
        for (int k = 0; k < n; ++k)
            add_row_slice<PER_LANE>(
                acc, p.pre_o + (static_cast<int64_t>(r0 + k) * pre_rows + bh) * D + lane * PER_LANE,
                __shfl_sync(0xffffffffu, wl, k));
    }
    wsum = warp_sum(wsum);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    if (p.st_o != nullptr) {
        // Partial state: normalised row and ln(sum_j e^{s_j}) = (M + log2 wsum) ln 2.
        float *so = p.st_o + bh * D + lane * PER_LANE;
#pragma unroll
        for (int i = 0; i < PER_LANE; ++i) so[i] = acc[i] * inv;
        if (lane == 0) p.st_lse[bh] = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
        return;
    }
#pragma unroll
    for (int i = 0; i < PER_LANE; i += 2)
        *reinterpret_cast<__nv_bfloat162 *>(dst + i) =
            __floats2bfloat162_rn(acc[i] * inv, acc[i + 1] * inv);
}

constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 2;

template <int D, bool FP8>
constexpr int decode_smem_bytes() {
    return FP8 ? kDecodeWarps * kFp8Stages * 2 * 16 * D : kDecodeWarps * kDecodeStages * 2 * 16 * D * 2;
}

template <int D, bool FP8>
cudaError_t launch_decode_d(const DecodeKernelParams &kp, const DecodePlan &plan, int batch,
                            cudaStream_t stream) {
    constexpr int smem = decode_smem_bytes<D, FP8>();
    static_assert(smem >= (kDecodeWarps * 16 * 2 + kDecodeWarps * 16 * (D + 4)) * 4,
                  "merge area must fit in the stage ring");
    // 8 heads per n-tile: a group of at most 8 query heads takes one, larger ones two.
    static std::atomic<uint64_t> smem_set[2];
    const int nt = kp.group <= 8 ? 0 : 1;
    auto kern = nt == 0 ? decode_split_kernel<D, kDecodeWarps, kDecodeStages, FP8, 1>
                        : decode_split_kernel<D, kDecodeWarps, kDecodeStages, FP8, 2>;
    cudaError_t e = smem_limit_once(kern, smem, smem_set[nt]);
    if (e != cudaSuccess) return e;
    dim3 grid(plan.num_splits, kp.num_kv_heads * plan.head_tiles, batch);
    if (kp.after_prefill) {
        // After the prefill kernel, as its programmatic dependent: the CTAs take the SMs
        // the prefill leaves free (the output rows are disjoint; the cache rows they read
        // were written by the store launch before the prefill).
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kDecodeWarps * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kern, kp);
        if (e != cudaSuccess) return e;
    } else {
        kern<<<grid, kDecodeWarps * 32, smem, stream>>>(kp);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess || (plan.num_splits == 1 && kp.st_o == nullptr && kp.pre_parts == 0))
        return e;
    // Programmatic stream serialization: the combine grid launches while the last split
    // CTAs finish, and waits for them on the device.
    const int warps = batch * kp.num_heads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((warps + 3) / 4);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, kp, batch);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool plan_decode(int batch, int num_heads, int num_kv_heads, int head_dim, int max_seq_len,
                 int sliding_window, int num_splits_request, DecodePlan *plan) {
    if (batch < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
        head_dim <= 0 || max_seq_len < 0)
        return false;
    DecodePlan p;
    p.group = num_heads / num_kv_heads;
    p.head_tiles = (p.group + 15) / 16;
    int64_t span = max_seq_len;
    if (sliding_window > 0 && static_cast<int64_t>(sliding_window) + 15 < span)
        span = static_cast<int64_t>(sliding_window) + 15;
    p.span = static_cast<int>(span);
    int splits;
    if (span <= 0 || batch == 0) {
        splits = 1;
    } else if (num_splits_request > 0) {
        splits = num_splits_request;
    } else {
        // Enough CTAs for ~12 per SM over the run (4 per resident slot: load balance
        // across ragged lengths), but no split shorter than 256 keys (4 units per warp).
        const int64_t units = static_cast<int64_t>(batch) * num_kv_heads * p.head_tiles;
        const int64_t target = 12LL * kPlanSms;
        int64_t s = (target + units - 1) / units;
        const int64_t by_len = (span + 255) / 256;
        if (s > by_len) s = by_len;
        // Long contexts: 8192-key chunks amortise each CTA's fixed cost (fill, merge)
        // better, as long as they still give two waves of resident CTAs.
        const int64_t s_long = (span + 8191) / 8192;
        if (s_long >= 2 && s_long < s && units * s_long >= 2LL * kDecodeCtasPerSm * kPlanSms)
            s = s_long;
        splits = static_cast<int>(s);
    }
    if (splits < 1) splits = 1;
    if (splits > 1024) splits = 1024;
    const int64_t span_pos = span > 0 ? span : 1;
    int64_t chunk = (span_pos + splits - 1) / splits;
    chunk = (chunk + 15) / 16 * 16;
    p.chunk = static_cast<int>(chunk);
    p.num_splits = static_cast<int>((span_pos + chunk - 1) / chunk);
    *plan = p;
    return true;
}

size_t decode_workspace_bytes(int batch, int num_heads, int head_dim, const DecodePlan &p,
                              bool state) {
    if (p.num_splits <= 1 && !state) return 0;  // one split writes its output directly
    const size_t rows = static_cast<size_t>(batch) * num_heads * p.num_splits;
    const size_t o_bytes = (rows * head_dim * sizeof(float) + 255) / 256 * 256;
    return o_bytes + rows * 2 * sizeof(float);
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
    if (a.batch == 0) return cudaSuccess;
    DecodeKernelParams kp;
    kp.out = static_cast<__nv_bfloat16 *>(a.out);
    kp.q = static_cast<const __nv_bfloat16 *>(a.q);
    kp.k_cache = static_cast<const __nv_bfloat16 *>(a.k_cache);
    kp.v_cache = static_cast<const __nv_bfloat16 *>(a.v_cache);
    kp.block_table = a.block_table;
    kp.max_num_blocks = a.max_num_blocks;
    kp.seq_lens = a.seq_lens;
    int log2_bs = 0;
    while ((1 << log2_bs) < a.block_size) ++log2_bs;
    kp.log2_bs = log2_bs;
    const int64_t table_cap = static_cast<int64_t>(a.max_num_blocks) << log2_bs;
    kp.seq_cap = table_cap < a.max_seq_len ? table_cap : a.max_seq_len;
    kp.num_blocks = a.num_blocks;
    kp.num_heads = a.num_heads;
    kp.num_kv_heads = a.num_kv_heads;
    kp.group = plan.group;
    kp.head_tiles = plan.head_tiles;
    kp.window = a.sliding_window;
    kp.scale_log2 = a.scale * kLog2e;
    kp.chunk = plan.chunk;
    kp.num_splits = plan.num_splits;
    if (plan.num_splits > 1 || a.state_o != nullptr || a.pre_parts > 0) {
        const size_t rows = static_cast<size_t>(a.batch) * a.num_heads * plan.num_splits;
        const size_t o_bytes = (rows * a.head_dim * sizeof(float) + 255) / 256 * 256;
        kp.ws_o = static_cast<float *>(a.workspace);
        kp.ws_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(a.workspace) + o_bytes);
    } else {
        kp.ws_o = nullptr;
        kp.ws_ml = nullptr;
    }
    kp.key = static_cast<const __nv_bfloat16 *>(a.key);
    kp.value = static_cast<const __nv_bfloat16 *>(a.value);
    kp.slot_mapping = a.slot_mapping;
    kp.kc_w = static_cast<__nv_bfloat16 *>(a.k_cache_w);
    kp.vc_w = static_cast<__nv_bfloat16 *>(a.v_cache_w);
    kp.key_begin = a.key_begin;
    kp.key_begin_all = a.key_begin_all;
    kp.st_o = a.state_o;
    kp.st_lse = a.state_lse;
    kp.pre_o = a.pre_o;
    kp.pre_lse = a.pre_lse;
    kp.pre_parts = a.pre_parts;
    kp.q_rows = a.q_rows;
    kp.total_q = a.total_q;
    kp.check_rows = a.check_rows ? 1 : 0;
    kp.max_seqlen_q = a.max_seqlen_q;
    kp.cu_k = a.cu_seqlens_k;
    kp.after_prefill = a.after_prefill ? 1 : 0;
    kp.err = a.err;
    if (a.fp8) {
        // E4M3 caches: codes read through the byte views, kv_scale on the scores (K) and,
        // in the kernel, on the results (V).
        kp.k8 = static_cast<const uint8_t *>(a.k_cache);
        kp.v8 = static_cast<const uint8_t *>(a.v_cache);
        kp.k8_w = static_cast<uint8_t *>(a.k_cache_w);
        kp.v8_w = static_cast<uint8_t *>(a.v_cache_w);
        kp.kv_scale = a.kv_scale;
        kp.scale_log2 = a.scale * a.kv_scale * kLog2e;
        kp.k_cache = nullptr;
        kp.v_cache = nullptr;
        switch (a.head_dim) {
            case 64: return launch_decode_d<64, true>(kp, plan, a.batch, stream);
            case 128: return launch_decode_d<128, true>(kp, plan, a.batch, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (a.head_dim) {
        case 64: return launch_decode_d<64, false>(kp, plan, a.batch, stream);
        case 128: return launch_decode_d<128, false>(kp, plan, a.batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
