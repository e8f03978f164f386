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
//  * Query tile = 128 MMA rows packing the G query heads of one kv head for
//    T = floor(128 / G) consecutive tokens (row m = token m / G, head m % G).  A work
//    item is two consecutive query tiles (2T tokens) of one (sequence, kv head), so every
//    K/V tile fetched feeds 256 rows: half the K/V bytes per FLOP of one tile.
//  * Persistent CTAs, one per SM.  The work list is ordered longest first and its valid
//    items are dealt to the CTAs in snake order; each CTA's scheduler warp publishes its
//    items to the other roles through a shared-memory ring.  The next item's Q is
//    prefetched into L2 while the current one runs.
//  * K/V come straight from the paged cache: the TMA producers walk block_table and
//    fetch each 16-key piece of a page as one 3-D box {64 dims, 1 kv head, 16 rows}
//    with 128-byte swizzle; pieces past the sequence come from an out-of-range
//    coordinate, which the TMA unit fills with zeros.
//  * Tensor memory (512 columns): S0, S1 (one 128x128 fp32 logit tile per query tile)
//    and O0, O1.  S_i = Q_i K^T runs as tcgen05.mma kind::f16 with both operands in
//    shared memory; softmax warpgroup i writes P_i as bf16 over the first 64 columns of
//    S_i, and O_i += P_i V takes P_i from tensor memory, V (N-major) from shared memory.
//  * One thread issues the MMAs in the order ... P0 V(t-1), S0(t), P1 V(t-1), S1(t) ...,
//    so each softmax warpgroup works on its tile while the tensor core runs the other
//    tile's products (ping-pong).
//  * Warp roles: 0-3 and 4-7 are the two softmax warpgroups (208 registers each after
//    setmaxnreg); 8 loads K, 9 issues MMAs, 10 loads V, 11 schedules the CTA's items and
//    loads Q (88 registers).  A softmax thread owns one TMEM lane (accumulator row):
//    mask, online softmax in base 2 with the scale folded into the exponent, lazy O
//    rescale (only when the running max grows by more than 2^8), epilogue.
//  * The K and V producers issue one page box per lane, in parallel; an item's last K/V
//    tile runs at half width (64 keys) when no row of the item sees its upper half.
//  * Every mbarrier wait is bounded: on timeout the CTA raises an error bit, drains,
//    frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "sm100_ptx.cuh"

namespace pa {

constexpr unsigned kErrTimeout = 0x20u;

namespace {

using namespace sm100;

constexpr int BM = 128;                  // MMA rows per query tile
constexpr int BN = 128;                  // keys per KV tile
constexpr uint32_t HALF = 128u * 128u;   // [128 rows][64 bf16] = 16 KB (one swizzle span)
constexpr int NSK = 3;                   // K stages
constexpr int NSV = 2;                   // V stages
// Warpgroups 0 and 1 (warps 0-3, 4-7) are the softmax of query tiles 0 and 1 (a warp
// reaches the TMEM lanes 32 * (warp % 4) ...); warpgroup 2 holds the producers and the
// MMA issuer.  The producer warpgroup gives up registers so that the
// softmax threads, which hold a 128-column logit row, get 208 (the launch's whole
// 168 x 384 registers: 208 x 256 + 88 x 128).
constexpr int kWarpK = 8, kWarpMma = 9, kWarpV = 10, kWarpSched = 11;
constexpr uint32_t kRing = 16;  // item-info ring slots
constexpr uint32_t kAhead = 14;  // items published beyond the last Q load (< kRing)
constexpr int kThreads = 12 * 32;
constexpr uint32_t kRegsSoftmax = 208, kRegsProducer = 88;
static_assert(kRegsSoftmax * 256 + kRegsProducer * 128 <= 168 * kThreads,
              "register split exceeds the launch's 168 per thread");
constexpr uint32_t kTmemCols = 512;
// Tensor-memory columns: S_i at 128 * i, O_i at 256 + 128 * i.
__host__ __device__ constexpr uint32_t col_s(int i) { return 128u * static_cast<uint32_t>(i); }
__host__ __device__ constexpr uint32_t col_o(int i) { return 256u + 128u * static_cast<uint32_t>(i); }
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait (default)

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
    int total_q;  // rows of q / out
    int max_seqlen_q;
    int q_items;  // ceil(max_seqlen_q / (2 * tok_per_tile))
    int n_items;  // q_items * num_kv_heads * num_seqs
    int64_t seq_cap;  // max_num_blocks * block_size, capped by max_seqlen_k
    int64_t num_blocks;
    int log2_bs;
    int num_heads;
    int num_kv_heads;
    int group;
    int tok_per_tile;  // floor(128 / group)
    int window;
    float scale_log2;  // scale * log2(e) > 0
    // Shared-prefix mode (cascade): the rows are the decode queries of num_req requests,
    // the keys the prefix_len keys of block_table row 0; the result of each split of
    // chunk_tiles key tiles is a partial state: st_o [n_splits, num_req * H, HD] fp32 and
    // st_lse [n_splits, num_req * H] (natural log).  req_lens bounds the window.
    const int32_t *req_lens;
    float *st_o;
    float *st_lse;
    int num_req;
    int prefix_len;
    int chunk_tiles;
    // Sequences with one query row are left to the decode kernel of the same call.
    int skip_decode_rows;
    float kv_scale;    // FP8 cache: attention reads code * kv_scale (folded into scale_log2 for K)
    uint64_t wait_ns;  // limit of every wait (kTimeoutNs unless a test lowers it)
    int stall;         // testing aid: publish no work item, so every wait runs out
    unsigned *err;
};

// Barrier indices.
enum : int {
    B_QFULL = 0,
    B_QEMPTY = 1,
    B_KFULL = 2,
    B_KEMPTY = B_KFULL + NSK,
    B_VFULL = B_KEMPTY + NSK,
    B_VEMPTY = B_VFULL + NSV,
    B_SFULL = B_VEMPTY + NSV,  // [2]: one per query tile
    B_PFULL = B_SFULL + 2,     // [2]
    B_ODONE = B_PFULL + 2,     // [2]
    B_IFULL = B_ODONE + 2,       // [kRing]: item-info ring slot written
    B_IEMPTY = B_IFULL + kRing,  // [kRing]: slot read by every consumer
    // FP8 cache: the codes of a K / V tile landed (before their conversion to f16), and
    // both query tiles converted to f16 by the softmax warps.
    B_LK = B_IEMPTY + kRing,     // [NSK]
    B_LV = B_LK + NSK,           // [NSV]
    B_QCONV = B_LV + NSV,
    NBARS = B_QCONV + 1
};

template <int HD>
struct Layout {
    static constexpr int NHALF = HD / 64;
    static constexpr uint32_t TILE = NHALF * HALF;  // one [128][HD] bf16 tile
    static constexpr uint32_t OFF_Q = 0;             // Q0, Q1
    static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;
    static constexpr uint32_t OFF_V = OFF_K + NSK * TILE;
    static constexpr uint32_t OFF_BAR = OFF_V + NSV * TILE;
    // 16-byte aligned: the item-info slots after it are read as 16-byte vectors.
    static constexpr uint32_t OFF_MISC = (OFF_BAR + NBARS * 8 + 15u) & ~15u;
    static constexpr uint32_t OFF_INFO = OFF_MISC + 16;   // item-info ring, kRing x 64 bytes
    static_assert(OFF_INFO % 16 == 0, "item-info slots are read as 16-byte vectors");
    static constexpr uint32_t BYTES = OFF_INFO + kRing * 64;
    // At least 116 KB so a single CTA owns an SM (and all of its TMEM).
    static constexpr uint32_t SMEM = (BYTES + 1024 > 118784u ? BYTES + 1024 : 118784u);
    static_assert(SMEM <= 232448u, "at most 227 KB of shared memory per CTA");
};

// Geometry of one work item; every role derives it identically.
struct Item {
    bool valid;
    bool has1;       // the second query tile has rows
    bool half_last;  // no row sees the upper 64 keys of the last K/V tile
    int seq, kvh, q0, rows0, rows1, q_start, sq, sk, kt0, n_tiles;
    int split;  // shared-prefix mode: key split of the item
};
// One slot of the item-info ring; end marks the end of the work list.
struct alignas(16) ItemSlot {
    Item it;
    int end;
};
static_assert(sizeof(ItemSlot) == 64, "item-info slots are 64 bytes");
constexpr int kConsumersPerItem = 11;  // K and V producers, MMA issuer, 8 softmax warps

// PREFIX: the shared-prefix (cascade) mode; item idx = (split, query-tile pair, kv head),
// the requests play the tokens of one sequence whose keys are the prefix.
template <bool PREFIX>
__device__ __forceinline__ Item get_item(const PrefillKernelParams &p, int idx, bool report) {
    Item it;
    it.split = 0;
    if constexpr (PREFIX) {
        const int per_s = p.num_kv_heads * p.q_items;
        it.split = idx / per_s;
        const int rem = idx - it.split * per_s;
        const int qi = rem / p.num_kv_heads;
        it.kvh = rem - qi * p.num_kv_heads;
        it.seq = 0;
        it.q_start = 0;
        it.sq = p.num_req;
        it.sk = p.prefix_len;
        it.valid = false;
        it.has1 = false;
        it.half_last = false;
        const int T = p.tok_per_tile;
        it.q0 = qi * 2 * T;
        if (it.q0 >= it.sq) return it;
        it.rows0 = min(T, it.sq - it.q0);
        it.rows1 = max(0, min(T, it.sq - it.q0 - T));
        it.has1 = it.rows1 > 0;
        const int total_tiles = (p.prefix_len + BN - 1) / BN;
        it.kt0 = it.split * p.chunk_tiles;
        it.n_tiles = min(p.chunk_tiles, total_tiles - it.kt0);
        it.valid = it.n_tiles > 0;
        it.half_last = p.prefix_len - 1 < (it.kt0 + it.n_tiles - 1) * BN + BN / 2;
        return it;
    }
    const int per_q = p.num_kv_heads * p.num_seqs;
    const int qi = p.q_items - 1 - idx / per_q;  // longest-running items first
    const int rem = idx - (idx / per_q) * per_q;
    it.seq = rem / p.num_kv_heads;
    it.kvh = rem - it.seq * p.num_kv_heads;
    it.valid = false;
    it.has1 = false;
    it.half_last = false;
    it.q_start = p.cu_q[it.seq];
    it.sq = p.cu_q[it.seq + 1] - it.q_start;
    if (it.q_start < 0 || it.sq < 0 || static_cast<int64_t>(it.q_start) + it.sq > p.total_q) {
        // Rows outside q / out (malformed cu_seqlens_q): flagged, never touched.
        if (report) flag_error(p.err, kErrQueryLen);
        return it;
    }
    int sk;
    if (p.seq_lens != nullptr) {
        sk = p.seq_lens[it.seq];
        if (report && p.cu_k != nullptr && p.cu_k[it.seq + 1] - p.cu_k[it.seq] != sk)
            flag_error(p.err, kErrSeqlensK);
    } else {
        sk = p.cu_k[it.seq + 1] - p.cu_k[it.seq];
    }
    if (sk < 0 || static_cast<int64_t>(sk) > p.seq_cap) {
        if (report) flag_error(p.err, kErrSeqRange);
        sk = sk < 0 ? 0 : static_cast<int>(p.seq_cap);
    }
    it.sk = sk;
    if (it.sq < 0 || it.sq > sk || it.sq > p.max_seqlen_q) {
        if (report) flag_error(p.err, kErrQueryLen);
        if (it.sq < 0 || it.sq > sk) return it;
    }
    if (p.skip_decode_rows && it.sq == 1) return it;  // the decode launch's row
    const int T = p.tok_per_tile;
    it.q0 = qi * 2 * T;
    if (it.q0 >= it.sq) return it;
    it.rows0 = min(T, it.sq - it.q0);
    it.rows1 = max(0, min(T, it.sq - it.q0 - T));
    it.has1 = it.rows1 > 0;
    const int p_lo = sk - it.sq + it.q0;
    const int p_hi = p_lo + it.rows0 + it.rows1 - 1;
    const int kmin = p.window > 0 ? max(0, p_lo - p.window + 1) : 0;
    it.kt0 = kmin / BN;
    it.n_tiles = p_hi / BN - it.kt0 + 1;
    it.half_last = p_hi < (it.kt0 + it.n_tiles - 1) * BN + BN / 2;
    it.valid = true;
    return it;
}

// Bounded wait by one thread.
__device__ __forceinline__ bool wait1(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      unsigned *err, uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 31u) {
            if (*abort_flag) return false;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            if (now - t0 > limit_ns) {
                *abort_flag = 1;
                flag_error(err, kErrTimeout);
                return false;
            }
        }
    }
}

// Bounded wait by a whole warp; every lane returns the same answer.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag, unsigned *err,
                                          uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        const bool ok = mbar_try_wait(bar, parity);
        if (__all_sync(0xffffffffu, ok)) return true;
        if ((it & 31u) == 31u) {
            bool stop = *abort_flag != 0;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            stop = stop || (now - t0 > limit_ns);
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

// ------------------------------------------------------------------ scheduler ---
// Run by one whole warp per CTA.  The work list is ordered longest first.  Its valid items
// (those with query rows) are dealt to the P CTAs in snake order: rank v goes to CTA v mod P
// in even rounds and to CTA P - 1 - (v mod P) in odd ones, which evens out the CTAs' total
// work.  The warp scans 32 list positions per step; every CTA scans the whole list, and
// position i reports its input errors only in CTA i mod P (and only where `reporter`).
// Items are published to the CTA's item ring up to kAhead beyond the last Q load, so the K
// and V producers can run ahead across short items.  Q loads go through the callbacks:
// q_free(l) (non-blocking) / q_wait(l) (bounded) tell whether the buffer of load l is free,
// q_load(l, item, next item or null) issues it.
template <bool PREFIX, class QFree, class QWait, class QLoad>
__device__ __forceinline__ void schedule_items(const PrefillKernelParams &p, ItemSlot *info,
                                               uint32_t bar_ifull, uint32_t bar_iempty,
                                               volatile int *abort_flag, uint32_t P,
                                               const uint32_t cta, const bool reporter,
                                               QFree q_free, QWait q_wait, QLoad q_load) {
    const int lane = threadIdx.x & 31;
    const int T = p.tok_per_tile;
    const int Hkv = p.num_kv_heads;
    auto ifull = [&](uint32_t i) { return bar_ifull + 8u * i; };
    auto iempty = [&](uint32_t i) { return bar_iempty + 8u * i; };
    int n_pairs = p.stall ? 0 : p.n_items / Hkv;  // (query block, sequence) pairs
    if (!PREFIX && p.skip_decode_rows) {
        // A batch whose single-row sequences go to the decode launch of the same call deals
        // its items to only as many CTAs as the same number of rounds needs; the decode
        // launch (a programmatic dependent of this kernel) takes the SMs of the others,
        // which find no item and exit.  Every CTA counts the same sequences, so all agree
        // on P.
        uint32_t pairs = 0, rows1 = 0;
        for (int i = lane; i < p.num_seqs; i += 32) {
            const int sq = p.cu_q[i + 1] - p.cu_q[i];
            if (sq == 1)
                ++rows1;
            else if (sq > 1)
                pairs += static_cast<uint32_t>(min((sq + 2 * T - 1) / (2 * T), p.q_items));
        }
        pairs = __reduce_add_sync(0xffffffffu, pairs);
        rows1 = __reduce_add_sync(0xffffffffu, rows1);
        const uint32_t v = pairs * static_cast<uint32_t>(Hkv);
        if (rows1 != 0) {
            // One round more when the decode rows outweigh the prefill items (with K keys a
            // row, decode time / prefill time ~ 0.68 rows1 / pairs).
            const uint32_t rounds = (v + P - 1) / P + (2u * rows1 >= 3u * pairs ? 1u : 0u);
            P = v == 0 ? 1u : (v + rounds - 1) / rounds;
        }
        if (cta >= P) n_pairs = 0;
    }
    // Target slot of round r: the snake order.
    auto target = [&](uint32_t r) -> uint32_t { return r * P + ((r & 1u) ? P - 1u - cta : cta); };
    uint32_t pub = 0, loaded = 0;  // items published / whose Q is loaded
    uint32_t vrank = 0;            // valid items in the scanned part of the list
    int scan = 0, win = 0;         // next pair to scan; first pair of the window
    uint32_t mine = 0;             // window pairs holding items of this CTA
    uint32_t r0_lane = 0;          // this lane's pair: rank of its first item
    int cur = -1;                  // pair being enumerated (window lane), or -1
    uint32_t cur_r0 = 0, cur_round = 0;
    bool ok = true;
    // One step per iteration, so a Q load (which gates the item's first S product) never
    // waits behind a scan: load Q when its buffer is free, else scan one window or publish
    // one item, else wait for the Q buffer.
    for (;;) {
        if (loaded < pub) {
            bool ready = true;
            if (lane == 0) ready = q_free(loaded);
            if (__shfl_sync(0xffffffffu, ready, 0)) {
                // The slots are intact: pub <= loaded + kAhead < loaded + kRing.
                if (lane == 0)
                    q_load(loaded, info[loaded % kRing].it,
                           loaded + 1 < pub ? &info[(loaded + 1) % kRing].it : nullptr);
                ++loaded;
                continue;
            }
        }
        if (pub < loaded + kAhead && (cur >= 0 || mine != 0 || scan < n_pairs)) {
            if (cur < 0 && mine == 0) {
                // Scan 32 pairs: the kv heads of a pair are all valid or none.
                const int pp = scan + lane;
                const bool v = pp < n_pairs &&
                               get_item<PREFIX>(p, pp * Hkv,
                                                reporter && static_cast<uint32_t>(pp) % P == cta)
                                   .valid;
                const uint32_t vm = __ballot_sync(0xffffffffu, v);
                r0_lane = vrank + static_cast<uint32_t>(Hkv) * __popc(vm & ((1u << lane) - 1u));
                // Does one of this CTA's ranks fall in [r0, r0 + Hkv)?  Only the first two
                // rounds from r0 / P can hold the first one.
                bool own = false;
                if (v) {
                    const uint32_t r = r0_lane / P;
                    const uint32_t t0 = target(r), t1 = target(r + 1);
                    own = (t0 >= r0_lane && t0 < r0_lane + Hkv) || t1 < r0_lane + Hkv;
                }
                mine = __ballot_sync(0xffffffffu, own);
                win = scan;
                scan += 32;
                vrank += static_cast<uint32_t>(Hkv) * __popc(vm);
                continue;
            }
            if (cur < 0) {
                cur = __ffs(mine) - 1;
                mine &= mine - 1u;
                cur_r0 = __shfl_sync(0xffffffffu, r0_lane, cur);
                cur_round = cur_r0 / P;
            }
            const uint32_t tv = target(cur_round++);
            if (tv < cur_r0) continue;
            if (tv >= cur_r0 + Hkv) {
                cur = -1;
                continue;
            }
            const int idx = (win + cur) * Hkv + static_cast<int>(tv - cur_r0);
            if (lane == 0) {
                const Item it = get_item<PREFIX>(p, idx, false);
                if (pub >= kRing && !wait1(iempty(pub % kRing), ((pub / kRing) - 1) & 1,
                                           abort_flag, p.err, p.wait_ns)) {
                    ok = false;
                } else {
                    info[pub % kRing].it = it;
                    info[pub % kRing].end = 0;
                    mbar_arrive(ifull(pub % kRing));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            ++pub;
            continue;
        }
        if (loaded == pub) break;  // the list is exhausted and every Q loaded
        // Only a Q load can make progress: wait for its buffer.
        if (lane == 0) ok = q_wait(loaded);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
    }
    // End of the list (never marked under the stall testing aid: every other role's first
    // wait then runs out, with nothing in flight).
    if (ok && lane == 0 && !*abort_flag && !p.stall &&
        (pub < kRing || wait1(iempty(pub % kRing), ((pub / kRing) - 1) & 1, abort_flag, p.err,
                              p.wait_ns))) {
        info[pub % kRing].end = 1;
        mbar_arrive(ifull(pub % kRing));
    }
}

// 32-byte global store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void *ptr, const uint32_t *w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]),
                 "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// One 128-key tile of E4M3 codes, [128 rows][128 codes] in the upper half of a stage with
// the 128-byte swizzle (16-byte chunk j of row r at r * 128 + ((j ^ r) & 7) * 16, so the
// lanes' reads of one chunk index hit 8 different bank groups), expanded in place into the
// f16 operand layout of the stage ([128][64] per 64-dim half, 128-byte swizzle), by one
// whole warp (4 rows a lane).  A row's f16 output of its
// upper half shares its 128-byte line with the row's own codes only, and the lane reads
// all of them before it writes, so no lane overwrites codes another lane still needs.
__device__ __forceinline__ void convert_tile_e4m3(uint32_t stage, int lane) {
    constexpr uint32_t kCodes = 128u * 128u;  // the f16 tile is 32 KB; its codes sit at 16 KB
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {
        const uint32_t r = static_cast<uint32_t>(lane + 32 * i);
        uint4 c[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) c[j] = ld_shared_v4(stage + kCodes + r * 128u + ((j ^ (r & 7u)) << 4));
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            // codes of head dims 16 j .. 16 j + 15: 64-dim half j / 4, 16-byte chunks 2 (j % 4)
            // and 2 (j % 4) + 1 of row r
            uint32_t w[8];
            e4m3x4_to_f16x2x2(c[j].x, w[0], w[1]);
            e4m3x4_to_f16x2x2(c[j].y, w[2], w[3]);
            e4m3x4_to_f16x2x2(c[j].z, w[4], w[5]);
            e4m3x4_to_f16x2x2(c[j].w, w[6], w[7]);
            const uint32_t line = stage + (j >> 2) * HALF + r * 128u;
            const uint32_t c0 = 2u * (j & 3);
            st_shared_v4(line + ((c0 ^ (r & 7u)) << 4), w[0], w[1], w[2], w[3]);
            st_shared_v4(line + (((c0 + 1u) ^ (r & 7u)) << 4), w[4], w[5], w[6], w[7]);
        }
    }
}

// FP8: the cache holds E4M3 codes (head_dim 128).  The producers TMA-load a tile's codes into
// the upper half of its shared-memory stage and expand them in place to f16 in the MMA
// operand layout (every E4M3 value is an f16); the softmax warps convert each query tile
// to f16 in place; the products are f16 MMAs with P in f16.
template <int HD, bool PREFIX, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PrefillKernelParams p) {
    static_assert(!FP8 || (HD == 128 && !PREFIX), "the FP8 cache path is built for head_dim 128");
    using L = Layout<HD>;
    constexpr int NHALF = L::NHALF;
    constexpr int KSTEPS_S = HD / 16;  // MMAs per S tile
    constexpr int KSTEPS_O = BN / 16;  // MMAs per PV tile

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *sb = smem_raw + (base - raw);
    const uint32_t sQ = base + L::OFF_Q;
    const uint32_t sK = base + L::OFF_K;
    const uint32_t sV = base + L::OFF_V;
    const uint32_t sBar = base + L::OFF_BAR;
    auto bar = [&](int i) -> uint32_t { return sBar + 8u * static_cast<uint32_t>(i); };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(sb + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sb + L::OFF_MISC + 4);
    // Item-info ring: the scheduler warp picks this CTA's items and hands each one to
    // every other role, so no role walks the work list or pays a global-memory round
    // trip when it changes item.
    ItemSlot *info = reinterpret_cast<ItemSlot *>(sb + L::OFF_INFO);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;
    const int T = p.tok_per_tile;
    const uint32_t q_tile_bytes = static_cast<uint32_t>(G * T) * 128u * NHALF;

    // ---- set-up: barriers, tensor memory ----
    if (threadIdx.x == 0) {
        mbar_init(bar(B_QFULL), 1);
        mbar_init(bar(B_QEMPTY), 1);
        for (int s = 0; s < NSK; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_KEMPTY + s), 1);
        }
        for (int s = 0; s < NSV; ++s) {
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_VEMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SFULL + i), 1);
            mbar_init(bar(B_PFULL + i), 4);
            mbar_init(bar(B_ODONE + i), 1);
        }
        for (uint32_t i = 0; i < kRing; ++i) {
            mbar_init(bar(B_IFULL + i), 1);
            mbar_init(bar(B_IEMPTY + i), kConsumersPerItem);
        }
        for (int s = 0; s < NSK; ++s) mbar_init(bar(B_LK + s), 1);
        for (int s = 0; s < NSV; ++s) mbar_init(bar(B_LV + s), 1);
        mbar_init(bar(B_QCONV), 8);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kWarpMma) {
        tmem_alloc(base + L::OFF_MISC, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Every CTA is resident: a programmatic dependent launched after this kernel (the
    // single-row decode of the same call, or the suffix decode of a cascade) may start
    // on the SMs this grid leaves free.
    griddep_launch_dependents();
    const int bs_mask = (1 << p.log2_bs) - 1;

    // Cache row (slot) of the 16-key piece of `it` starting at key k0, or an
    // out-of-range row (zero fill) past the sequence or for an invalid block index.
    auto kv_row = [&](const Item &it, int k0) -> int {
        if (k0 >= it.sk) return -16;
        const int blk = __ldg(p.block_table + static_cast<int64_t>(it.seq) * p.max_num_blocks +
                              (k0 >> p.log2_bs));
        if (blk < 0 || blk >= p.num_blocks) {
            flag_error(p.err, kErrBlockRange);
            return -16;
        }
        return (blk << p.log2_bs) | (k0 & bs_mask);
    };
    // One K or V tile (128 keys) of item `it` into shared memory at dst, issued by a whole
    // warp: each lane issues one box (16-key piece u, 64-dim half h), so the block-table
    // reads and the box issues overlap instead of queueing behind one thread.
    auto load_kv = [&](const CUtensorMap *map, const Item &it, int key0, uint32_t dst,
                       uint32_t full) {
        static_assert((BN / 16) * NHALF <= 32, "one lane per box");
        if (lane < (BN / 16) * NHALF) {
            const int u = lane / NHALF;
            const int h = lane - u * NHALF;
            const int row = kv_row(it, key0 + u * 16);
            tma_load_3d(dst + h * HALF + u * 2048, map, h * 64, it.kvh, row, full);
        }
    };

    if (warp >= 8) {
        // The register limit must be set inside each role's branch: code after a
        // merge of the two paths would get the smaller of the two limits.
        setmaxnreg_dec<kRegsProducer>();
        // Take ring slot ic (every consumer): false at the end of the list or on abort.
        auto take_item = [&](uint32_t ic, Item &it) -> bool {
            if (!wait_warp(bar(B_IFULL + ic % kRing), (ic / kRing) & 1, abort_flag, p.err, p.wait_ns))
                return false;
            it = info[ic % kRing].it;
            const bool end = info[ic % kRing].end != 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_IEMPTY + ic % kRing));
            return !end;
        };
        if (warp == kWarpSched) {
            // ---------------- scheduler + Q producer (whole warp) ----------------
            if (lane == 0) prefetch_tmap(&p.tmap_q);
            // Q0 and Q1 of an item share one buffer pair, free once the previous item's last
            // S products have read it.
            auto q_free = [&](uint32_t l) -> bool {
                return l == 0 || mbar_test_wait(bar(B_QEMPTY), (l - 1) & 1);
            };
            auto q_wait = [&](uint32_t l) -> bool {
                return wait1(bar(B_QEMPTY), (l - 1) & 1, abort_flag, p.err, p.wait_ns);
            };
            auto q_load = [&](uint32_t, const Item &it, const Item *nit) {
                mbar_arrive_expect_tx(bar(B_QFULL), q_tile_bytes * (it.has1 ? 2u : 1u));
#pragma unroll
                for (int h = 0; h < NHALF; ++h) {
                    tma_load_3d(sQ + h * HALF, &p.tmap_q, h * 64, it.kvh * G,
                                it.q_start + it.q0, bar(B_QFULL));
                    if (it.has1)
                        tma_load_3d(sQ + L::TILE + h * HALF, &p.tmap_q, h * 64, it.kvh * G,
                                    it.q_start + it.q0 + T, bar(B_QFULL));
                }
                if (nit != nullptr) {  // pull the next item's Q into L2
#pragma unroll
                    for (int h = 0; h < NHALF; ++h) {
                        tma_prefetch_l2_3d(&p.tmap_q, h * 64, nit->kvh * G, nit->q_start + nit->q0);
                        if (nit->has1)
                            tma_prefetch_l2_3d(&p.tmap_q, h * 64, nit->kvh * G,
                                               nit->q_start + nit->q0 + T);
                    }
                }
            };
            schedule_items<PREFIX>(p, info, bar(B_IFULL), bar(B_IEMPTY), abort_flag, gridDim.x,
                                   blockIdx.x, true, q_free, q_wait, q_load);
        } else if (warp == kWarpK || warp == kWarpV) {
            // ---------------- K / V producer (whole warp) ----------------
            auto produce = [&](auto is_k_tag) {
            constexpr bool is_k = decltype(is_k_tag)::value;
            const CUtensorMap *map = is_k ? &p.tmap_k : &p.tmap_v;
            const uint32_t sbase = is_k ? sK : sV;
            constexpr uint32_t NS = is_k ? NSK : NSV;
            constexpr int b_full = is_k ? B_KFULL : B_VFULL, b_empty = is_k ? B_KEMPTY : B_VEMPTY;
            if (lane == 0) prefetch_tmap(map);
            uint32_t t = 0;  // tiles issued
            bool ok = true;
            Item it;
            if constexpr (!FP8) {
                for (uint32_t ic = 0; ok && take_item(ic, it); ++ic) {
                    for (int j = 0; j < it.n_tiles; ++j, ++t) {
                        const uint32_t st = t % NS;
                        if (t >= NS && !wait_warp(bar(b_empty + st), ((t / NS) - 1) & 1, abort_flag,
                                                  p.err, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) mbar_arrive_expect_tx(bar(b_full + st), L::TILE);
                        __syncwarp();
                        load_kv(map, it, (it.kt0 + j) * BN, sbase + st * L::TILE, bar(b_full + st));
                    }
                }
            } else {
                // The codes of tile t land in the upper half of its stage (barrier B_LK / B_LV)
                // and are expanded there to f16.  The warp polls and does whichever step is
                // ready: take the next item, issue the next tile's codes once its stage is
                // free, expand the oldest tile whose codes have landed.  So a tile is expanded
                // as soon as it lands, while the tensor core still reads the tile before it,
                // and no issue waits behind an expansion it does not need.
                constexpr int b_land = is_k ? B_LK : B_LV;
                uint32_t tc = 0;  // tiles expanded
                uint32_t ic = 0;  // items taken
                int j = 0;
                bool have = false, done = false;
                uint64_t idle0 = 0;  // start of the current idle spell (0: none)
                for (uint32_t spin = 0; ok;) {
                    if (!have && !done &&
                        __all_sync(0xffffffffu, mbar_test_wait(bar(B_IFULL + ic % kRing), (ic / kRing) & 1))) {
                        if (take_item(ic, it)) {
                            have = it.n_tiles > 0;
                            j = 0;
                        } else {
                            done = true;
                        }
                        ++ic;
                        idle0 = 0;
                        continue;
                    }
                    if (have) {
                        const uint32_t st = t % NS;
                        if (t < NS ||
                            __all_sync(0xffffffffu, mbar_test_wait(bar(b_empty + st), ((t / NS) - 1) & 1))) {
                            if (lane == 0) mbar_arrive_expect_tx(bar(b_land + st), L::TILE / 2);
                            __syncwarp();
                            if (lane < BN / 16) {  // one 16-key piece of codes per lane
                                const int row = kv_row(it, (it.kt0 + j) * BN + 16 * lane);
                                tma_load_3d(sbase + st * L::TILE + L::TILE / 2 + lane * 2048, map, 0,
                                            it.kvh, row, bar(b_land + st));
                            }
                            ++t;
                            if (++j == it.n_tiles) have = false;
                            idle0 = 0;
                            continue;
                        }
                    }
                    if (tc < t) {
                        const uint32_t sc = tc % NS;
                        if (__all_sync(0xffffffffu, mbar_test_wait(bar(b_land + sc), (tc / NS) & 1))) {
                            convert_tile_e4m3(sbase + sc * L::TILE, lane);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(bar(b_full + sc));
                            ++tc;
                            idle0 = 0;
                            continue;
                        }
                    }
                    if (done && tc == t) break;
                    // Nothing ready: bounded like every wait.
                    if ((++spin & 31u) == 0) {
                        const uint64_t now = globaltimer_ns();
                        if (idle0 == 0) idle0 = now;
                        const bool stop = *abort_flag != 0 || now - idle0 > p.wait_ns;
                        if (__any_sync(0xffffffffu, stop)) {
                            if (lane == 0) {
                                *abort_flag = 1;
                                flag_error(p.err, kErrTimeout);
                            }
                            ok = false;
                        }
                    }
                }
            }
            };
            if (warp == kWarpK)
                produce(std::true_type{});
            else
                produce(std::false_type{});
        } else if (warp == kWarpMma) {
            // ---------------- MMA issuer ----------------
            // Order on the tensor pipe, across items: P0 V(g-1), S0(g), P1 V(g-1), S1(g).
            if (lane == 0) {
                constexpr uint32_t idesc_s = idesc_bf16_f32(BM, BN, false, FP8);
                // Half tile: the item's last K/V tile when no row sees its upper 64 keys
                // (diagonal of a query block that ends in the tile's lower half): S over
                // 64 keys, P V over 64 keys.  The softmax needs no change: the causal mask
                // already sets columns 64..127 to -inf.
                constexpr uint32_t idesc_s_half = idesc_bf16_f32(BM, BN / 2, false, FP8);
                constexpr uint32_t idesc_o = idesc_bf16_f32(BM, HD, true, FP8);
                uint32_t g = 0;                  // global KV tile counter
                uint32_t cnt[2] = {0, 0};        // tiles issued per query tile (S / P V)
                uint32_t ic = 0;                 // items
                bool ok = true;
                // Pending P V of the previous KV tile: its V stage, whether it is the first tile
                // of its item (overwrite O), and whether query tile 1 takes part.
                bool have_prev = false, prev_first = false, prev_has1 = false, prev_half = false;
                uint32_t prev_g = 0;
                auto issue_pv = [&](int i, uint32_t gv, bool first, bool half) -> bool {
                    const uint32_t c = cnt[i]++;
                    if (!wait1(bar(B_PFULL + i), c & 1, abort_flag, p.err, p.wait_ns)) return false;
                    if (i == 0 && !wait1(bar(B_VFULL + gv % NSV), (gv / NSV) & 1, abort_flag, p.err, p.wait_ns))
                        return false;
                    tc_fence_after();
                    const uint64_t b0 = smem_desc_sw128(sV + (gv % NSV) * L::TILE, HALF, 1024);
    #pragma unroll
                    for (int k = 0; k < KSTEPS_O; ++k) {
                        if (half && k >= KSTEPS_O / 2) break;
                        mma_bf16_ts(tmem + col_o(i), tmem + col_s(i) + k * 8, desc_advance(b0, k * 2048),
                                    idesc_o, (!first || k > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_ODONE + i));
                    return true;
                };
                auto issue_s = [&](int i, uint32_t gk, bool half) {
                    const uint64_t a0 = smem_desc_sw128(sQ + i * L::TILE, 16, 1024);
                    const uint64_t b0 = smem_desc_sw128(sK + (gk % NSK) * L::TILE, 16, 1024);
                    const uint32_t id = half ? idesc_s_half : idesc_s;
    #pragma unroll
                    for (int k = 0; k < KSTEPS_S; ++k) {
                        const uint32_t off = (k >> 2) * HALF + (k & 3) * 32;
                        mma_bf16_ss(tmem + col_s(i), desc_advance(a0, off), desc_advance(b0, off), id, k > 0);
                    }
                    mma_commit(bar(B_SFULL + i));
                };
                // Issue the P V products still pending from the previous KV tile.
                auto flush = [&]() -> bool {
                    if (!have_prev) return true;
                    have_prev = false;
                    if (!issue_pv(0, prev_g, prev_first, prev_half)) return false;
                    if (prev_has1 && !issue_pv(1, prev_g, prev_first, prev_half)) return false;
                    mma_commit(bar(B_VEMPTY + prev_g % NSV));
                    return true;
                };
                for (;; ++ic) {
                    if (!wait1(bar(B_IFULL + ic % kRing), (ic / kRing) & 1, abort_flag, p.err, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const Item it = info[ic % kRing].it;
                    const bool end = info[ic % kRing].end != 0;
                    mbar_arrive(bar(B_IEMPTY + ic % kRing));
                    if (end) break;
                    // Finish the previous item before waiting for this item's Q, so its
                    // epilogue never waits on a Q load.
                    if (!flush() || !wait1(bar(FP8 ? B_QCONV : B_QFULL), ic & 1, abort_flag, p.err, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    for (int j = 0; j < it.n_tiles; ++j, ++g) {
                        const int st = g % NSK;
                        // query tile 0: P0 V of the previous tile needs no K, so it goes to
                        // the tensor core before the wait for K(g)
                        const bool half = it.half_last && j == it.n_tiles - 1;
                        if (have_prev && !issue_pv(0, prev_g, prev_first, prev_half)) {
                            ok = false;
                            break;
                        }
                        if (!wait1(bar(B_KFULL + st), (g / NSK) & 1, abort_flag, p.err, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        issue_s(0, g, half);
                        // query tile 1
                        if (have_prev && prev_has1 && !issue_pv(1, prev_g, prev_first, prev_half)) {
                            ok = false;
                            break;
                        }
                        if (have_prev) mma_commit(bar(B_VEMPTY + prev_g % NSV));
                        if (it.has1) issue_s(1, g, half);
                        mma_commit(bar(B_KEMPTY + st));
                        if (j == it.n_tiles - 1) mma_commit(bar(B_QEMPTY));
                        have_prev = true;
                        prev_g = g;
                        prev_first = j == 0;
                        prev_has1 = it.has1;
                        prev_half = half;
                    }
                    if (!ok) break;
                }
                if (ok) flush();
            }
        }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ---------------- softmax warpgroups (warps 0..3: tile 0, 4..7: tile 1) ----------------
        const int wg = warp >> 2;
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t scol = tmem + t_lane + col_s(wg);
        const uint32_t ocol = tmem + t_lane + col_o(wg);
        const int tok = wg * T + row / G;  // token offset within the item
        const int g = row - (row / G) * G;
        const bool row_in_tile = row < G * T;
        const float sl2 = p.scale_log2;
        const int w = p.window;
        uint32_t gt = 0;   // global KV tile counter
        uint32_t c = 0;    // tiles this warpgroup has processed
        bool ok = true;
        for (uint32_t ic = 0; ok; ++ic) {
            if (!wait_warp(bar(B_IFULL + ic % kRing), (ic / kRing) & 1, abort_flag, p.err, p.wait_ns)) break;
            const Item it = info[ic % kRing].it;
            const bool end = info[ic % kRing].end != 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_IEMPTY + ic % kRing));
            if (end) break;
            if constexpr (FP8) {
                // The item's query tiles to f16, in place (a thread converts its row; the
                // 16-byte chunks of a row share its 128-byte line whatever the swizzle, and
                // taking them in swizzled order puts the 8 rows of a lane octet on 8 bank
                // groups).  Both warpgroups wait for the item's Q load even when tile 1 has no
                // rows, so neither arrives on QCONV for a later item before this one's phase
                // is done.
                if (!wait_warp(bar(B_QFULL), ic & 1, abort_flag, p.err, p.wait_ns)) break;
                if (wg == 0 || it.has1) {
                    if (row_in_tile) {
#pragma unroll
                        for (int h = 0; h < NHALF; ++h)
#pragma unroll
                            for (int c8 = 0; c8 < 8; ++c8) {
                                const uint32_t a = sQ + wg * L::TILE + h * HALF + row * 128 +
                                                   ((c8 ^ (row & 7)) << 4);
                                const uint4 v = ld_shared_v4(a);
                                st_shared_v4(a, bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y),
                                             bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
                            }
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_QCONV));
            }
            if (wg == 1 && !it.has1) {
                gt += it.n_tiles;
                continue;
            }
            const bool valid = row_in_tile && tok < it.rows0 + it.rows1;
            int pos, lo;
            if constexpr (PREFIX) {
                // Every prefix key is before the request's query; a window drops those
                // before the request's last w keys.
                pos = it.sk - 1;
                const int req_len = p.req_lens[min(it.q0 + tok, p.num_req - 1)];
                lo = w > 0 ? req_len - w : INT_MIN;
            } else {
                pos = it.sk - it.sq + it.q0 + tok;
                lo = w > 0 ? pos - w + 1 : INT_MIN;
            }
            float m_ref = -INFINITY;  // reference max (base-2 units) the weights use
            float l_sum = 0.f;
            for (int j = 0; j < it.n_tiles; ++j, ++gt, ++c) {
                if (!wait_warp(bar(B_SFULL + wg), c & 1, abort_flag, p.err, p.wait_ns)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float sc[BN / 32][32];
#pragma unroll
                for (int cc = 0; cc < BN / 32; ++cc) tmem_ld_32x32b_x32(scol + cc * 32, sc[cc]);
                // The waits name the loaded registers, so no use of them moves above.
#pragma unroll
                for (int cc = 0; cc < BN / 32; ++cc) tmem_wait_ld_regs(sc[cc]);
                float *s = &sc[0][0];

                const int key0 = (it.kt0 + j) * BN;
                // Row maximum as 8 independent 3-input max chains, then a tree (a single
                // dependent chain of 128 maxima would cost ~4 cycles per element).
                // Edge tiles: the causal bound and the window's lower bound are masked
                // separately, so a diagonal tile pays for one compare per element.
                if (key0 + BN - 1 > pos) {
                    const int last = pos - key0;  // columns past it lie in the future
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (i > last) s[i] = -INFINITY;
                }
                if (key0 < lo) {
                    const int first = lo - key0;  // columns before it lie outside the window
#pragma unroll
                    for (int i = 0; i < BN; ++i)
                        if (i < first) s[i] = -INFINITY;
                }
                static_assert(BN == 128, "the max tree covers 128 columns");
                float mx8[8];  // mx8[a] = max over s[a + 8k], k = 0..15
#pragma unroll
                for (int a = 0; a < 8; ++a) mx8[a] = max3f(s[a], s[a + 8], s[a + 16]);
#pragma unroll
                for (int k = 3; k < 15; k += 2) {
#pragma unroll
                    for (int a = 0; a < 8; ++a)
                        mx8[a] = max3f(mx8[a], s[a + 8 * k], s[a + 8 * k + 8]);
                }
#pragma unroll
                for (int a = 0; a < 8; ++a) mx8[a] = fmaxf(mx8[a], s[a + 120]);
                const float mx = fmaxf(fmaxf(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5])),
                                       fmaxf(mx8[6], mx8[7]));
                const float m_new = fmaxf(m_ref, mx * sl2);
                if (j == 0) {
                    m_ref = m_new;  // O holds nothing of this item yet
                } else {
                    const bool need = m_new > m_ref + 8.f;
                    if (__any_sync(0xffffffffu, need)) {
                        // S(c) was issued after P V(c-1), so seeing it complete means O
                        // already holds every earlier tile: rescale it in place.
                        const float f = need ? ex2_approx(m_ref - m_new) : 1.f;
#pragma unroll 1
                        for (int cc = 0; cc < HD / 32; ++cc) {
                            float o[32];
                            tmem_ld_32x32b_x32(ocol + cc * 32, o);
                            tmem_wait_ld_regs(o);
#pragma unroll
                            for (int i = 0; i < 32; ++i) o[i] *= f;
                            tmem_st_32x32b_x32(ocol + cc * 32, o);
                        }
                        l_sum *= f;
                        if (need) m_ref = m_new;
                    }
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;

                // P = 2^(s * scale_log2 - m) as bf16 over the low 64 columns of S; the
                // denominator sums the bf16 weights the MMA actually uses.
                // Pairs of columns go through packed f32x2 arithmetic; 2^x on the MUFU unit
                // (moving part of it to a polynomial on the FMA pipe measured slower: the
                // softmax is bound by instruction issue).
                const uint64_t sl2x2 = f2_pack(sl2, sl2);
                const uint64_t negm2 = f2_pack(-m_use, -m_use);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};  // partial sums of the bf16 weights
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const uint64_t x = f2_fma(f2_pack(s[cc * 64 + 2 * i], s[cc * 64 + 2 * i + 1]),
                                                  sl2x2, negm2);
                        float x0, x1;
                        f2_unpack(x, x0, x1);
                        if constexpr (FP8) {
                            pk[i] = pack_f16x2(ex2_approx(x0), ex2_approx(x1));
                            add_f16x2_f32(acc[2 * (i & 1)], acc[2 * (i & 1) + 1], pk[i]);
                        } else {
                            pk[i] = pack_bf16x2(ex2_approx(x0), ex2_approx(x1));
                            add_bf16x2_f32(acc[2 * (i & 1)], acc[2 * (i & 1) + 1], pk[i]);
                        }
                    }
                    tmem_st_32x32b_x32_u(scol + cc * 32, pk);
                }
                l_sum += (acc[0] + acc[1]) + (acc[2] + acc[3]);
                // Keys of the sequence's last, partly filled 16-key piece that lie past sk
                // are stale cache rows: warpgroup 0 zeroes them in the V tile (before
                // either P V of this tile is issued) so 0 * V stays 0.
                if (wg == 0 && ((it.sk - 1) / BN) == it.kt0 + j && (it.sk & 15) != 0) {
                    const int st = gt % NSV;
                    if (!wait_warp(bar(B_VFULL + st), (gt / NSV) & 1, abort_flag, p.err, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const int r0 = it.sk - key0;  // first stale row in the tile
                    const int nrows = 16 - (it.sk & 15);
                    const uint32_t vb = sV + st * L::TILE;
                    for (int i2 = row; i2 < nrows * 8 * NHALF; i2 += 128) {
                        const int r = r0 + i2 / (8 * NHALF);
                        const int rest = i2 % (8 * NHALF);
                        st_shared_v4(vb + (rest >> 3) * HALF + r * 128 + ((rest & 7) << 4), 0u, 0u,
                                     0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B_PFULL + wg));
            }
            if (!ok) break;
            // ---- epilogue: O / l -> bf16 rows (P V of the item's last tile is number c-1) ----
            if (!wait_warp(bar(B_ODONE + wg), (c - 1) & 1, abort_flag, p.err, p.wait_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // (FP8: V elements are code * kv_scale.)
            const float inv = l_sum > 0.f ? (FP8 ? p.kv_scale : 1.f) / l_sum : 0.f;
            if constexpr (PREFIX) {
                // Partial state of this key split: fp32 row and ln of its denominator.
                const int64_t rows = static_cast<int64_t>(p.num_req) * p.num_heads;
                const int64_t r = static_cast<int64_t>(it.q0 + tok) * p.num_heads +
                                  it.kvh * G + g;
                float *so = p.st_o + (static_cast<int64_t>(it.split) * rows + r) * HD;
#pragma unroll 1
                for (int cc = 0; cc < HD / 32; ++cc) {
                    float o[32];
                    tmem_ld_32x32b_x32(ocol + cc * 32, o);
                    tmem_wait_ld_regs(o);
                    if (valid) {
                        float4 *d4 = reinterpret_cast<float4 *>(so + cc * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            d4[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv,
                                                o[4 * i + 2] * inv, o[4 * i + 3] * inv);
                    }
                }
                if (valid) {
                    const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                    p.st_lse[static_cast<int64_t>(it.split) * rows + r] =
                        l_sum > 0.f ? (m_use + log2f(l_sum)) * kLn2 : -INFINITY;
                }
                tc_fence_before();
                continue;
            }
            __nv_bfloat16 *dst = p.out + (static_cast<int64_t>(it.q_start + it.q0 + tok) *
                                              p.num_heads + it.kvh * G + g) * HD;
            // A row is one thread's: 32-byte stores write whole sectors (16-byte ones leave
            // the L2 half-sector writes); the output is 32-byte aligned in practice.
            const bool v8 = (reinterpret_cast<uintptr_t>(p.out) & 31u) == 0;
            if (HD == 128 && v8 && (G & 3) == 0) {
                // The 4 rows of a lane quad are 4 consecutive heads of one token: 1 KB of
                // contiguous output.  Two xor-shuffle rounds give lane j of the quad the
                // j-th 32-byte slice (of each 128-column half) of all 4 rows, so every
                // store instruction writes whole 128-byte lines, 4 lanes per line.
                const int j = lane & 3;
                const bool b0 = (j & 1) != 0, b1 = (j & 2) != 0;
                __nv_bfloat16 *qdst = dst - j * HD;  // the quad's first row
#pragma unroll 1
                for (int t = 0; t < 2; ++t) {
                    float o[2][32];
                    tmem_ld_32x32b_x32(ocol + t * 64, o[0]);
                    tmem_ld_32x32b_x32(ocol + t * 64 + 32, o[1]);
                    tmem_wait_ld_regs(o[0]);
                    tmem_wait_ld_regs(o[1]);
                    // a[c][k]: word k of 32-byte slice c (columns 64t + 16c ...) of my row
                    uint32_t a[4][8];
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            a[c][k] = pack_bf16x2(o[c >> 1][(c & 1) * 16 + 2 * k] * inv,
                                                  o[c >> 1][(c & 1) * 16 + 2 * k + 1] * inv);
                    // Exchange 1 (partner j ^ 2): bb[r1][b] = (row (j & 1) | 2 r1, slice (j & 2) | b)
                    uint32_t bb[2][2][8];
#pragma unroll
                    for (int b = 0; b < 2; ++b)
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t send = b1 ? a[b][k] : a[2 | b][k];
                            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
                            bb[0][b][k] = b1 ? recv : a[b][k];
                            bb[1][b][k] = b1 ? a[2 | b][k] : recv;
                        }
                    // Exchange 2 (partner j ^ 1): f[r] = (row r, slice j)
                    uint32_t f[4][8];
#pragma unroll
                    for (int r1 = 0; r1 < 2; ++r1)
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t send = b0 ? bb[r1][0][k] : bb[r1][1][k];
                            const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
                            f[2 * r1][k] = b0 ? recv : bb[r1][0][k];
                            f[2 * r1 + 1][k] = b0 ? bb[r1][1][k] : recv;
                        }
                    if (valid) {
#pragma unroll
                        for (int r = 0; r < 4; ++r) st_global_v8(qdst + r * HD + (j + 4 * t) * 16, f[r]);
                    }
                }
                tc_fence_before();
                continue;
            }
#pragma unroll 1
            for (int cc = 0; cc < HD / 32; ++cc) {
                float o[32];
                tmem_ld_32x32b_x32(ocol + cc * 32, o);
                tmem_wait_ld_regs(o);
                if (valid) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(o[2 * i] * inv, o[2 * i + 1] * inv);
                    if (v8) {
                        st_global_v8(dst + cc * 32, w);
                        st_global_v8(dst + cc * 32 + 16, w + 8);
                    } else {
                        uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            d4[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
            }
            tc_fence_before();
        }
    }

    // ---- teardown: everyone done, then free tensor memory ----
    __syncthreads();
    if (*abort_flag) {
        // Bounded drain: let tensor-core work and TMA loads still in flight land before
        // this CTA's shared and tensor memory are released.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ------------------------------------------------------------------ host side ---

// Testing aid (pa_debug_prefill_stall): later launches publish no item / use this limit.
std::atomic<int> g_debug_stall{0};
std::atomic<uint64_t> g_debug_wait_ns{0};

void set_launch_limits(PrefillKernelParams &kp) {
    const uint64_t w = g_debug_wait_ns.load(std::memory_order_relaxed);
    kp.wait_ns = w != 0 ? w : kTimeoutNs;
    kp.stall = g_debug_stall.load(std::memory_order_relaxed);
}

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
               uint32_t b2, bool codes = false) {
    auto fn = get_encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    // codes: one-byte FP8 codes (128-byte rows, swizzled like the bf16 halves)
    const CUresult r = fn(map, codes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                          const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    static std::atomic<int> counts[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return kPlanSms;
    int n = counts[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = kPlanSms;
        counts[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

template <int HD, bool PREFIX, bool FP8 = false>
cudaError_t launch_prefill_d(PrefillKernelParams &kp, const PrefillArgs &a, cudaStream_t stream) {
    using L = Layout<HD>;
    const int64_t slots = a.num_blocks * a.block_size;
    if (!encode_3d(&kp.tmap_q, a.q, HD, a.num_heads, a.total_q, HD * 2ull,
                   static_cast<uint64_t>(a.num_heads) * HD * 2ull, 64, kp.group, kp.tok_per_tile))
        return cudaErrorInvalidValue;
    // K / V boxes: one 16-row piece of a page and a 64-dim half (bf16), or the piece's whole
    // rows of codes (FP8).
    const uint64_t eb = FP8 ? 1ull : 2ull;  // bytes per cache element
    for (int kv = 0; kv < 2; ++kv) {
        if (!encode_3d(kv ? &kp.tmap_v : &kp.tmap_k, kv ? a.v_cache : a.k_cache, HD,
                       a.num_kv_heads, static_cast<uint64_t>(slots), HD * eb,
                       static_cast<uint64_t>(a.num_kv_heads) * HD * eb, FP8 ? HD : 64, 1, 16, FP8))
            return cudaErrorInvalidValue;
    }
    auto kern = prefill_kernel<HD, PREFIX, FP8>;
    static std::atomic<uint64_t> smem_set;
    cudaError_t e = smem_limit_once(kern, static_cast<int>(L::SMEM), smem_set);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    const int grid = kp.n_items < sms ? kp.n_items : sms;
    kern<<<grid, kThreads, L::SMEM, stream>>>(kp);
    return cudaGetLastError();
}

}  // namespace

void debug_prefill_stall(int stall, uint64_t wait_ns) {
    g_debug_wait_ns.store(wait_ns, std::memory_order_relaxed);
    g_debug_stall.store(stall != 0 ? 1 : 0, std::memory_order_relaxed);
}

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
    kp.total_q = a.total_q;
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
    const int item_tokens = 2 * kp.tok_per_tile;
    kp.q_items = (a.max_seqlen_q + item_tokens - 1) / item_tokens;
    const int64_t n_items = static_cast<int64_t>(kp.q_items) * a.num_kv_heads * a.num_seqs;
    if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
    kp.n_items = static_cast<int>(n_items);
    kp.window = a.sliding_window;
    kp.kv_scale = a.fp8 ? a.kv_scale : 1.f;
    kp.scale_log2 = a.scale * kp.kv_scale * kLog2e;  // FP8: K elements are code * kv_scale
    kp.err = a.err;
    set_launch_limits(kp);
    // Sequences with a single query row (decode rows of a mixed batch) would fill one
    // token of a 128-row tile: with seq_lens given, a single-split decode launch takes
    // them (it needs no workspace) and the prefill kernel skips them.
    const bool route = a.seq_lens != nullptr;
    kp.skip_decode_rows = route ? 1 : 0;
    const bool prefill_launched = !route || a.max_seqlen_q > 1;
    if (prefill_launched) {
        cudaError_t e;
        if (a.fp8) {
            if (a.head_dim != 128) return cudaErrorInvalidValue;
            e = launch_prefill_d<128, false, true>(kp, a, stream);
        } else {
            switch (a.head_dim) {
                case 64: e = launch_prefill_d<64, false>(kp, a, stream); break;
                case 128: e = launch_prefill_d<128, false>(kp, a, stream); break;
                default: return cudaErrorInvalidValue;
            }
        }
        if (e != cudaSuccess || !route) return e;
    }
    DecodePlan plan;
    if (!plan_decode(a.num_seqs, a.num_heads, a.num_kv_heads, a.head_dim, a.max_seqlen_k,
                     a.sliding_window, 1, &plan))
        return cudaErrorInvalidValue;
    DecodeArgs d{};
    d.out = a.out;
    d.q = a.q;
    d.k_cache = a.k_cache;
    d.v_cache = a.v_cache;
    d.block_table = a.block_table;
    d.max_num_blocks = a.max_num_blocks;
    d.seq_lens = a.seq_lens;
    d.batch = a.num_seqs;
    d.max_seq_len = a.max_seqlen_k;
    d.num_blocks = a.num_blocks;
    d.block_size = a.block_size;
    d.num_heads = a.num_heads;
    d.num_kv_heads = a.num_kv_heads;
    d.head_dim = a.head_dim;
    d.sliding_window = a.sliding_window;
    d.scale = a.scale;
    d.q_rows = a.cu_seqlens_q;
    d.total_q = a.total_q;
    d.check_rows = !prefill_launched;
    d.max_seqlen_q = a.max_seqlen_q;
    d.cu_seqlens_k = a.cu_seqlens_k;
    d.fp8 = a.fp8;
    d.kv_scale = a.kv_scale;
    d.after_prefill = prefill_launched;
    d.err = a.err;
    return launch_decode(d, plan, stream);
}

void plan_prefix_splits(int num_req, int num_heads, int num_kv_heads, int prefix_len,
                        int *n_splits, int *chunk_tiles) {
    const int group = num_heads / num_kv_heads;
    const int tok = BM / (group > 0 ? group : 1);
    const int q_items = (num_req + 2 * tok - 1) / (2 * tok);
    const int tiles = (prefix_len + BN - 1) / BN;
    const int per_split = q_items * num_kv_heads;
    // About one prefix item per 8 SMs (at least one tile each): the prefix is little work
    // (each page is read once for all requests), and the suffix decode, which reads every
    // request's own keys, runs beside it on the SMs the prefix leaves free.  Over 64
    // requests sharing 4096 keys: 0.045 ms against 0.052 (one item per 16 SMs) and 0.057
    // (one per SM).
    int want = (sm_count() / 8 + per_split - 1) / (per_split > 0 ? per_split : 1);
    if (want < 1) want = 1;
    if (want > tiles) want = tiles;
    const int chunk = tiles > 0 ? (tiles + want - 1) / want : 1;
    *chunk_tiles = chunk;
    *n_splits = tiles > 0 ? (tiles + chunk - 1) / chunk : 0;
}

cudaError_t launch_prefix_states(const PrefixArgs &a, cudaStream_t stream) {
    if (a.num_req == 0 || a.n_splits == 0) return cudaSuccess;
    const int64_t slots = a.num_blocks * a.block_size;
    if (slots > 0x7fffffffLL - 256 || a.num_req > 0x7fffffff - 256) return cudaErrorInvalidValue;
    PrefillKernelParams kp;
    memset(&kp, 0, sizeof kp);
    kp.block_table = a.block_table;
    kp.max_num_blocks = a.prefix_len / a.block_size;
    kp.num_seqs = 1;
    int log2_bs = 0;
    while ((1 << log2_bs) < a.block_size) ++log2_bs;
    kp.log2_bs = log2_bs;
    kp.seq_cap = a.prefix_len;
    kp.num_blocks = a.num_blocks;
    kp.num_heads = a.num_heads;
    kp.num_kv_heads = a.num_kv_heads;
    kp.group = a.num_heads / a.num_kv_heads;
    kp.tok_per_tile = BM / kp.group;
    kp.q_items = (a.num_req + 2 * kp.tok_per_tile - 1) / (2 * kp.tok_per_tile);
    kp.max_seqlen_q = a.num_req;
    const int64_t n_items = static_cast<int64_t>(a.n_splits) * kp.q_items * a.num_kv_heads;
    if (n_items > 0x7fffffffLL) return cudaErrorInvalidValue;
    kp.n_items = static_cast<int>(n_items);
    kp.window = a.sliding_window;
    kp.scale_log2 = a.scale * kLog2e;
    kp.req_lens = a.req_lens;
    kp.st_o = a.st_o;
    kp.st_lse = a.st_lse;
    kp.num_req = a.num_req;
    kp.prefix_len = a.prefix_len;
    kp.chunk_tiles = a.chunk_tiles;
    kp.err = a.err;
    set_launch_limits(kp);
    // The launcher's view of the call: requests as the tokens of one sequence.
    PrefillArgs pa_{};
    pa_.q = a.q;
    pa_.k_cache = a.k_cache;
    pa_.v_cache = a.v_cache;
    pa_.total_q = a.num_req;
    pa_.num_blocks = a.num_blocks;
    pa_.block_size = a.block_size;
    pa_.num_heads = a.num_heads;
    pa_.num_kv_heads = a.num_kv_heads;
    pa_.head_dim = a.head_dim;
    switch (a.head_dim) {
        case 64: return launch_prefill_d<64, true>(kp, pa_, stream);
        case 128: return launch_prefill_d<128, true>(kp, pa_, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa
