// Sparse-attention indexer top-k + output transform for GB300 (sm_103a).
//
// The kernels here select, for every row, the k <= 2048 largest fp32 scores of
// a window and write each selected position through the PAGED page-table map
// or the RAGGED offset (sglang PR #35175 page, "Implementation breakdown" and
// "Key source snippets"; "#26788 [JIT Kernel] DeepSeek-V4 DSA indexer: faster
// top-k + page-table transform (runtime k <= 2048)" page). The public C ABI is
// declared in include/topk.h.
//
// Design (own design for sm_103a; the pages' CUDA/HIP kernels are prior art):
//
//  * Keys. A score's fp32 bits map to an order-preserving uint32 key. Every
//    selection step works on keys, so no score is compared as a float.
//  * Radix select on a 64-bit composite (key << 32 | ~position). Levels take
//    12, 8, 8 and 4 bits of the key from the top (the 12-bit first level is
//    the one the PR #36684 page, "Feature and motivation", describes), then,
//    only when equal scores straddle the threshold and TOPK_DETERMINISTIC is
//    set, 8/8/8/8 bits of ~position, so the lowest positions win. A level
//    stops the descent as soon as its threshold bin holds exactly the count
//    still needed.
//  * Threshold bin search: for the 4096-bin level every thread owns a run of
//    bins and a warp-shuffle suffix sum plus one pass over the warp totals
//    finds the bin where the count from the top first reaches the target
//    (cf. warp_inclusive_sum on the PR #36684 page, "Key source snippets");
//    the small levels use one warp.
//  * Routes, chosen per row by length (the plan kernel orders rows longest
//    first and hands long rows of small batches to the cluster path):
//      trivial   L <= k: positions 0..L-1 then -1, scores never read;
//      register  L <= 8192: the window lives in registers (16-byte loads);
//                a 14-bit first digit in packed 16-bit counters finds the
//                threshold bin, the elements above it go to a slot-ordered
//                list and the few in it are ranked against each other (every
//                remaining digit at once); the list is written out coalesced.
//                Very full threshold bins fall back to the 12-bit levels;
//      streaming longer rows: one pass over HBM builds the level-1 histogram
//                while collecting into shared memory every element whose top
//                12 key bits clear a lower bound estimated from the first tile
//                of the row; level 2 and the emit then run on that candidate
//                buffer, and the few elements equal to the 20-bit threshold
//                prefix are ranked. If the estimate was too high, or the
//                buffer overflowed, the row is re-read from global memory
//                (always exact, only slower);
//      cluster   for few long rows: the same streaming pass split over a
//                thread-block cluster of 4 CTAs (each slice bounds itself
//                from its own head tile), histograms merged through
//                distributed shared memory (reduce-scatter + all-gather) and
//                output slots allocated with atomics on the leader CTA's
//                shared memory (cf. TopKCluster on the PR #36684 page). A key
//                level whose group has no bit set below its digit (scores
//                rounded to bf16 or coarser) ends the key descent early.
//  * Compaction uses a warp scan and one shared-memory atomic per warp; the
//    emit gives slots by a block-wide scan (cf. warp_sum_bool, same page).
//  * PAGED rows copy their page-table entries into shared memory with
//    cp.async while the scores load, so the emit's lookups stay on chip.
//  * Unaligned window heads: 16-byte loads start at the aligned address below
//    the window and the up-to-3 leading / trailing lanes are excluded by
//    position. Scores are never written (the pages' kernel masks them in place).
//  * Every kernel is launched with programmatic dependent launch and waits
//    (griddepcontrol.wait) before touching global memory, so it is scheduled
//    while the previous kernel on the stream drains without breaking stream
//    order. No wait here spins: all waits are __syncthreads, hardware cluster
//    barriers or that grid dependency.

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "topk.h"

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = 512;                 // threads per CTA, all routes
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;                   // histogram bins (12-bit digit)
constexpr int kFineShift = 18;                // register route: a 14-bit first digit ...
constexpr int kFineWords = 8192;              // ... two 16-bit counters per word
constexpr int kCandCap = 6144;                // candidate buffer entries per CTA
constexpr int kPageCache = 4096;              // page-table entries of a row held in shared memory
constexpr int kTileVecs = 4;                  // 16-byte vectors per thread per streaming step
constexpr int kClusterSize = 4;               // CTAs per long row on the cluster path
constexpr int kPlanThreads = 1024;
constexpr int32_t kClusterFloor = 32768;      // rows longer than this may use the cluster path
constexpr int32_t kClusterMaxBatch = 64;      // ... when the batch is at most this
constexpr uint32_t kFull = 0xFFFFFFFFu;

constexpr int kBandTrivial = 32;              // plan bands: 0..31 by length, then these two
constexpr int kBandCluster = 33;
constexpr int kBands = 34;

struct alignas(64) PlanHeader {
    uint32_t magic;
    int32_t batch;
    int32_t k;
    int32_t n_order;      // rows listed in order[] (all rows not on the cluster path)
    int32_t n_cluster;    // rows listed in cluster_rows[]
    uint32_t error_rows;  // device-side data errors
    uint32_t flags;       // TOPK_DEVICE_FLAG_*
    int32_t reserved[9];
};
static_assert(sizeof(PlanHeader) == 64, "header layout");
constexpr uint32_t kPlanMagic = 0x6E616C50u;

size_t workspace_bytes_for(int32_t batch) {
    if (batch < 0) return 0;
    size_t bytes = sizeof(PlanHeader) + 2 * sizeof(int32_t) * static_cast<size_t>(batch);
    return (bytes + 255) / 256 * 256;
}

// Shared memory carve-up (dynamic). hist/mhist are 4096 counters each, the
// candidate buffer is (key, position)
// pairs, then the row's page-table entries (PAGED) and small scratch. The
// register route overlays its 16384 packed 16-bit counters on the candidate
// buffer, and the finishes keep their slot-ordered position list in hist's
// upper half and short tie lists in its lower half.
struct Shared {
    uint32_t* hist;      // local histogram
    uint32_t* mhist;     // merged histogram (== hist on a single CTA)
    uint32_t* cand_key;
    int32_t* cand_pos;
    int32_t* pages;      // kPageCache page-table entries
    uint32_t* red;       // 2 * kWarps words for scans
    uint32_t* res;       // threshold search results
    uint32_t* cnt;       // [0] candidates, [1] definite slots, [2] threshold-group slots
};

constexpr size_t kScratchWords = 2 * kWarps + 32;  // red: 2 words per warp; res: 16; cnt: 16
constexpr size_t kSmemRows = (kBins + 2 * kCandCap + kPageCache + kScratchWords) * 4;
constexpr size_t kSmemCluster = (2 * kBins + 2 * kCandCap + kPageCache + kScratchWords) * 4;

__device__ __forceinline__ Shared carve(uint8_t* base, bool merged_separate) {
    Shared s;
    uint32_t* w = reinterpret_cast<uint32_t*>(base);
    s.hist = w;
    w += kBins;
    if (merged_separate) {
        s.mhist = w;
        w += kBins;
    } else {
        s.mhist = s.hist;
    }
    s.cand_key = w;
    w += kCandCap;
    s.cand_pos = reinterpret_cast<int32_t*>(w);
    w += kCandCap;
    s.pages = reinterpret_cast<int32_t*>(w);
    w += kPageCache;
    s.red = w;
    s.res = w + 2 * kWarps;
    s.cnt = w + 2 * kWarps + 16;
    return s;
}

struct Params {
    const float* scores;
    int64_t score_stride;
    const int32_t* row_starts;
    const int32_t* seq_lens;
    const int32_t* out_offsets;
    const int32_t* page_table;
    int64_t page_table_stride;
    int32_t page_bits;
    int32_t batch;
    int32_t k;
    uint32_t flags;
    int32_t* out;
    int32_t* out_raw;
    PlanHeader* hdr;
    const int32_t* order;
    const int32_t* cluster_rows;
    const int32_t* pt_row_starts;  // packed PAGED: request-local token of each row's position 0, or null
    const int32_t* row_to_batch;   // packed PAGED: each row's page-table row, or null
};

// ----------------------------------------------------------------------------
// small device helpers
// ----------------------------------------------------------------------------

// Order-preserving fp32 -> uint32: flip all bits of negatives, set the sign bit
// of non-negatives.
__device__ __forceinline__ uint32_t score_key(float x) {
    const uint32_t b = __float_as_uint(x);
    return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}

__device__ __forceinline__ float4 load_stream(const float4* p) {
    float4 r;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "l"(p));
    return r;
}

// The same 16 bytes as raw integer bits (keys and key compares are integer
// work; the bits never pass through a float register).
__device__ __forceinline__ int4 load_stream_bits(const float4* p) {
    int4 r;
    asm("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Order-preserving key of raw fp32 bits (same map as score_key).
__device__ __forceinline__ uint32_t bits_key(uint32_t b) {
    return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t warp_inclusive_scan(uint32_t v) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, v, off);
        if (lane_id() >= static_cast<uint32_t>(off)) v += y;
    }
    return v;
}

__device__ __forceinline__ uint64_t composite(uint32_t key, int32_t pos) {
    return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~pos);
}

// Radix levels over the 64-bit composite: 12/8/8/4 bits of the key, then
// 8/8/8/8 bits of ~position (deterministic tie-break only).
constexpr int kKeyLevels = 4;
constexpr int kAllLevels = 8;
__device__ __forceinline__ int level_shift(int lvl) {
    return lvl == 0 ? 52 : lvl == 1 ? 44 : lvl == 2 ? 36 : lvl == 3 ? 32 : 8 * (7 - lvl);
}
__device__ __forceinline__ int level_bins(int lvl) { return lvl == 0 ? kBins : lvl == 3 ? 16 : 256; }

// Finds the largest bin d of h[0..nb) with sum_{c >= d} h[c] >= target and
// returns it with above = sum_{c > d} h[c] and count = h[d]; `found` is false
// (with above = the total) when target exceeds the total. nb is 4096, 256 or
// 16 (h 16-byte aligned); target >= 1. All threads call it.
//  * nb = 4096 (find_threshold_wide): thread t holds bins Rt..Rt+R-1
//    (R = 4096 / threads); a warp-shuffle suffix sum plus the warp totals in
//    shared memory give every thread the count above its run, and the one
//    thread whose run crosses the target resolves the bin. Two barriers.
//  * nb <= 256: warp 0 holds the bins (lane l: 8l..8l+7), one warp-shuffle
//    suffix sum; the other warps wait at the single barrier.
struct Threshold {
    uint32_t bin, above, count;
    bool found;
};

// First half of the 4096-bin search: every thread returns the histogram's
// total and the thread whose run crosses the target writes the bin to
// sh.res. One barrier (after it every bin has been read); the caller reads
// the result with find_wide_result after a barrier of its own.
__device__ uint32_t find_wide_publish(const uint32_t* h, uint32_t target, const Shared& sh) {
    constexpr int R = kBins / kThreads;  // bins per thread
    static_assert(R % 4 == 0 && R * kThreads == kBins, "whole 16-byte runs of bins per thread");
    const uint32_t lane = lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    uint32_t b[R];
#pragma unroll
    for (int q = 0; q < R / 4; ++q) {
        const uint4 u = reinterpret_cast<const uint4*>(h)[(R / 4) * threadIdx.x + q];
        b[4 * q] = u.x, b[4 * q + 1] = u.y, b[4 * q + 2] = u.z, b[4 * q + 3] = u.w;
    }
    uint32_t s8 = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) s8 += b[i];
    uint32_t x = s8;  // sum over the lanes >= this lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, x, off);
        if (lane + off < 32) x += y;
    }
    if (lane == 0) sh.red[warp] = x;
    __syncthreads();
    uint32_t above = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t r = sh.red[w];
        total += r;
        above += w > warp ? r : 0u;
    }
    const uint32_t incl = above + x, excl = incl - s8;
    if (excl < target && incl >= target) {
        uint32_t r = excl;
#pragma unroll
        for (int i = R - 1; i >= 0; --i) {
            if (r + b[i] >= target) {
                sh.res[0] = R * threadIdx.x + static_cast<uint32_t>(i);
                sh.res[1] = r;
                sh.res[2] = b[i];
                break;
            }
            r += b[i];
        }
    }
    return total;
}

__device__ __forceinline__ Threshold find_wide_result(uint32_t total, uint32_t target, const Shared& sh) {
    if (total < target) return Threshold{0u, total, 0u, false};
    return Threshold{sh.res[0], sh.res[1], sh.res[2], true};
}

// find_wide_publish for the register route's 16384 bins of 16-bit counters,
// two per word (bin 2w in the low half of word w): thread t holds words
// 16t..16t+15. Per-thread sums add whole words (each half stays below 2^16:
// a row holds at most 8192 elements).
__device__ uint32_t find_fine_publish(const uint32_t* h, uint32_t target, const Shared& sh) {
    constexpr int W = kFineWords / kThreads;
    static_assert(W % 4 == 0 && W * kThreads == kFineWords, "whole 16-byte runs of words per thread");
    const uint32_t lane = lane_id();
    const int warp = static_cast<int>(threadIdx.x >> 5);
    uint32_t wd[W];
#pragma unroll
    for (int q = 0; q < W / 4; ++q) {
        const uint4 u = reinterpret_cast<const uint4*>(h)[(W / 4) * threadIdx.x + q];
        wd[4 * q] = u.x, wd[4 * q + 1] = u.y, wd[4 * q + 2] = u.z, wd[4 * q + 3] = u.w;
    }
    uint32_t pair = 0;
#pragma unroll
    for (int i = 0; i < W; ++i) pair += wd[i];
    const uint32_t s32 = (pair & 0xFFFFu) + (pair >> 16);
    uint32_t x = s32;  // sum over the lanes >= this lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, x, off);
        if (lane + off < 32) x += y;
    }
    if (lane == 0) sh.red[warp] = x;
    __syncthreads();
    uint32_t above = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t r = sh.red[w];
        total += r;
        above += w > warp ? r : 0u;
    }
    const uint32_t incl = above + x, excl = incl - s32;
    if (excl < target && incl >= target) {
        // the word first (both halves at once), then the half; the run ends
        // in word 0 at the latest
        uint32_t r = excl, wsel = 0, rsel = 0;
        int isel = 0;
        bool done = false;
#pragma unroll
        for (int i = W - 1; i >= 0; --i) {
            const uint32_t c2 = (wd[i] & 0xFFFFu) + (wd[i] >> 16);
            if (!done && (i == 0 || r + c2 >= target)) {
                wsel = wd[i];
                isel = i;
                rsel = r;
                done = true;
            }
            r += c2;
        }
        const uint32_t hi = wsel >> 16, lo = wsel & 0xFFFFu;
        const bool in_hi = rsel + hi >= target;
        sh.res[0] = 2 * (W * threadIdx.x + static_cast<uint32_t>(isel)) + (in_hi ? 1u : 0u);
        sh.res[1] = in_hi ? rsel : rsel + hi;
        sh.res[2] = in_hi ? hi : lo;
    }
    return total;
}

__device__ Threshold find_threshold_wide(const uint32_t* h, uint32_t target, const Shared& sh) {
    const uint32_t total = find_wide_publish(h, target, sh);
    __syncthreads();
    return find_wide_result(total, target, sh);
}

__device__ Threshold find_threshold(const uint32_t* h, int nb, uint32_t target, const Shared& sh) {
    if (nb == kBins) return find_threshold_wide(h, target, sh);
    if (threadIdx.x < 32) {
        const uint32_t lane = lane_id();
        uint32_t run = 0;  // count in the bins above the current block
        bool found = false;
        for (int top = nb; top > 0 && !found; top -= 256) {
            const int lo = max(top - 256, 0) + 8 * static_cast<int>(lane);
            uint32_t b[8];
            if (lo < top) {
                const uint4 u = reinterpret_cast<const uint4*>(h + lo)[0];
                const uint4 v = reinterpret_cast<const uint4*>(h + lo)[1];
                b[0] = u.x, b[1] = u.y, b[2] = u.z, b[3] = u.w, b[4] = v.x, b[5] = v.y, b[6] = v.z, b[7] = v.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) b[i] = 0;
            }
            const uint32_t s8 = b[0] + b[1] + b[2] + b[3] + b[4] + b[5] + b[6] + b[7];
            uint32_t x = s8;  // sum over lanes >= this lane
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_down_sync(kFull, x, off);
                if (lane + off < 32) x += y;
            }
            const uint32_t block = __shfl_sync(kFull, x, 0);
            if (run + block >= target) {  // warp-uniform
                found = true;
                const uint32_t incl = run + x, excl = incl - s8;
                if (excl < target && incl >= target) {
                    uint32_t r = excl;
#pragma unroll
                    for (int i = 7; i >= 0; --i) {
                        if (r + b[i] >= target) {
                            sh.res[0] = static_cast<uint32_t>(lo + i);
                            sh.res[1] = r;
                            sh.res[2] = b[i];
                            break;
                        }
                        r += b[i];
                    }
                }
            } else {
                run += block;
            }
        }
        if (lane == 0) {
            if (!found) {
                sh.res[0] = 0;
                sh.res[1] = run;
                sh.res[2] = 0;
            }
            sh.res[3] = found ? 1u : 0u;
        }
    }
    __syncthreads();
    return Threshold{sh.res[0], sh.res[1], sh.res[2], sh.res[3] != 0};
}

__device__ __forceinline__ void clear_hist(uint32_t* h, int nb) {
    for (int i = threadIdx.x; i < nb / 4; i += kThreads) reinterpret_cast<uint4*>(h)[i] = make_uint4(0, 0, 0, 0);
}

// Sum over the CTA of h[c] for c >= from (bins of the local histogram).
__device__ uint32_t count_from(const uint32_t* h, int nb, uint32_t from, const Shared& sh) {
    uint32_t s = 0;
    for (int c = threadIdx.x; c < nb; c += kThreads)
        if (static_cast<uint32_t>(c) >= from) s += h[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
    __syncthreads();
    if (lane_id() == 0) sh.red[threadIdx.x >> 5] = s;
    __syncthreads();
    uint32_t t = 0;
    for (int w = 0; w < kWarps; ++w) t += sh.red[w];
    __syncthreads();
    return t;
}

// ----------------------------------------------------------------------------
// merge policies: a single CTA, or a thread-block cluster over DSMEM
// ----------------------------------------------------------------------------

struct SoloMerge {
    static constexpr bool kSolo = true;
    __device__ __forceinline__ const uint32_t* merge(const Shared& sh, int) const {
        __syncthreads();
        return sh.hist;
    }
    // The level-1 merge: this CTA's bound and overflow flag are the row's.
    __device__ __forceinline__ const uint32_t* merge_level1(const Shared& sh, uint32_t bound, bool ovf,
                                                            uint32_t& max_bound, bool& any_ovf) const {
        max_bound = bound;
        any_ovf = ovf;
        return merge(sh, kBins);
    }
    __device__ __forceinline__ uint32_t* counter(const Shared& sh, int i) const { return &sh.cnt[i]; }
};

struct ClusterMerge {
    static constexpr bool kSolo = false;
    // hist (local) -> mhist (sum over the cluster), identical in every CTA.
    // CTA r sums the 16-byte words w = r, r + kClusterSize, ... over all CTAs
    // (reduce-scatter); then every CTA gathers the words it does not own.
    __device__ const uint32_t* merge(const Shared& sh, int nb) const {
        cg::this_cluster().sync();  // every local histogram is complete
        return merge_words(sh, 0, nb / 4);
    }
    // The level-1 merge limited to the bins the slices' candidates occupy:
    // each CTA publishes its bound, its highest occupied bin and its overflow
    // flag, and only 16-byte words from the highest bound to the highest bin
    // are summed (mhist is zero elsewhere: it is cleared at the row's start).
    // Bins below the highest bound cannot hold an exact level-1 threshold.
    __device__ const uint32_t* merge_level1(const Shared& sh, uint32_t bound, bool ovf, uint32_t& max_bound,
                                            bool& any_ovf) const {
        cg::cluster_group cluster = cg::this_cluster();
        // highest occupied bin at or above the bound
        uint32_t top = 0;
        for (int b = kBins - 1 - static_cast<int>(threadIdx.x); b >= static_cast<int>(bound); b -= kThreads)
            if (sh.hist[b] != 0u) {
                top = static_cast<uint32_t>(b);
                break;
            }
        top = __reduce_max_sync(kFull, top);
        if (lane_id() == 0 && top != 0u) atomicMax(&sh.cnt[5], top);
        if (threadIdx.x == 0) {
            sh.cnt[4] = bound;
            sh.cnt[6] = ovf ? 1u : 0u;
        }
        cluster.sync();  // every local histogram and every published word is complete
        uint32_t lo = 0, hi = 0, o = 0;
#pragma unroll
        for (int q = 0; q < kClusterSize; ++q) {
            const uint32_t* c = cluster.map_shared_rank(sh.cnt, q);
            lo = max(lo, c[4]);
            hi = max(hi, c[5]);
            o |= c[6];
        }
        max_bound = lo;
        any_ovf = o != 0u;
        hi = max(hi, lo);
        return merge_words(sh, static_cast<int>(lo / 4), static_cast<int>(hi / 4) + 1);
    }
    // Sums the 16-byte words [w0, w1) of the CTAs' histograms into mhist; the
    // CTAs must have passed a cluster barrier since their last histogram write.
    __device__ const uint32_t* merge_words(const Shared& sh, int w0, int w1) const {
        cg::cluster_group cluster = cg::this_cluster();
        const int rank = static_cast<int>(cluster.block_rank());
        const int words = w1;
        for (int w = w0 + ((rank - w0 % kClusterSize + kClusterSize) % kClusterSize) +
                     kClusterSize * static_cast<int>(threadIdx.x);
             w < words; w += kClusterSize * kThreads) {
            uint4 t = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int q = 0; q < kClusterSize; ++q) {
                const uint4 r = reinterpret_cast<const uint4*>(cluster.map_shared_rank(sh.hist, q))[w];
                t.x += r.x, t.y += r.y, t.z += r.z, t.w += r.w;
            }
            reinterpret_cast<uint4*>(sh.mhist)[w] = t;
        }
        cluster.sync();  // every owned word of the sum is complete
        for (int w = w0 + static_cast<int>(threadIdx.x); w < words; w += kThreads) {
            const int q = w % kClusterSize;
            if (q != rank)
                reinterpret_cast<uint4*>(sh.mhist)[w] =
                    reinterpret_cast<const uint4*>(cluster.map_shared_rank(sh.mhist, q))[w];
        }
        __syncthreads();
        return sh.mhist;
    }
    __device__ __forceinline__ uint32_t* counter(const Shared& sh, int i) const {
        return cg::this_cluster().map_shared_rank(&sh.cnt[i], 0);
    }
};

// ----------------------------------------------------------------------------
// element sources: registers, the candidate buffer, global memory
// ----------------------------------------------------------------------------

// Register tile: v[u] holds vector j = u*kThreads + tid of the aligned window.
template <int NV>
struct RegSource {
    const float4 (&v)[NV];
    int rem, len;
    template <class F>
    __device__ __forceinline__ void visit(F&& f) const {
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            const int j = u * kThreads + static_cast<int>(threadIdx.x);
            const int p0 = 4 * j - rem;
            const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int p = p0 + c;
                f(score_key(e[c]), p, static_cast<unsigned>(p) < static_cast<unsigned>(len));
            }
        }
    }
};

struct CandSource {
    const uint32_t* key;
    const int32_t* pos;
    uint32_t n;
    template <class F>
    __device__ __forceinline__ void visit(F&& f) const {
        const uint32_t n_round = (n + kThreads - 1) / kThreads * kThreads;
        for (uint32_t i = threadIdx.x; i < n_round; i += kThreads) {
            const bool valid = i < n;
            f(valid ? key[i] : 0u, valid ? pos[i] : 0, valid);
        }
    }
};

// Global memory: vectors [jb, je) of the aligned window, re-read.
struct GlobalSource {
    const float4* vbase;
    int jb, je, rem, len;
    template <class F>
    __device__ __forceinline__ void visit(F&& f) const {
        for (int j0 = jb; j0 < je; j0 += kTileVecs * kThreads) {
            float4 v[kTileVecs];
#pragma unroll
            for (int u = 0; u < kTileVecs; ++u) {
                const int j = j0 + u * kThreads + static_cast<int>(threadIdx.x);
                v[u] = j < je ? load_stream(vbase + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kTileVecs; ++u) {
                const int j = j0 + u * kThreads + static_cast<int>(threadIdx.x);
                const int p0 = 4 * j - rem;
                const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int p = p0 + c;
                    f(score_key(e[c]), p, j < je && static_cast<unsigned>(p) < static_cast<unsigned>(len));
                }
            }
        }
    }
};

// ----------------------------------------------------------------------------
// selection state and the radix levels
// ----------------------------------------------------------------------------

// After the levels: an element whose composite, masked to the resolved high
// bits, exceeds `prefix` is selected; one equal to `prefix` belongs to the
// threshold group, of which `need` are selected (all of them when `exact`).
struct SelState {
    uint64_t prefix;
    uint64_t mask;
    uint32_t need;
    bool exact;
};

__device__ __forceinline__ void apply_level(SelState& st, int lvl, const Threshold& t) {
    const int shift = level_shift(lvl);
    const uint64_t digit_mask = static_cast<uint64_t>(level_bins(lvl) - 1);
    st.need -= t.above;
    st.prefix |= static_cast<uint64_t>(t.bin) << shift;
    st.mask |= digit_mask << shift;
    st.exact = (t.count == st.need);
}

// Levels first..last of the radix descent, stopping once exact. A key level
// also counts, in the word after its bins, the elements of the current group
// with any key bit below its digit set; when the merged count is 0 every such
// bit is 0 throughout the group (scores rounded to bf16 or coarser), so the
// key is settled and the remaining key levels are skipped.
template <class Merge, class Src>
__device__ void run_levels(SelState& st, int first, int last, const Src& src, const Shared& sh,
                           const Merge& mg) {
    for (int lvl = first; lvl <= last && !st.exact; ++lvl) {
        const int nb = level_bins(lvl);
        const int shift = level_shift(lvl);
        uint32_t* hist = sh.hist;
        const uint32_t digit = static_cast<uint32_t>(nb - 1);
        const bool key_level = lvl < kKeyLevels;
        const int words = key_level ? nb + 4 : nb;
        clear_hist(sh.hist, words);
        __syncthreads();
        uint32_t below = 0;
        if (key_level) {  // key digits: a 32-bit filter on the resolved key bits
            const uint32_t pfx = static_cast<uint32_t>(st.prefix >> 32), msk = static_cast<uint32_t>(st.mask >> 32);
            const int sh32 = shift - 32;
            below = (1u << sh32) - 1u;
            uint32_t nz = 0;
            src.visit([&](uint32_t key, int32_t, bool valid) {
                if (valid && (key & msk) == pfx) {
                    atomicAdd(&hist[(key >> sh32) & digit], 1u);
                    nz += (key & below) != 0u;
                }
            });
            nz = __reduce_add_sync(kFull, nz);
            if (lane_id() == 0 && nz != 0) atomicAdd(&hist[nb], nz);
        } else {  // position digits of the elements tied at the threshold
            const uint64_t prefix = st.prefix, mask = st.mask;
            src.visit([&](uint32_t key, int32_t pos, bool valid) {
                const uint64_t c = composite(key, pos);
                if (valid && (c & mask) == prefix) atomicAdd(&hist[static_cast<uint32_t>(c >> shift) & digit], 1u);
            });
        }
        const uint32_t* merged = mg.merge(sh, words);
        const bool settled = key_level && merged[nb] == 0u;  // read before find's barrier
        const Threshold t = find_threshold(merged, nb, st.need, sh);
        apply_level(st, lvl, t);
        if (settled && lvl < kKeyLevels - 1) {
            st.mask |= static_cast<uint64_t>(below) << 32;  // those bits are 0 in the prefix too
            lvl = kKeyLevels - 1;
        }
    }
}

// Output transform of one selected position.
template <bool kPaged>
struct Emitter {
    int32_t* out;
    int32_t* out_raw;
    const int32_t* pt_row;     // the row's page-table row (packed rows: its request's)
    const int32_t* pt_cached;  // the row's page-table entries from pt_first on, in shared memory, or null
    int32_t token0;            // page-table token of position 0 (0 unless packed)
    int32_t pt_first;          // first page-table entry the window touches
    int32_t page_bits;
    int32_t offset;
    uint32_t k;
    uint32_t* flags;  // device flags word of the workspace
    __device__ __forceinline__ void write(uint32_t slot, int32_t pos) const {
        if (slot >= k) {  // never taken when the selection is consistent
            atomicOr(flags, TOPK_DEVICE_FLAG_INTERNAL);
            return;
        }
        int32_t v;
        if (kPaged) {
            const int32_t t = pos + token0;
            const int32_t page = pt_cached ? pt_cached[(t >> page_bits) - pt_first] : __ldg(pt_row + (t >> page_bits));
            v = (page << page_bits) | (t & ((1 << page_bits) - 1));
        } else {
            v = pos + offset;
        }
        out[slot] = v;
        if (out_raw) out_raw[slot] = pos;
    }
    // Straight-line form for loops over candidates: writes when `w` (and the
    // slot is in range); every load it makes is in bounds whether or not it
    // writes. The caller reports out-of-range slots (see flag_if).
    __device__ __forceinline__ void write_if(bool w, uint32_t slot, int32_t pos) const {
        const bool ok = w && slot < k;
        int32_t v;
        if (kPaged) {
            const int32_t t = pos + token0;
            const int32_t q = ok ? (t >> page_bits) : pt_first;  // pt_first exists: the row is not empty
            const int32_t page = pt_cached ? pt_cached[q - pt_first] : __ldg(pt_row + q);
            v = (page << page_bits) | (t & ((1 << page_bits) - 1));
        } else {
            v = pos + offset;
        }
        if (ok) out[slot] = v;
        if (ok && out_raw) out_raw[slot] = pos;
    }
    // Reports an out-of-range slot found by a caller that assigns slots itself.
    __device__ __forceinline__ void flag_if(bool bad) const {
        if (bad) atomicOr(flags, TOPK_DEVICE_FLAG_INTERNAL);
    }
};

// Writes the k selected elements of `src`: definite elements to slots
// [0, k - need), the first `need` members of the threshold group (all of it
// when exact) to [k - need, k). Two visits with the same thread-to-element
// assignment: the first counts each thread's elements of both kinds, a
// block-wide exclusive scan (plus, on a cluster, one atomic per CTA on the
// leader's counters) gives every thread its first slots, the second writes.
template <bool kPaged, class Merge, class Src>
__device__ void emit_selected(const SelState& st, uint32_t k, const Src& src, const Shared& sh,
                              const Merge& mg, const Emitter<kPaged>& em) {
    // this thread's page-table copies have landed; the barrier after the
    // counting pass publishes them to the CTA
    if (kPaged) asm volatile("cp.async.wait_all;" ::: "memory");
    const uint32_t need = st.need;
    const bool exact = st.exact;
    const bool key_only = static_cast<uint32_t>(st.mask) == 0;  // only key levels ran
    const uint32_t pfx = static_cast<uint32_t>(st.prefix >> 32);
    const uint64_t prefix = st.prefix, mask = st.mask;
    // with a top-aligned mask, "masked key above the prefix" is a plain
    // compare against the prefix (exact) or tau
    auto classify = [&](uint32_t key, int32_t pos, bool valid, bool& def, bool& grp) {
        if (key_only) {
            def = valid && (exact ? key >= pfx : key > pfx);
            grp = valid && !exact && key == pfx;
        } else {
            const uint64_t hi = composite(key, pos) & mask;
            def = valid && (hi > prefix || (exact && hi == prefix));
            grp = valid && !exact && hi == prefix;
        }
    };
    uint32_t nd = 0, ng = 0;
    src.visit([&](uint32_t key, int32_t pos, bool valid) {
        bool d, g;
        classify(key, pos, valid, d, g);
        nd += d;
        ng += g;
    });
    const uint32_t xd = warp_inclusive_scan(nd), xg = warp_inclusive_scan(ng);
    const int warp = static_cast<int>(threadIdx.x >> 5);
    if (lane_id() == 31) {
        sh.red[warp] = xd;
        sh.red[kWarps + warp] = xg;
    }
    __syncthreads();
    uint32_t bd = xd - nd, bg = xg - ng, td = 0, tg = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t rd = sh.red[w], rg = sh.red[kWarps + w];
        bd += w < warp ? rd : 0u;
        bg += w < warp ? rg : 0u;
        td += rd;
        tg += rg;
    }
    if (!Merge::kSolo) {  // this CTA's share of the cluster-wide slot ranges
        __syncthreads();
        if (threadIdx.x == 0) {
            sh.red[0] = td ? atomicAdd(mg.counter(sh, 1), td) : 0u;
            sh.red[1] = tg ? atomicAdd(mg.counter(sh, 2), tg) : 0u;
        }
        __syncthreads();
        bd += sh.red[0];
        bg += sh.red[1];
    }
    src.visit([&](uint32_t key, int32_t pos, bool valid) {
        bool d, g;
        classify(key, pos, valid, d, g);
        if (d) em.write(bd++, pos);
        if (g) {
            if (bg < need) em.write(k - need + bg, pos);
            ++bg;
        }
    });
    __syncthreads();  // red is free again
}

// ----------------------------------------------------------------------------
// routes
// ----------------------------------------------------------------------------

template <bool kPaged>
__device__ void trivial_row(int32_t len, uint32_t k, const Emitter<kPaged>& em) {
    for (uint32_t t = threadIdx.x; t < k; t += kThreads) {
        if (static_cast<int32_t>(t) < len) {
            em.write(t, static_cast<int32_t>(t));
        } else {
            em.out[t] = -1;
            if (em.out_raw) em.out_raw[t] = -1;
        }
    }
}





// Raw bits of one tile: kTileVecs vectors per thread from vector j0 (vectors
// at or past je read as zero bits and are never in the window).
__device__ __forceinline__ void load_bits(int4 (&v)[kTileVecs], const float4* vbase, int j0, int je) {
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
        const int j = j0 + u * kThreads + static_cast<int>(threadIdx.x);
        v[u] = j < je ? load_stream_bits(vbase + j) : make_int4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ int tile_elem(const int4 (&v)[kTileVecs], int e) {
    const int4 q = v[e / 4];
    return (e % 4) == 0 ? q.x : (e % 4) == 1 ? q.y : (e % 4) == 2 ? q.z : q.w;
}

// Bit e set: element e of this thread's tile at vector j0 lies in the window
// (vector u of the tile holds positions 4j - rem .. 4j - rem + 3 for
// j = j0 + u * kThreads + tid; vectors at or past je are not in it).
__device__ __forceinline__ uint32_t tile_valid(int j0, int je, int rem, int len) {
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
        const int j = j0 + u * kThreads + static_cast<int>(threadIdx.x);
        const int lo = 4 * j - rem;
        const int a = max(-lo, 0), b = min(len - lo, 4);  // lanes [a, b) are in the window
        const uint32_t vm = (j < je && a < b) ? (1u << b) - (1u << a) : 0u;
        m |= vm << (4 * u);
    }
    return m;
}

// Bit mask of the tile's elements whose key is at least bound_key (tile_ge),
// by one compare of the raw bits per element: for bound_key >= 2^31 (a
// non-negative bound) key >= bound_key <=> bits >= bound_key ^ 2^31 as signed
// integers; below it, key >= bound_key <=> bits <= ~bound_key as unsigned
// ones. tile_pass keeps the in-window ones: only a tile that reaches past
// either end of the window is masked.
__device__ __forceinline__ uint32_t tile_ge(const int4 (&v)[kTileVecs], uint32_t bound_key) {
    uint32_t pass = 0;
    if (bound_key >= 0x80000000u) {
        const int32_t bb = static_cast<int32_t>(bound_key ^ 0x80000000u);
#pragma unroll
        for (int e = 0; e < 4 * kTileVecs; ++e) pass |= static_cast<uint32_t>(tile_elem(v, e) >= bb) << e;
    } else {
        const uint32_t ub = ~bound_key;
#pragma unroll
        for (int e = 0; e < 4 * kTileVecs; ++e)
            pass |= static_cast<uint32_t>(static_cast<uint32_t>(tile_elem(v, e)) <= ub) << e;
    }
    return pass;
}

__device__ __forceinline__ uint32_t tile_pass(const int4 (&v)[kTileVecs], int j0, int je, int rem, int len,
                                              uint32_t bound_key) {
    const uint32_t pass = tile_ge(v, bound_key);
    const bool interior =
        4 * j0 - rem >= 0 && 4 * (j0 + kTileVecs * kThreads) - rem <= len && j0 + kTileVecs * kThreads <= je;
    return interior ? pass : pass & tile_valid(j0, je, rem, len);
}

// Element e of the tile with e known only at run time: a select tree over the
// registers (no local-memory copy of the tile).
__device__ __forceinline__ int tile_elem_at(const int4 (&v)[kTileVecs], int e) {
    static_assert(kTileVecs == 4, "select tree for four vectors");
    const int c = e & 3;
    const bool hi = (e & 8) != 0, odd = (e & 4) != 0;
    const int4 a = hi ? v[2] : v[0], b = hi ? v[3] : v[1];
    const int4 q = odd ? b : a;
    const int lo2 = (c & 1) ? q.y : q.x, hi2 = (c & 1) ? q.w : q.z;
    return (c & 2) ? hi2 : lo2;
}

// Appends the tile elements flagged in `pass` to the candidate buffer: one
// warp scan and one shared atomic per warp reserve the slots, then each
// thread walks the set bits of its own mask (so a warp's loop runs as many
// times as its busiest lane has candidates, not once per tile element). With
// kCountLevel1 each appended element is also counted in the level-1
// histogram.
constexpr int kCountNone = 0, kCountLevel1 = 1;
template <int kCount = kCountNone>
__device__ __forceinline__ void collect_bits(const int4 (&v)[kTileVecs], uint32_t pass, int j0, int rem,
                                             const Shared& sh) {
    const uint32_t c = __popc(pass);
    const uint32_t incl = warp_inclusive_scan(c);
    const uint32_t total = __shfl_sync(kFull, incl, 31);
    if (total == 0) return;
    uint32_t base = 0;
    if (lane_id() == 31) base = atomicAdd(&sh.cnt[0], total);
    base = __shfl_sync(kFull, base, 31);
    uint32_t idx = base + incl - c;
    const int p0 = 4 * (j0 + static_cast<int>(threadIdx.x)) - rem;  // element 0's position
    for (uint32_t rest = pass; rest != 0; rest &= rest - 1u) {
        const int e = __ffs(static_cast<int>(rest)) - 1;
        const uint32_t kk = bits_key(static_cast<uint32_t>(tile_elem_at(v, e)));
        if (kCount == kCountLevel1) atomicAdd(&sh.hist[kk >> 20], 1u);
        if (idx < static_cast<uint32_t>(kCandCap)) {
            sh.cand_key[idx] = kk;
            sh.cand_pos[idx] = p0 + (e >> 2) * (4 * kThreads) + (e & 3);
        }
        ++idx;
    }
}

// Ranks the threshold bin's elements, n <= kThreads of them in tkey/tpos
// (16-byte aligned, room for n rounded up to 4): the rank of an element is
// the number of bin members whose composite (key, ~position) is larger, and
// the ones ranked below `need` take slots k - need + rank: put(slot, pos)
// stores each one. This settles every
// remaining key and position digit at once (ties go to the lowest position).
// Up to 32 members are ranked by one warp through shuffles. Longer lists are
// padded to a multiple of 4 with entries that rank below everything; each
// element is compared by kThreads / m threads (m = n rounded up to a power of
// two), each over one segment, and the partial ranks meet in the
// shared-memory counters `rank` (n words). A caller's barrier must make the
// lists visible first; the function ends without one.
template <class Put>
__device__ void rank_threshold_bin(uint32_t n, uint32_t need, uint32_t k, uint32_t* tkey, int32_t* tpos,
                                   uint32_t* rank, const Put& put) {
    if (n <= 32u) {  // the usual case: warp 0 alone, the members passed round by shuffles
        if (threadIdx.x < 32) {
            const uint32_t lane = lane_id();
            const uint32_t ki = lane < n ? tkey[lane] : 0u;
            const int32_t pi = lane < n ? tpos[lane] : INT32_MAX;
            uint32_t r = 0;
            for (uint32_t j = 0; j < n; ++j) {
                const uint32_t kj = __shfl_sync(kFull, ki, static_cast<int>(j));
                const int32_t pj = __shfl_sync(kFull, pi, static_cast<int>(j));
                r += static_cast<uint32_t>(kj > ki || (kj == ki && pj < pi));
            }
            if (lane < n && r < need) put(k - need + r, pi);
        }
        return;
    }
    const uint32_t n4 = (n + 3u) & ~3u;
    if (threadIdx.x < n4 - n) {
        tkey[n + threadIdx.x] = 0u;
        tpos[n + threadIdx.x] = INT32_MAX;
    }
    if (threadIdx.x < n) rank[threadIdx.x] = 0u;
    __syncthreads();
    uint32_t m = 32;
    while (m < n) m <<= 1;
    const uint32_t segs = static_cast<uint32_t>(kThreads) / m;
    const uint32_t i = threadIdx.x & (m - 1u), seg = threadIdx.x / m;
    const uint32_t per = (n4 / 4u + segs - 1u) / segs * 4u;
    const uint32_t j0 = seg * per, j1 = min(n4, j0 + per);
    if (i < n && j0 < j1) {
        const uint32_t ki = tkey[i];
        const int32_t pi = tpos[i];
        uint32_t r = 0;
        for (uint32_t j = j0; j < j1; j += 4) {
            const uint4 kj = *reinterpret_cast<const uint4*>(tkey + j);
            const int4 pj = *reinterpret_cast<const int4*>(tpos + j);
            r += static_cast<uint32_t>(kj.x > ki || (kj.x == ki && pj.x < pi));
            r += static_cast<uint32_t>(kj.y > ki || (kj.y == ki && pj.y < pi));
            r += static_cast<uint32_t>(kj.z > ki || (kj.z == ki && pj.z < pi));
            r += static_cast<uint32_t>(kj.w > ki || (kj.w == ki && pj.w < pi));
        }
        atomicAdd(&rank[i], r);
    }
    __syncthreads();
    if (seg == 0 && i < n) {
        const uint32_t r = rank[i];
        if (r < need) put(k - need + r, tpos[i]);
    }
}

// Writes the slot-ordered position list (k entries in shared memory) to the
// output row: thread t takes slots t, t + kThreads, ..., so every warp store
// covers 32 consecutive slots. Follows a barrier that completes the list.
template <bool kPaged>
__device__ __forceinline__ void write_slots(const int32_t* slots, uint32_t k, const Emitter<kPaged>& em) {
    for (uint32_t s = threadIdx.x; s < k; s += kThreads) em.write(s, slots[s]);
}

// The finish of a solo streaming row once level 1 is known and every
// element at or above its threshold bin sits in the candidate buffer (n of
// them): level 2 is histogrammed over the threshold bin's candidates (unless
// level 1 is exact); then one counting pass and one writing pass over the
// buffer send every element above the threshold prefix to its slot (a block
// scan orders them) and copy the elements equal to it to a tie list (in the
// histogram's storage), which rank_threshold_bin orders into the last slots. Returns false,
// having written nothing, when the level-2 threshold bin is too full to rank
// (many equal scores): the caller continues with the radix levels from
// level 3 (st then holds levels 1 and 2).
template <bool kPaged>
__device__ bool finish_candidates(SelState& st, uint32_t bin1, uint32_t n, uint32_t k, const Shared& sh,
                                  const Emitter<kPaged>& em) {
    int shift = 20;
    uint32_t tau = bin1, n_tie = 0;
    if (!st.exact) {
        clear_hist(sh.hist, level_bins(1));
        __syncthreads();
        for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
            const uint32_t kk = sh.cand_key[i];
            if ((kk >> 20) == bin1) atomicAdd(&sh.hist[(kk >> 12) & 0xFFu], 1u);
        }
        __syncthreads();
        const Threshold t2 = find_threshold(sh.hist, level_bins(1), st.need, sh);
        apply_level(st, 1, t2);
        shift = 12;
        tau = (bin1 << 8) | t2.bin;
        n_tie = t2.count;
        if (!st.exact && n_tie > static_cast<uint32_t>(kThreads)) return false;
    }
    if (kPaged) asm volatile("cp.async.wait_all;" ::: "memory");  // published by the barrier below
    const bool exact = st.exact;
    uint32_t c = 0;  // selected in the low half, ties in the high half (n <= kCandCap < 2^16)
    for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t pf = sh.cand_key[i] >> shift;
        c += (exact ? pf >= tau : pf > tau) ? 1u : (!exact && pf == tau) ? 0x10000u : 0u;
    }
    const uint32_t incl = warp_inclusive_scan(c);
    const int warp = static_cast<int>(threadIdx.x >> 5);
    if (lane_id() == 31) sh.red[warp] = incl;
    __syncthreads();
    uint32_t base = incl - c;
    for (int w = 0; w < warp; ++w) base += sh.red[w];
    uint32_t slot = base & 0xFFFFu, tslot = base >> 16;
    uint32_t* tkey = sh.hist;                                  // tie list: kThreads + 4 entries each
    int32_t* tpos = reinterpret_cast<int32_t*>(sh.hist + 2 * kThreads);
    for (uint32_t i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t kk = sh.cand_key[i];
        const uint32_t pf = kk >> shift;
        const bool w = exact ? pf >= tau : pf > tau;
        const bool t = !exact && pf == tau;
        const int32_t pos = sh.cand_pos[i];
        em.write_if(w, slot, pos);
        if (t) {
            tkey[tslot] = kk;
            tpos[tslot] = pos;
        }
        slot += w;
        tslot += t;
    }
    em.flag_if(slot > k - (exact ? 0u : st.need));
    if (!exact) {
        __syncthreads();
        rank_threshold_bin(n_tie, st.need, k, tkey, tpos, sh.cand_key,
                           [&](uint32_t s, int32_t pos) { em.write(s, pos); });
    }
    return true;
}

// The register route's finish once the selection prefix is known: every
// tile element whose prefix (key >> shift) is above tau (at least tau when
// exact) is selected and goes to its slot in a slot-ordered list (one block
// scan of both counts orders the slots), the elements equal to it (not
// exact) go to a tie list in the candidate buffer, which rank_threshold_bin
// orders into the last `need` slots, and the list is written out coalesced.
template <bool kPaged>
__device__ void finish_registers(const int4 (&v)[kTileVecs], uint32_t valid, int rem, int shift, uint32_t tau,
                                 bool exact, uint32_t need, uint32_t n_tie, uint32_t k, const Shared& sh,
                                 const Emitter<kPaged>& em) {
    if (kPaged) asm volatile("cp.async.wait_all;" ::: "memory");  // published by the barrier below
    // prefix >= tau and prefix > tau as raw-bit compares against the
    // smallest keys with prefix tau and tau + 1
    const uint32_t ge_tau = tile_ge(v, tau << shift);
    const bool top_bin = tau + 1u == (1u << (32 - shift));
    const uint32_t gt_tau = (exact || top_bin) ? 0u : tile_ge(v, (tau + 1u) << shift);
    const uint32_t def = (exact ? ge_tau : gt_tau) & valid;
    const uint32_t tie = exact ? 0u : (ge_tau & ~gt_tau & valid);
    // both counts in one scan: selected in the low half, ties in the high
    // half (a CTA holds at most 8192 elements)
    const uint32_t c = static_cast<uint32_t>(__popc(def)) | (static_cast<uint32_t>(__popc(tie)) << 16);
    const uint32_t incl = warp_inclusive_scan(c);
    const int warp = static_cast<int>(threadIdx.x >> 5);
    if (lane_id() == 31) sh.red[warp] = incl;
    __syncthreads();
    uint32_t base = incl - c;
    for (int w = 0; w < warp; ++w) base += sh.red[w];
    uint32_t slot = base & 0xFFFFu, tslot = base >> 16;
    int32_t* slots = reinterpret_cast<int32_t*>(sh.hist + kBins - TOPK_MAX_K);  // slot-ordered positions
    const int32_t p0 = 4 * static_cast<int32_t>(threadIdx.x) - rem;  // position of element 0
    // walk the set bits only (a warp loops as often as its busiest lane)
    for (uint32_t rest = def; rest != 0; rest &= rest - 1u) {
        const int e = __ffs(static_cast<int>(rest)) - 1;
        if (slot < k) slots[slot] = p0 + (e >> 2) * (4 * kThreads) + (e & 3);
        ++slot;
    }
    for (uint32_t rest = tie; rest != 0; rest &= rest - 1u) {
        const int e = __ffs(static_cast<int>(rest)) - 1;
        sh.cand_key[tslot] = bits_key(static_cast<uint32_t>(tile_elem_at(v, e)));
        sh.cand_pos[tslot] = p0 + (e >> 2) * (4 * kThreads) + (e & 3);
        ++tslot;
    }
    em.flag_if(slot > k - (exact ? 0u : need));
    __syncthreads();
    if (!exact) {
        rank_threshold_bin(n_tie, need, k, sh.cand_key, sh.cand_pos, sh.hist,
                           [&](uint32_t s, int32_t pos) { slots[s] = pos; });
        __syncthreads();
    }
    write_slots<kPaged>(slots, k, em);
}

// Register route: the whole aligned window (nv <= kTileVecs * kThreads
// vectors) is one register tile.
//  * The first digit is 14 bits wide: 16384 16-bit counters (two per word,
//    in the candidate buffer's storage), one shared atomic per element. When
//    its threshold bin holds at most kThreads elements (the usual case; about
//    40 for a row of 8192 normal scores), finish_registers writes every
//    element above it to its slot and ranks the bin's members for the rest.
//  * Otherwise (many equal scores) the 12-bit levels run: level 1 from the
//    tile, level 2 over its threshold bin from the registers, the same finish
//    when that bin is small, else the radix levels on the candidate buffer
//    (or on the registers when the bins do not fit it).
template <bool kPaged>
__device__ void register_row(const float4* vbase, int nv, int rem, int len, uint32_t k, bool det,
                             const Shared& sh, const Emitter<kPaged>& em) {
    int4 v[kTileVecs];
    load_bits(v, vbase, 0, nv);  // in flight while the histogram is cleared
    static_assert(kFineWords <= 2 * kCandCap, "the fine histogram lives in the candidate buffer");
    uint32_t* fine = sh.cand_key;
    clear_hist(fine, kFineWords);
    __syncthreads();
    const uint32_t valid = tile_valid(0, nv, rem, len);
#pragma unroll
    for (int e = 0; e < 4 * kTileVecs; ++e) {
        const uint32_t d = bits_key(static_cast<uint32_t>(tile_elem(v, e))) >> kFineShift;
        if ((valid >> e) & 1u) atomicAdd(&fine[d >> 1], (d & 1u) ? 0x10000u : 1u);
    }
    __syncthreads();
    {
        const uint32_t total = find_fine_publish(fine, k, sh);
        __syncthreads();  // the fine bins are read: the candidate buffer is free again
        const Threshold tf = find_wide_result(total, k, sh);
        const uint32_t need = k - tf.above;
        const bool exact = tf.count == need;
        if (exact || tf.count <= static_cast<uint32_t>(kThreads)) {
            finish_registers<kPaged>(v, valid, rem, kFineShift, tf.bin, exact, need, tf.count, k, sh, em);
            return;
        }
    }
    clear_hist(sh.hist, kBins);
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 4 * kTileVecs; ++e)
        if ((valid >> e) & 1u) atomicAdd(&sh.hist[bits_key(static_cast<uint32_t>(tile_elem(v, e))) >> 20], 1u);
    __syncthreads();
    // Level 1; its bins are free once the search has read them, so the
    // level-2 bins are cleared before the barrier that publishes the result.
    const uint32_t total1 = find_wide_publish(sh.hist, k, sh);
    clear_hist(sh.hist, level_bins(1));
    __syncthreads();
    const Threshold t1 = find_wide_result(total1, k, sh);
    SoloMerge mg;
    SelState st{0ull, 0ull, k, false};
    apply_level(st, 0, t1);
    const int last = (det ? kAllLevels : kKeyLevels) - 1;
    // Level 2 inside the threshold bin, histogrammed from the registers.
    int shift = 20;           // the selection prefix is key >> shift ...
    uint32_t tau = t1.bin;    // ... compared with tau
    uint32_t n_tie = 0;
    if (!st.exact) {
#pragma unroll
        for (int e = 0; e < 4 * kTileVecs; ++e) {
            const uint32_t kk = bits_key(static_cast<uint32_t>(tile_elem(v, e)));
            if (((valid >> e) & 1u) && (kk >> 20) == t1.bin) atomicAdd(&sh.hist[(kk >> 12) & 0xFFu], 1u);
        }
        __syncthreads();
        const Threshold t2 = find_threshold(sh.hist, level_bins(1), st.need, sh);
        apply_level(st, 1, t2);
        shift = 12;
        tau = (t1.bin << 8) | t2.bin;
        n_tie = t2.count;
    }
    if (st.exact || n_tie <= static_cast<uint32_t>(kThreads)) {
        finish_registers<kPaged>(v, valid, rem, shift, tau, st.exact, st.need, n_tie, k, sh, em);
        return;
    }
    // A threshold bin too full to rank (many equal scores): the radix levels
    // continue from level 3 on the candidate buffer, or on the registers when
    // the bins at or above the level-1 threshold do not fit it.
    if (t1.above + t1.count <= static_cast<uint32_t>(kCandCap)) {
        __syncthreads();
        collect_bits(v, tile_pass(v, 0, nv, rem, len, t1.bin << 20), 0, rem, sh);
        __syncthreads();
        const CandSource src{sh.cand_key, sh.cand_pos, min(sh.cnt[0], static_cast<uint32_t>(kCandCap))};
        run_levels(st, 2, last, src, sh, mg);
        emit_selected<kPaged>(st, k, src, sh, mg, em);
    } else {
        float4 f[kTileVecs];
#pragma unroll
        for (int u = 0; u < kTileVecs; ++u)
            f[u] = make_float4(__int_as_float(v[u].x), __int_as_float(v[u].y), __int_as_float(v[u].z),
                               __int_as_float(v[u].w));
        const RegSource<kTileVecs> src{f, rem, len};
        run_levels(st, 2, last, src, sh, mg);
        emit_selected<kPaged>(st, k, src, sh, mg, em);
    }
}

// Number of window positions p in [4*ja - rem, 4*jb - rem) (vectors [ja, jb)).
__device__ __forceinline__ int window_count(int ja, int jb, int rem, int len) {
    const int lo = max(4 * ja - rem, 0), hi = min(4 * jb - rem, len);
    return max(hi - lo, 0);
}


// Streaming route over vectors [jb, je) of the aligned window: the whole row
// on one CTA, or this CTA's slice of a row cut over a thread-block cluster.
//  1. The slice's head tile gets a full level-1 histogram, which sets the
//     slice's own lower bound on the threshold bin, aiming about 4 sigma
//     above the slice head's expected share of the top-k (no cluster
//     exchange).
//  2. One pass over the rest collects every element at or above the bound.
//  3. Level 1 comes from the merged histograms (on a cluster, merged only
//     over the bins the slices' candidates occupy). It is exact when its
//     threshold bin clears every slice's bound (each slice's counts are
//     exact from its bound up); otherwise, or if a buffer overflowed, a full
//     histogram pass and a re-collection run (always exact, only slower).
//  4. Solo rows finish with finish_candidates; cluster rows run the radix
//     levels and emit_selected over the slices' candidate buffers.
template <bool kPaged, class Merge>
__device__ void streaming_row(const float4* vbase, int jb, int je, int rem, int len, uint32_t k, bool det,
                              const Shared& sh, const Merge& mg, const Emitter<kPaged>& em) {
    constexpr int T = kTileVecs * kThreads;
    int4 cur[kTileVecs], nxt[kTileVecs];
    load_bits(cur, vbase, jb, je);                   // the head tile
    if (jb + T < je) load_bits(nxt, vbase, jb + T, je);  // the next tile is in flight meanwhile
    {
        const uint32_t valid = tile_valid(jb, je, rem, len);
#pragma unroll
        for (int e = 0; e < 4 * kTileVecs; ++e)
            if ((valid >> e) & 1u) atomicAdd(&sh.hist[bits_key(static_cast<uint32_t>(tile_elem(cur, e))) >> 20], 1u);
    }
    __syncthreads();  // the head histogram is complete
    // this part's lower bound, from its own head tile
    const int n_head = window_count(jb, min(je, jb + T), rem, len);
    uint32_t bound_bin = 0;
    if (n_head > 0) {
        const float expect = static_cast<float>(k) * static_cast<float>(n_head) / static_cast<float>(len);
        const float tgt = fminf(expect + 4.0f * sqrtf(expect) + 16.0f, static_cast<float>(n_head));
        bound_bin = find_threshold(sh.hist, kBins, max(static_cast<uint32_t>(tgt), 1u), sh).bin;
    }
    const uint32_t bound_key = bound_bin << 20;
    collect_bits(cur, tile_pass(cur, jb, je, rem, len, bound_key), jb, rem, sh);
    // two register tiles in turn: one is collected while the next loads
    for (int j0 = jb + T; j0 < je;) {
        if (j0 + T < je) load_bits(cur, vbase, j0 + T, je);
        collect_bits<kCountLevel1>(nxt, tile_pass(nxt, j0, je, rem, len, bound_key), j0, rem, sh);
        j0 += T;
        if (j0 >= je) break;
        if (j0 + T < je) load_bits(nxt, vbase, j0 + T, je);
        collect_bits<kCountLevel1>(cur, tile_pass(cur, j0, je, rem, len, bound_key), j0, rem, sh);
        j0 += T;
    }
    __syncthreads();
    // Each part's histogram holds every head-tile element and every candidate
    // after it, so its counts are exact for every bin at or above its bound;
    // the merged level 1 is exact when its threshold bin clears every part's
    // bound.
    uint32_t max_bound = 0;
    bool overflow = false;
    const uint32_t* merged =
        mg.merge_level1(sh, bound_bin, sh.cnt[0] > static_cast<uint32_t>(kCandCap), max_bound, overflow);
    Threshold t1 = find_threshold(merged, kBins, k, sh);
    bool cands_ok = true;
    if (overflow || !t1.found || t1.bin < max_bound) {  // uniform over a cluster
        // full level-1 histogram of this CTA's elements, then re-collect
        clear_hist(sh.hist, kBins);
        __syncthreads();
        uint32_t* hist = sh.hist;
        const GlobalSource all{vbase, jb, je, rem, len};
        all.visit([&](uint32_t kk, int32_t, bool valid) {
            if (valid) atomicAdd(&hist[kk >> 20], 1u);
        });
        merged = mg.merge(sh, kBins);
        t1 = find_threshold(merged, kBins, k, sh);
        cands_ok = false;
        if (count_from(sh.hist, kBins, t1.bin, sh) <= static_cast<uint32_t>(kCandCap)) {
            if (threadIdx.x == 0) sh.cnt[0] = 0;
            __syncthreads();
            for (int j0 = jb; j0 < je; j0 += T) {
                load_bits(cur, vbase, j0, je);
                collect_bits(cur, tile_pass(cur, j0, je, rem, len, t1.bin << 20), j0, rem, sh);
            }
            __syncthreads();
            cands_ok = true;
        }
    }
    SelState st{0ull, 0ull, k, false};
    apply_level(st, 0, t1);
    const int last = (det ? kAllLevels : kKeyLevels) - 1;
    if (cands_ok) {
        const CandSource src{sh.cand_key, sh.cand_pos, min(sh.cnt[0], static_cast<uint32_t>(kCandCap))};
        int first = 1;
        if (Merge::kSolo) {
            if (finish_candidates<kPaged>(st, t1.bin, src.n, k, sh, em)) return;
            first = 2;
        }
        run_levels(st, first, last, src, sh, mg);
        emit_selected<kPaged>(st, k, src, sh, mg, em);
    } else {
        const GlobalSource src{vbase, jb, je, rem, len};
        run_levels(st, 1, last, src, sh, mg);
        emit_selected<kPaged>(st, k, src, sh, mg, em);
    }
}

// ----------------------------------------------------------------------------
// kernels
// ----------------------------------------------------------------------------

// Programmatic dependent launch. Every kernel here is launched so that it may
// be scheduled while the previous kernel on the stream is still running, and
// reads or writes no global memory before grid_dependency_wait(), which
// returns once the previous kernels have completed and their writes are
// visible: stream order is kept, only the launch latency is hidden.
// allow_dependents() lets the next kernel on the stream be scheduled early
// under the same rule (a kernel launched without the attribute is unaffected).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ bool plan_matches(const Params& p) {
    const PlanHeader* h = p.hdr;
    return h->magic == kPlanMagic && h->batch == p.batch && h->k == p.k;
}

template <bool kPaged>
__device__ __forceinline__ Emitter<kPaged> make_emitter(const Params& p, int b, int32_t offset, int32_t table_row,
                                                        int32_t token0) {
    Emitter<kPaged> em;
    em.out = p.out + static_cast<int64_t>(b) * p.k;
    em.out_raw = p.out_raw ? p.out_raw + static_cast<int64_t>(b) * p.k : nullptr;
    em.pt_row = kPaged ? p.page_table + static_cast<int64_t>(table_row) * p.page_table_stride : nullptr;
    em.pt_cached = nullptr;
    em.token0 = token0;
    em.pt_first = kPaged ? (token0 >> p.page_bits) : 0;
    em.page_bits = p.page_bits;
    em.offset = offset;
    em.k = static_cast<uint32_t>(p.k);
    em.flags = &p.hdr->flags;
    return em;
}

// PAGED, non-trivial row: starts asynchronous copies of the page-table
// entries its window's tokens token0 .. token0 + len - 1 map to (each one a
// page some window position maps to) into shared memory when they fit; the
// emit waits for them.
template <bool kPaged>
__device__ __forceinline__ void prefetch_pages(Emitter<kPaged>& em, int32_t len, const Shared& sh) {
    if (!kPaged) return;
    const int n = ((em.token0 + len - 1) >> em.page_bits) - em.pt_first + 1;
    if (n > kPageCache) return;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(sh.pages + i));
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(em.pt_row + em.pt_first + i)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    em.pt_cached = sh.pages;
}

// One CTA per row; rows come from the plan's order (longest first), rows the
// plan gave to the cluster path are skipped (their CTAs exit at once).
// kMinBlocks = 2 keeps two CTAs per SM (64 registers a thread); batches that
// fit one CTA per SM use kMinBlocks = 1, which lets the code keep more in
// registers.
template <bool kPaged, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) topk_rows_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const Shared sh = carve(smem, false);
    grid_dependency_wait();
    allow_dependents();
    // The header, this CTA's order entry and the row data of row blockIdx.x
    // are read together: when the plan kept rows in place (a batch in one
    // length band) the row is blockIdx.x and no second round trip is needed.
    // (blockIdx.x < batch, so every read is in bounds.)
    const int b0 = static_cast<int>(blockIdx.x);
    const PlanHeader* hdr = p.hdr;
    const uint32_t magic = hdr->magic;
    const int32_t h_batch = hdr->batch, h_k = hdr->k, n_order = hdr->n_order;
    const int32_t ord = p.order[b0];
    const int32_t len0 = p.seq_lens[b0];
    const int32_t start0 = p.row_starts ? p.row_starts[b0] : 0;
    const int32_t off0 = kPaged ? 0 : p.out_offsets[b0];
    const int32_t table0 = (kPaged && p.row_to_batch) ? p.row_to_batch[b0] : b0;
    const int32_t token00 = (kPaged && p.pt_row_starts) ? p.pt_row_starts[b0] : 0;
    const bool planned = magic == kPlanMagic && h_batch == p.batch && h_k == p.k;
    if (threadIdx.x < 4) sh.res[threadIdx.x] = 0;
    int b = b0;
    if (planned) {
        if (b0 >= n_order) return;
        b = ord;
    } else if (blockIdx.x == 0 && threadIdx.x == 0) {
        atomicOr(&p.hdr->flags, TOPK_DEVICE_FLAG_PLAN_MISMATCH);
    }
    const bool same = b == b0;
    int32_t len = same ? len0 : p.seq_lens[b];
    const int32_t start = same ? start0 : (p.row_starts ? p.row_starts[b] : 0);
    const int32_t offset = kPaged ? 0 : (same ? off0 : p.out_offsets[b]);
    const int32_t table_row = same ? table0 : ((kPaged && p.row_to_batch) ? p.row_to_batch[b] : b);
    const int32_t token0 = same ? token00 : ((kPaged && p.pt_row_starts) ? p.pt_row_starts[b] : 0);
    if (len < 0 || start < 0 || token0 < 0) {
        // seq_len < 0 was counted by the plan; count the rest here
        if (threadIdx.x == 0 && (!planned || len >= 0)) atomicAdd(&p.hdr->error_rows, 1u);
        len = 0;
    }
    const uint32_t k = static_cast<uint32_t>(p.k);
    Emitter<kPaged> em = make_emitter<kPaged>(p, b, offset, table_row, token0 < 0 ? 0 : token0);
    if (len <= p.k) {
        trivial_row<kPaged>(len, k, em);
        return;
    }
    prefetch_pages<kPaged>(em, len, sh);
    if (threadIdx.x < 8) sh.cnt[threadIdx.x] = 0;
    const int rem = start & 3;
    const float4* vbase = reinterpret_cast<const float4*>(
        p.scores + static_cast<int64_t>(b) * p.score_stride + (start - rem));
    const int nv = (len + rem + 3) >> 2;
    const bool det = (p.flags & TOPK_DETERMINISTIC) != 0;
    if (nv <= kTileVecs * kThreads) {
        register_row<kPaged>(vbase, nv, rem, len, k, det, sh, em);
    } else {
        clear_hist(sh.hist, kBins);
        __syncthreads();
        streaming_row<kPaged>(vbase, 0, nv, rem, len, k, det, sh, SoloMerge{}, em);
    }
}

// One thread-block cluster per long row (looping over the plan's cluster list).
// As for the rows kernel, kMinBlocks = 1 (no 64-register cap) serves launches
// whose clusters all fit one CTA per SM.
template <bool kPaged, int kMinBlocks>
__global__ void __cluster_dims__(kClusterSize, 1, 1) __launch_bounds__(kThreads, kMinBlocks)
    topk_cluster_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const Shared sh = carve(smem, true);
    grid_dependency_wait();
    allow_dependents();
    if (threadIdx.x < 4) sh.res[threadIdx.x] = 0;
    if (!plan_matches(p)) return;  // uniform over the cluster: no barrier is skipped
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int n_slots = static_cast<int>(gridDim.x) / kClusterSize;
    const int slot = static_cast<int>(blockIdx.x) / kClusterSize;
    const int n_rows = p.hdr->n_cluster;
    const ClusterMerge mg;
    const bool det = (p.flags & TOPK_DETERMINISTIC) != 0;
    const uint32_t k = static_cast<uint32_t>(p.k);
    for (int i = slot; i < n_rows; i += n_slots) {
        const int b = p.cluster_rows[i];
        int32_t len = p.seq_lens[b];
        const int32_t start = p.row_starts ? p.row_starts[b] : 0;
        const int32_t table_row = (kPaged && p.row_to_batch) ? p.row_to_batch[b] : b;
        const int32_t token0 = (kPaged && p.pt_row_starts) ? p.pt_row_starts[b] : 0;
        if (len < 0 || start < 0 || token0 < 0) {
            // seq_len < 0 was counted by the plan (cluster rows have seq_len > 32768)
            if (rank == 0 && threadIdx.x == 0 && len >= 0) atomicAdd(&p.hdr->error_rows, 1u);
            len = 0;
        }
        Emitter<kPaged> em =
            make_emitter<kPaged>(p, b, kPaged ? 0 : p.out_offsets[b], table_row, token0 < 0 ? 0 : token0);
        if (len <= p.k) {
            if (rank == 0) trivial_row<kPaged>(len, k, em);
            cluster.sync();
            continue;
        }
        prefetch_pages<kPaged>(em, len, sh);
        if (threadIdx.x < 8) sh.cnt[threadIdx.x] = 0;
        clear_hist(sh.hist, kBins);
        clear_hist(sh.mhist, kBins);
        const int rem = start & 3;
        const float4* vbase = reinterpret_cast<const float4*>(
            p.scores + static_cast<int64_t>(b) * p.score_stride + (start - rem));
        const int nv = (len + rem + 3) >> 2;
        const int per = (nv + kClusterSize - 1) / kClusterSize;
        const int jb = min(nv, rank * per);
        const int je = min(nv, jb + per);
        // counters of the leader CTA must be zero before any CTA emits: the
        // merges below pass several cluster barriers first
        __syncthreads();
        streaming_row<kPaged>(vbase, jb, je, rem, len, k, det, sh, mg, em);
        cluster.sync();  // all emits done before the leader's counters are reset
    }
}

// Plan: bands rows by length (longest first), lists rows for the cluster path,
// counts seq_len < 0. A batch whose rows all fall in one band keeps its order
// (order[i] = i), which lets the rows kernel read its row's data without
// waiting for the order entry.
__device__ __forceinline__ int band_of(int32_t len, int32_t k, bool allow_cluster) {
    if (len <= k) return kBandTrivial;
    if (allow_cluster && len > kClusterFloor) return kBandCluster;
    return __clz(len);  // 31 - floor(log2 len): longer rows get lower bands, go first
}

__global__ void __launch_bounds__(kPlanThreads) topk_plan_kernel(const int32_t* seq_lens, int32_t batch,
                                                                 int32_t k, PlanHeader* hdr,
                                                                 int32_t* order, int32_t* cluster_rows) {
    __shared__ uint32_t count[kBands];
    __shared__ uint32_t offset[kBands];
    __shared__ uint32_t n_err;
    __shared__ bool in_place;
    grid_dependency_wait();
    allow_dependents();
    const int tid = static_cast<int>(threadIdx.x);
    if (tid < kBands) count[tid] = 0;
    if (tid == 0) n_err = 0;
    __syncthreads();
    const bool allow_cluster = batch <= kClusterMaxBatch;
    const int nt = static_cast<int>(blockDim.x);  // a multiple of 32, at least 64
    const int n_iter = (batch + nt - 1) / nt;
    const uint32_t lt = lanemask_lt();
    for (int it = 0; it < n_iter; ++it) {
        const int i = it * nt + tid;
        const bool valid = i < batch;
        const int32_t len = valid ? seq_lens[i] : 0;
        const uint32_t merr = __ballot_sync(kFull, valid && len < 0);
        if (lane_id() == 0 && merr) atomicAdd(&n_err, __popc(merr));
        const int band = valid ? band_of(max(len, 0), k, allow_cluster) : kBands;
        const uint32_t peers = __match_any_sync(kFull, band);
        if (valid && (peers & lt) == 0) atomicAdd(&count[band], __popc(peers));
    }
    __syncthreads();
    if (tid < 32) {  // band offsets: warp 0, lane l holding bands 2l and 2l + 1
        static_assert(kBandTrivial + 1 <= 64, "two ordered bands per lane");
        const int b0 = 2 * tid, b1 = 2 * tid + 1;
        const uint32_t c0 = b0 <= kBandTrivial ? count[b0] : 0u, c1 = b1 <= kBandTrivial ? count[b1] : 0u;
        const uint32_t incl = warp_inclusive_scan(c0 + c1);
        const uint32_t excl = incl - c0 - c1;
        if (b0 <= kBandTrivial) offset[b0] = excl;
        if (b1 <= kBandTrivial) offset[b1] = excl + c0;
        const uint32_t run = __shfl_sync(kFull, incl, 31);
        // one band holds every row: the rows keep their own order
        const bool one_band = __any_sync(kFull, (b0 <= kBandTrivial && c0 == static_cast<uint32_t>(batch)) ||
                                                    (b1 <= kBandTrivial && c1 == static_cast<uint32_t>(batch)));
        if (tid == 0) {
            offset[kBandCluster] = 0;
            in_place = one_band;
            hdr->n_order = static_cast<int32_t>(run);
            hdr->n_cluster = static_cast<int32_t>(count[kBandCluster]);
            hdr->error_rows = n_err;
            hdr->flags = 0;
            hdr->batch = batch;
            hdr->k = k;
            hdr->magic = kPlanMagic;
        }
    }
    __syncthreads();
    if (in_place) {
        for (int i = tid; i < batch; i += nt) order[i] = i;
        return;
    }
    for (int it = 0; it < n_iter; ++it) {
        const int i = it * nt + tid;
        const bool valid = i < batch;
        const int32_t len = valid ? seq_lens[i] : 0;
        const int band = valid ? band_of(max(len, 0), k, allow_cluster) : kBands;
        const uint32_t peers = __match_any_sync(kFull, band);
        const int leader = __ffs(peers) - 1;
        uint32_t base = 0;
        if (valid && static_cast<int>(lane_id()) == leader) base = atomicAdd(&offset[band], __popc(peers));
        base = __shfl_sync(kFull, base, leader);
        if (valid) {
            const uint32_t slot = base + __popc(peers & lt);
            if (band == kBandCluster) cluster_rows[slot] = i;
            else order[slot] = i;
        }
    }
}

// ----------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------

struct DeviceState {
    bool ready = false;
    cudaError_t err = cudaSuccess;
    int max_clusters = 0;       // co-resident clusters of the two-CTA-per-SM cluster build
    int max_clusters_wide = 0;  // ... of the one-CTA-per-SM build
    int sms = 0;                // streaming multiprocessors
};

constexpr int kMaxDevices = 64;
DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;

// Shared-memory size and co-resident cluster count of one cluster-kernel build.
template <bool kPaged, int kMinBlocks>
cudaError_t prepare_cluster_kernel(int& max_clusters) {
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel<kPaged, kMinBlocks>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmemCluster));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterSize, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemCluster;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterSize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel<kPaged, kMinBlocks>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();  // the query is advisory: fall back to a conservative count
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = sms > 2 * kClusterSize ? sms / (2 * kClusterSize) : 1;
    }
    max_clusters = max_clusters == 0 ? n : min(max_clusters, n);
    return cudaSuccess;
}

template <bool kPaged>
cudaError_t prepare_kernels(int& max_clusters, int& max_clusters_wide) {
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<kPaged, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemRows));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_rows_kernel<kPaged, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemRows));
    if (e != cudaSuccess) return e;
    e = prepare_cluster_kernel<kPaged, 2>(max_clusters);
    if (e != cudaSuccess) return e;
    return prepare_cluster_kernel<kPaged, 1>(max_clusters_wide);
}

cudaError_t device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& st = g_devices[dev];
    if (!st.ready) {
        int mc = 0, mcw = 0;
        e = prepare_kernels<true>(mc, mcw);
        if (e == cudaSuccess) e = prepare_kernels<false>(mc, mcw);
        if (e != cudaSuccess) return e;
        st.max_clusters = mc > 0 ? mc : 1;
        st.max_clusters_wide = mcw > 0 ? mcw : 1;
        e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        st.ready = true;
    }
    *out = &st;
    return cudaSuccess;
}

bool valid_k(int32_t k) { return k >= 1 && k <= TOPK_MAX_K; }

// Launches with the programmatic-stream-serialization attribute (see
// grid_dependency_wait); a cluster kernel's shape comes from __cluster_dims__.
template <class... Args, class... Vals>
cudaError_t launch_pdl(void (*kernel)(Args...), int grid, int block, size_t smem, cudaStream_t stream,
                       Vals... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(block), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <bool kPaged>
int launch_transform(const Params& prm, cudaStream_t stream) {
    DeviceState* ds = nullptr;
    if (device_state(&ds) != cudaSuccess) return TOPK_ERR_CUDA;
    const cudaError_t le =
        prm.batch <= ds->sms ? launch_pdl(topk_rows_kernel<kPaged, 1>, prm.batch, kThreads, kSmemRows, stream, prm)
                             : launch_pdl(topk_rows_kernel<kPaged, 2>, prm.batch, kThreads, kSmemRows, stream, prm);
    if (le != cudaSuccess) return TOPK_ERR_CUDA;
    if (prm.batch <= kClusterMaxBatch) {
        // every row's cluster resident at once with one CTA per SM: the wide build
        const cudaError_t ce =
            prm.batch <= ds->max_clusters_wide
                ? launch_pdl(topk_cluster_kernel<kPaged, 1>, kClusterSize * prm.batch, kThreads, kSmemCluster, stream,
                             prm)
                : launch_pdl(topk_cluster_kernel<kPaged, 2>, kClusterSize * min(prm.batch, ds->max_clusters),
                             kThreads, kSmemCluster, stream, prm);
        if (ce != cudaSuccess) return TOPK_ERR_CUDA;
    }
    return TOPK_OK;
}

int common_checks(const float* scores, int64_t score_stride, const int32_t* seq_lens, int32_t batch,
                  int32_t k, void* workspace, size_t workspace_bytes, int32_t* out, uint32_t flags) {
    if (!valid_k(k)) return TOPK_ERR_K;
    if ((flags & ~TOPK_DETERMINISTIC) != 0) return TOPK_ERR_ARG;
    if (batch < 0 || score_stride < 0 || (score_stride & 3) != 0) return TOPK_ERR_ARG;
    if (batch > 0 && (scores == nullptr || seq_lens == nullptr || out == nullptr)) return TOPK_ERR_ARG;
    if (batch > 0 && (reinterpret_cast<uintptr_t>(scores) & 15u) != 0) return TOPK_ERR_ALIGN;
    if (workspace == nullptr || workspace_bytes < workspace_bytes_for(batch)) return TOPK_ERR_WORKSPACE;
    return TOPK_OK;
}

Params make_params(const float* scores, int64_t score_stride, const int32_t* row_starts,
                   const int32_t* seq_lens, int32_t batch, int32_t k, void* workspace, int32_t* out,
                   int32_t* out_raw, uint32_t flags) {
    Params p = {};
    p.scores = scores;
    p.score_stride = score_stride;
    p.row_starts = row_starts;
    p.seq_lens = seq_lens;
    p.batch = batch;
    p.k = k;
    p.flags = flags;
    p.out = out;
    p.out_raw = out_raw;
    p.hdr = static_cast<PlanHeader*>(workspace);
    p.order = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(workspace) + sizeof(PlanHeader));
    p.cluster_rows = p.order + batch;
    return p;
}

}  // namespace

extern "C" {

size_t topk_workspace_bytes(int32_t batch) { return workspace_bytes_for(batch); }

int topk_plan(const int32_t* seq_lens, int32_t batch, int32_t k, void* workspace, size_t workspace_bytes,
              topk_stream_t stream) {
    if (!valid_k(k)) return TOPK_ERR_K;
    if (batch < 0 || (batch > 0 && seq_lens == nullptr)) return TOPK_ERR_ARG;
    if (workspace == nullptr || workspace_bytes < workspace_bytes_for(batch)) return TOPK_ERR_WORKSPACE;
    PlanHeader* hdr = static_cast<PlanHeader*>(workspace);
    int32_t* order = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + sizeof(PlanHeader));
    // one thread per row up to kPlanThreads (small batches get a small block)
    const int threads = min(kPlanThreads, max(64, (batch + 31) / 32 * 32));
    const cudaError_t e = launch_pdl(topk_plan_kernel, 1, threads, 0, reinterpret_cast<cudaStream_t>(stream),
                                     seq_lens, batch, k, hdr, order, order + batch);
    return e == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}

int topk_transform_paged_packed(const float* scores, int64_t score_stride, const int32_t* row_starts,
                                const int32_t* seq_lens, const int32_t* page_table, int64_t page_table_stride,
                                int32_t page_size, const int32_t* page_table_row_starts,
                                const int32_t* row_to_batch, int32_t batch, int32_t k, void* workspace,
                                size_t workspace_bytes, int32_t* out, int32_t* out_raw, uint32_t flags,
                                topk_stream_t stream) {
    const int st = common_checks(scores, score_stride, seq_lens, batch, k, workspace, workspace_bytes, out, flags);
    if (st != TOPK_OK) return st;
    if (page_size < 1 || page_size > TOPK_MAX_PAGE_SIZE || (page_size & (page_size - 1)) != 0)
        return TOPK_ERR_PAGE_SIZE;
    if (page_table_stride < 0 || (batch > 0 && page_table == nullptr)) return TOPK_ERR_ARG;
    if (batch == 0) return TOPK_OK;
    Params p = make_params(scores, score_stride, row_starts, seq_lens, batch, k, workspace, out, out_raw, flags);
    p.page_table = page_table;
    p.page_table_stride = page_table_stride;
    p.pt_row_starts = page_table_row_starts;
    p.row_to_batch = row_to_batch;
    int bits = 0;
    while ((1 << bits) < page_size) ++bits;
    p.page_bits = bits;
    return launch_transform<true>(p, reinterpret_cast<cudaStream_t>(stream));
}

int topk_transform_paged(const float* scores, int64_t score_stride, const int32_t* row_starts,
                         const int32_t* seq_lens, const int32_t* page_table, int64_t page_table_stride,
                         int32_t page_size, int32_t batch, int32_t k, void* workspace,
                         size_t workspace_bytes, int32_t* out, int32_t* out_raw, uint32_t flags,
                         topk_stream_t stream) {
    return topk_transform_paged_packed(scores, score_stride, row_starts, seq_lens, page_table, page_table_stride,
                                       page_size, nullptr, nullptr, batch, k, workspace, workspace_bytes, out,
                                       out_raw, flags, stream);
}

int topk_transform_ragged(const float* scores, int64_t score_stride, const int32_t* row_starts,
                          const int32_t* seq_lens, const int32_t* out_offsets, int32_t batch, int32_t k,
                          void* workspace, size_t workspace_bytes, int32_t* out, int32_t* out_raw,
                          uint32_t flags, topk_stream_t stream) {
    const int st = common_checks(scores, score_stride, seq_lens, batch, k, workspace, workspace_bytes, out, flags);
    if (st != TOPK_OK) return st;
    if (batch > 0 && out_offsets == nullptr) return TOPK_ERR_ARG;
    if (batch == 0) return TOPK_OK;
    Params p = make_params(scores, score_stride, row_starts, seq_lens, batch, k, workspace, out, out_raw, flags);
    p.out_offsets = out_offsets;
    return launch_transform<false>(p, reinterpret_cast<cudaStream_t>(stream));
}

int topk_read_device_errors(const void* workspace, int32_t* host_error_rows, uint32_t* host_flags,
                            topk_stream_t stream) {
    if (workspace == nullptr || host_error_rows == nullptr) return TOPK_ERR_ARG;
    PlanHeader h;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return TOPK_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return TOPK_ERR_CUDA;
    *host_error_rows = static_cast<int32_t>(h.error_rows);
    if (host_flags) *host_flags = h.flags;
    return TOPK_OK;
}

const char* topk_status_string(int status) {
    switch (status) {
        case TOPK_OK: return "ok";
        case TOPK_ERR_ARG: return "invalid argument";
        case TOPK_ERR_ALIGN: return "scores not 16-byte aligned";
        case TOPK_ERR_K: return "k outside [1, 2048]";
        case TOPK_ERR_PAGE_SIZE: return "page_size not a power of two in [1, 2^19]";
        case TOPK_ERR_WORKSPACE: return "workspace missing or too small";
        case TOPK_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Allocation-free entry point (plan + RAGGED transform on a built-in workspace)
// ----------------------------------------------------------------------------

namespace {

constexpr size_t kNoAllocWorkspaceBytes =
    (sizeof(PlanHeader) + 2 * sizeof(int32_t) * static_cast<size_t>(TOPK_NOALLOC_MAX_BATCH) + 255) / 256 * 256;

}  // namespace

// The plan workspace used by topk_transform_ragged_noalloc: one per GPU that
// loads the library, kept until the process exits. Host code must not pass
// this name to a kernel (on the host it is only a stand-in symbol); it uses the
// device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];

namespace {

struct NoAllocState {
    bool ready = false;
    void* ptr = nullptr;  // device address of g_noalloc_workspace on this device
};
NoAllocState g_noalloc[kMaxDevices];
std::mutex g_noalloc_mutex;

// Looks up the device address of the built-in workspace, once per device,
// with that device current.
cudaError_t noalloc_workspace(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocState& st = g_noalloc[dev];
    if (!st.ready) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_workspace);
        if (e != cudaSuccess || ptr == nullptr) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
        st.ptr = ptr;
        st.ready = true;
    }
    *out = st.ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" int topk_transform_ragged_noalloc(const float* scores, int64_t score_stride, const int32_t* row_starts,
                                             const int32_t* seq_lens, const int32_t* out_offsets, int32_t batch,
                                             int32_t k, int32_t* out, int32_t* out_raw, uint32_t flags,
                                             topk_stream_t stream) {
    if (batch > TOPK_NOALLOC_MAX_BATCH) return TOPK_ERR_WORKSPACE;
    // validate everything before anything is enqueued (a stand-in non-null
    // workspace pointer: the real one is looked up below)
    const int st =
        common_checks(scores, score_stride, seq_lens, batch, k, g_noalloc, kNoAllocWorkspaceBytes, out, flags);
    if (st != TOPK_OK) return st;
    if (batch > 0 && out_offsets == nullptr) return TOPK_ERR_ARG;
    if (batch == 0) return TOPK_OK;
    void* ws = nullptr;
    if (noalloc_workspace(&ws) != cudaSuccess) return TOPK_ERR_CUDA;
    // the plan rewrites the whole header and both row lists, so nothing left
    // by an earlier call is read
    const int ps = topk_plan(seq_lens, batch, k, ws, kNoAllocWorkspaceBytes, stream);
    if (ps != TOPK_OK) return ps;
    return topk_transform_ragged(scores, score_stride, row_starts, seq_lens, out_offsets, batch, k, ws,
                                 kNoAllocWorkspaceBytes, out, out_raw, flags, stream);
}
