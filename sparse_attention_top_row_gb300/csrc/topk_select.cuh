// Selection kernels of the indexer top-k + output transform for GB300
// (sm_103a), written once and compiled twice (topk_select512.cu,
// topk_select256.cu) for TOPK_THREADS threads per row inside namespace
// topk_impl::TOPK_NS; TOPK_WITH_CLUSTER adds the thread-block-cluster route.
// They select, for every row, the k <= 2048 largest fp32 scores of a window
// and write each selected position through the PAGED page-table map or the
// RAGGED offset (sglang PR #35175 page, "Implementation breakdown" and "Key
// source snippets"; "#26788 [JIT Kernel] DeepSeek-V4 DSA indexer: faster
// top-k + page-table transform (runtime k <= 2048)" page).
//
// Design (own design for sm_103a; the pages' CUDA/HIP kernels are prior art):
//
//  * Keys. A score's fp32 bits map to an order-preserving uint32 key. Every
//    selection step works on keys (or on raw bits compared as integers), so no
//    score is compared as a float.
//  * Fast path, every non-trivial row: bound, filter, finish.
//      bound   a sample of the row gives a lower bound on the k-th largest
//              key: the sample's expected share of the top k plus four
//              standard deviations plus 2, located in a histogram of the
//              sample. Register rows sample every fourth position from their
//              registers (two 256-bin levels); streamed and cluster rows take
//              a spread sample of 128 whole 64-byte blocks across the row
//              (2048 bins on the top 11 key bits, then 256 on the next 8);
//      filter  one pass over the window compares every element's raw bits
//              with the bound (one integer compare). Register rows and
//              cluster slices append (raw bits, position) to their warp's
//              region of a shared-memory candidate buffer (a warp scan of the
//              per-thread counts orders the slots); streamed rows append
//              (top 16 bits, 16-bit index) to per-thread compact lists. The
//              stores are predicated, nothing branches per element;
//      finish  the candidates are histogrammed on their 16-bit key prefix
//              relative to the bound (256 bins), one warp finds the bin where
//              the count from the top reaches k (a warp-shuffle suffix sum;
//              cf. warp_inclusive_sum on the PR #36684 page, "Key source
//              snippets"), every candidate above it takes an output slot (per
//              warp from the histograms, by ballot inside a warp; cf.
//              warp_sum_bool, same page), and the members of the threshold
//              bin are ranked by (key, position), which settles the remaining
//              key bits and the lowest-position tie-break at once. A
//              threshold past the first 255 prefixes over the bound re-bins
//              the top bin in narrowing windows (compact lists, cluster
//              rows and the 512-thread build's register rows).
//    The bound is only an estimate, so the fast path checks itself: when the
//    candidates number fewer than k, overflow their buffer, or crowd one bin
//    too densely to rank, the row finishes on the exact radix path below
//    (always exact, only slower).
//  * Exact radix path: a radix select on the 64-bit composite
//    (key << 32 | ~position), 12/8/8/4 bits of the key from the top (the
//    12-bit first digit of the PR #36684 page, "Feature and motivation"), then,
//    only when equal scores straddle the threshold and TOPK_DETERMINISTIC is
//    set, 8/8/8/8 bits of ~position, so the lowest positions win; a level ends
//    the descent as soon as its threshold bin holds exactly the count still
//    needed.
//  * Routes, chosen per row by length (the plan kernel orders rows longest
//    first and hands long rows of small batches to the cluster path):
//      trivial   L <= k: positions 0..L-1 then -1, scores never read;
//      register  L <= 16 * TOPK_THREADS (8192 on the 512-thread build, 4096
//                on the 256-thread one): the window lives in registers
//                (16-byte loads);
//      streaming longer rows: one register tile per thread, each tile's
//                successor loaded right after it is filtered and asked into
//                L2 by one bulk prefetch a step earlier;
//      cluster   few long rows: each row is cut into slices over a
//                thread-block cluster of 4 CTAs; each CTA stages its slice in
//                its own shared memory with 1-D bulk copies (cp.async.bulk,
//                completing on mbarriers) and filters it from there; the
//                candidate histograms are summed into every CTA of the
//                cluster with distributed-shared-memory reductions, and
//                output slots come from atomics on the leader CTA's shared
//                memory (cf. TopKCluster on the PR #36684 page).
//  * PAGED rows copy their page-table entries into shared memory with
//    cp.async while the scores load, so the emit's lookups stay on chip.
//  * Unaligned window heads: 16-byte loads start at the aligned address below
//    the window and the up-to-3 leading / trailing lanes are excluded by
//    position. Scores are never written (the pages' kernel masks them in place).
//  * Every kernel is launched with programmatic dependent launch and waits
//    (griddepcontrol.wait) before touching global memory, so it is scheduled
//    while the previous kernel on the stream drains without breaking stream
//    order. The only spin-waits are on the bulk copies' mbarriers, and each is
//    bounded: past its limit the kernel flags TOPK_DEVICE_FLAG_TIMEOUT and goes
//    on, so no wait can hang the GPU.

#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "topk_common.cuh"

#ifndef TOPK_THREADS
#error "TOPK_THREADS must be set"
#endif
#ifndef TOPK_WARP_CAP
#define TOPK_WARP_CAP 512  // candidate entries per warp region of a single-CTA row
#endif
#ifndef TOPK_PAGE_CACHE
#define TOPK_PAGE_CACHE 4096  // page-table entries of a single-CTA row held in shared memory
#endif
#ifndef TOPK_COMPACT_LISTS
#define TOPK_COMPACT_LISTS 1  // 1: streamed rows collect candidates in per-thread compact lists
#endif

namespace topk_impl {
namespace TOPK_NS {

namespace cg = cooperative_groups;

namespace {

constexpr int kThreads = TOPK_THREADS;        // threads of the team that processes one row (the CTA)
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 4096;                   // exact path: first radix level (12-bit digit)
constexpr int kSmall = 256;                   // fast path: sample levels, candidate histogram, later levels
constexpr int kSmallWords = kSmall + 4;       // + one word counting set bits below a level's digit
constexpr int kTileVecs = 4;                  // 16-byte vectors per thread per tile
constexpr int kTileElems = 4 * kTileVecs;
constexpr int kWarpCap = TOPK_WARP_CAP;       // candidate entries per warp region (single-CTA rows)
constexpr int kClusterWarpCap = 256;          // ... (a slice of a cluster row)
constexpr int kXHistWords = kBins + 8;        // exact path: level bins (+ the below count), 16-byte padded
constexpr int kCandBytes = kWarps * kWarpCap * 8;
constexpr int kXListCap = (kCandBytes - kXHistWords * 4) / 8;  // exact path: contiguous candidate list
constexpr int kClusterCandBytes = (kWarps * kClusterWarpCap * 8 > 2 * kXHistWords * 4)
                                      ? kWarps * kClusterWarpCap * 8 : 2 * kXHistWords * 4;
constexpr int kPageCache = TOPK_PAGE_CACHE;   // page-table entries of a row held in shared memory
constexpr int kClusterPageCache = 2048;       // ... of a slice (cluster kernel)
constexpr int kStageVecs = kTileVecs * kThreads;  // one staged chunk: 2048 vectors (32 KB)
constexpr int kStages = 4;                    // staged chunks in flight per CTA (128 KB)
constexpr int kMaxRankTies = kThreads;        // largest threshold bin the finish ranks directly
constexpr int kTieWords = 3 * (kMaxRankTies + 4);  // tie list: keys, positions, rank counters
constexpr long long kWaitCycles = 1ll << 31;  // bound on an mbarrier wait (about a second)



// Shared memory carve-up (dynamic), in this order:
//   stage   the cluster kernel's staged slice chunks (kStages x 32 KB)
//   cand    per-warp regions of (raw bits, position) on the fast path; the
//           exact path lays out in the same bytes its 4096-bin level
//           histogram (xhist; on a cluster also the merged one, xmhist) and a
//           contiguous (key, position) list (xlist)
//   pages   the row's (slice's) page-table entries
//   ties    the threshold bin's members (keys, positions, rank counters)
//   shist   the two 256-bin levels of the sample histogram
//   hist    the 256-bin candidate histogram, or a later radix level's bins
//   mhist   the cluster sum of the candidate histograms or of a later radix
//           level (cluster kernel)
//   whist   each warp's own 256-bin candidate histogram
//   mbar    one mbarrier per stage (cluster kernel)
//   scratch red (2 words per warp), res (16), cnt (16), wcnt (16)
// lvl / mlvl name the level histogram and its cluster sum that the radix
// levels use: hist / mhist, or xhist / xmhist on the exact path.
struct Shared {
    float4* stage;       // null in the rows kernel
    uint2* cand;
    int32_t* pages;
    uint8_t* tail;       // ties, shist, hist, mhist, mbar, scratch, at fixed offsets
    uint32_t* lvl;
    uint32_t* mlvl;
    __device__ __forceinline__ uint32_t* ties() const { return reinterpret_cast<uint32_t*>(tail); }
    __device__ __forceinline__ uint32_t* shist() const { return ties() + kTieWords; }
    __device__ __forceinline__ uint32_t* hist() const { return shist() + 2 * kSmallWords; }
    __device__ __forceinline__ uint32_t* mhist() const { return hist() + kSmallWords; }
    __device__ __forceinline__ uint32_t* whist() const { return mhist() + kSmallWords; }  // kWarps x kSmall
    __device__ __forceinline__ uint64_t* mbar() const {
        return reinterpret_cast<uint64_t*>(whist() + kWarps * kSmall);
    }
    __device__ __forceinline__ uint32_t* red() const { return reinterpret_cast<uint32_t*>(mbar() + kStages); }
    __device__ __forceinline__ uint32_t* res() const { return red() + 2 * kWarps; }
    // [0] exact-path list length, [1] definite slots, [2] tie-list length, [3] overflow flag
    __device__ __forceinline__ uint32_t* cnt() const { return red() + 2 * kWarps + 16; }
    __device__ __forceinline__ uint32_t* wcnt() const { return red() + 2 * kWarps + 32; }  // per-warp counts
    // the row's RowInfo, parked while the score pass needs the registers
    __device__ __forceinline__ int32_t* row() const { return reinterpret_cast<int32_t*>(red() + 2 * kWarps + 48); }
};

constexpr size_t kScratchWords = 2 * kWarps + 56;
constexpr size_t kTailBytes = (kTieWords + 4 * kSmallWords + kWarps * kSmall) * 4 + kStages * 8 + kScratchWords * 4;
constexpr size_t kSmemRows = static_cast<size_t>(kCandBytes) + kPageCache * 4 + kTailBytes;
constexpr size_t kSmemCluster = static_cast<size_t>(kStages) * kStageVecs * 16 + kClusterCandBytes +
                                kClusterPageCache * 4 + kTailBytes;
static_assert(kCandBytes % 16 == 0 && kClusterCandBytes % 16 == 0 && kTieWords % 4 == 0 && kSmallWords % 4 == 0,
              "16-byte aligned parts");

template <bool kCluster>
__device__ __forceinline__ Shared carve(uint8_t* base) {
    Shared s;
    uint8_t* p = base;
    if (kCluster) {
        s.stage = reinterpret_cast<float4*>(p);
        p += static_cast<size_t>(kStages) * kStageVecs * 16;
    } else {
        s.stage = nullptr;
    }
    s.cand = reinterpret_cast<uint2*>(p);
    p += kCluster ? kClusterCandBytes : kCandBytes;
    s.pages = reinterpret_cast<int32_t*>(p);
    p += static_cast<size_t>(kCluster ? kClusterPageCache : kPageCache) * 4;
    s.tail = p;
    s.lvl = s.hist();
    s.mlvl = kCluster ? s.mhist() : s.hist();
    return s;
}

// The exact path's view: 4096-bin levels in the candidate bytes (on a
// cluster also their sum, kXHistWords further on), the contiguous list after
// the first.
__device__ __forceinline__ Shared exact_view(const Shared& sh, bool cluster) {
    Shared x = sh;
    x.lvl = reinterpret_cast<uint32_t*>(sh.cand);
    x.mlvl = cluster ? x.lvl + kXHistWords : x.lvl;
    return x;
}
__device__ __forceinline__ uint2* exact_list(const Shared& sh) {
    return reinterpret_cast<uint2*>(reinterpret_cast<uint32_t*>(sh.cand) + kXHistWords);
}

// The dynamic shared memory of every kernel here. Every address in it is
// this symbol plus a constant of the kernel's layout, so a route rebuilds its
// Shared from the layout where it needs it instead of keeping pointers live.
extern __shared__ __align__(128) uint8_t g_smem[];

// Layouts: the rows kernel; the cluster kernel; the cluster kernel's view
// for a single-CTA row (rows-kernel buffers inside the idle stage area).
enum Layout { kLayRows = 0, kLayCluster = 1, kLayClusterSolo = 2 };

template <int kLay>
__device__ __forceinline__ Shared layout() {
    if (kLay == kLayRows) return carve<false>(g_smem);
    Shared s = carve<true>(g_smem);
    if (kLay == kLayClusterSolo) {
        static_assert(kCandBytes + kPageCache * 4 <= kStages * kStageVecs * 16, "solo buffers fit the stages");
        s.cand = reinterpret_cast<uint2*>(s.stage);
        s.pages = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(s.stage) + kCandBytes);
        s.lvl = s.hist();
        s.mlvl = s.hist();
    }
    return s;
}


// ----------------------------------------------------------------------------
// small device helpers
// ----------------------------------------------------------------------------

// Order-preserving fp32 bits -> uint32: flip all bits of negatives, set the
// sign bit of non-negatives.
__device__ __forceinline__ uint32_t bits_key(uint32_t b) {
    return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}

// 16 bytes of scores as raw integer bits (keys and key compares are integer
// work; the bits never pass through a float register).
__device__ __forceinline__ int4 load_stream_bits(const float4* p) {
    int4 r;
    asm("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}



__device__ __forceinline__ uint64_t composite(uint32_t key, int32_t pos) {
    return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~pos);
}

// Shared-memory access through 32-bit shared addresses (the hot loops name
// the state space explicitly instead of relying on generic addressing).
__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void red_add_shared(uint32_t a, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void st_shared_u32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
__device__ __forceinline__ uint2 ld_shared_v2(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
    return v;
}

// Radix levels over the 64-bit composite (key << 32 | ~position). Level i
// takes `bins` values of the digit at composite bit `shift`:
//   0..3  the key from scratch: 12, 8, 8, 4 bits;
//   4..5  the key's low 16 bits once its 16-bit prefix is known: 8, 8 bits;
//   6..9  ~position, 8 bits each (deterministic tie-break only).
constexpr int kLvlKey12 = 0, kLvlKeyLast = 3, kLvlLow16 = 4, kLvlLow16Last = 5, kLvlPos = 6, kLvlPosLast = 9;
__device__ __forceinline__ int level_shift(int lvl) {
    switch (lvl) {
        case 0: return 52;
        case 1: return 44;
        case 2: return 36;
        case 3: return 32;
        case 4: return 40;
        case 5: return 32;
        default: return 8 * (9 - lvl);
    }
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
// sh.res(). One barrier (after it every bin has been read); the caller reads
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
    if (lane == 0) sh.red()[warp] = x;
    __syncthreads();
    uint32_t above = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t r = sh.red()[w];
        total += r;
        above += w > warp ? r : 0u;
    }
    const uint32_t incl = above + x, excl = incl - s8;
    if (excl < target && incl >= target) {
        uint32_t r = excl;
#pragma unroll
        for (int i = R - 1; i >= 0; --i) {
            if (r + b[i] >= target) {
                sh.res()[0] = R * threadIdx.x + static_cast<uint32_t>(i);
                sh.res()[1] = r;
                sh.res()[2] = b[i];
                break;
            }
            r += b[i];
        }
    }
    return total;
}

__device__ __forceinline__ Threshold find_wide_result(uint32_t total, uint32_t target, const Shared& sh) {
    if (total < target) return Threshold{0u, total, 0u, false};
    return Threshold{sh.res()[0], sh.res()[1], sh.res()[2], true};
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
                            sh.res()[0] = static_cast<uint32_t>(lo + i);
                            sh.res()[1] = r;
                            sh.res()[2] = b[i];
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
                sh.res()[0] = 0;
                sh.res()[1] = run;
                sh.res()[2] = 0;
            }
            sh.res()[3] = found ? 1u : 0u;
        }
    }
    __syncthreads();
    return Threshold{sh.res()[0], sh.res()[1], sh.res()[2], sh.res()[3] != 0};
}

__device__ __forceinline__ void clear_words(uint32_t* h, int n) {
    for (int i = threadIdx.x; i < n / 4; i += kThreads) reinterpret_cast<uint4*>(h)[i] = make_uint4(0, 0, 0, 0);
}

// Sum over the CTA of h[c] for c >= from (bins of the local histogram).
__device__ uint32_t count_from(const uint32_t* h, int nb, uint32_t from, const Shared& sh) {
    uint32_t s = 0;
    for (int c = threadIdx.x; c < nb; c += kThreads)
        if (static_cast<uint32_t>(c) >= from) s += h[c];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(kFull, s, off);
    __syncthreads();
    if (lane_id() == 0) sh.red()[threadIdx.x >> 5] = s;
    __syncthreads();
    uint32_t t = 0;
    for (int w = 0; w < kWarps; ++w) t += sh.red()[w];
    __syncthreads();
    return t;
}

// ----------------------------------------------------------------------------
// merge policies of the exact radix path: a single CTA, or a thread-block
// cluster over distributed shared memory
// ----------------------------------------------------------------------------

struct SoloMerge {
    static constexpr bool kSolo = true;
    __device__ __forceinline__ const uint32_t* merge(const Shared& sh, int) const {
        __syncthreads();
        return sh.lvl;
    }
    __device__ __forceinline__ uint32_t* counter(const Shared& sh, int i) const { return &sh.cnt()[i]; }
};

struct ClusterMerge {
    static constexpr bool kSolo = false;
    // lvl (local) -> mlvl (sum over the cluster), identical in every CTA.
    // CTA r sums the 16-byte words w = r, r + kClusterSize, ... over all CTAs
    // (reduce-scatter); then every CTA gathers the words it does not own.
    __device__ const uint32_t* merge(const Shared& sh, int nb) const {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();  // every local histogram is complete
        const int rank = static_cast<int>(cluster.block_rank());
        const int words = nb / 4;
        for (int w = rank + kClusterSize * static_cast<int>(threadIdx.x); w < words; w += kClusterSize * kThreads) {
            uint4 t = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int q = 0; q < kClusterSize; ++q) {
                const uint4 r = reinterpret_cast<const uint4*>(cluster.map_shared_rank(sh.lvl, q))[w];
                t.x += r.x, t.y += r.y, t.z += r.z, t.w += r.w;
            }
            reinterpret_cast<uint4*>(sh.mlvl)[w] = t;
        }
        cluster.sync();  // every owned word of the sum is complete
        for (int w = static_cast<int>(threadIdx.x); w < words; w += kThreads) {
            const int q = w % kClusterSize;
            if (q != rank)
                reinterpret_cast<uint4*>(sh.mlvl)[w] =
                    reinterpret_cast<const uint4*>(cluster.map_shared_rank(sh.mlvl, q))[w];
        }
        __syncthreads();
        return sh.mlvl;
    }
    __device__ __forceinline__ uint32_t* counter(const Shared& sh, int i) const {
        return cg::this_cluster().map_shared_rank(&sh.cnt()[i], 0);
    }
};

// ----------------------------------------------------------------------------
// element sources of the exact path: registers, a candidate list, the
// per-warp candidate regions, shared memory, global memory. visit(f) calls
// f(key, position, valid) with a fixed thread-to-element assignment.
// ----------------------------------------------------------------------------

// Register tile: v[u] holds vector j = u*kThreads + tid of the aligned window.
struct RegSource {
    const int4 (&v)[kTileVecs];
    int rem, len;
    template <class F>
    __device__ __forceinline__ void visit(F&& f) const {
#pragma unroll
        for (int u = 0; u < kTileVecs; ++u) {
            const int p0 = 4 * (u * kThreads + static_cast<int>(threadIdx.x)) - rem;
            const int e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int p = p0 + c;
                f(bits_key(static_cast<uint32_t>(e[c])), p, static_cast<unsigned>(p) < static_cast<unsigned>(len));
            }
        }
    }
};

// A contiguous list of n (key, position) entries.
struct CandSource {
    const uint2* c;
    uint32_t n;
    template <class F>
    __device__ __forceinline__ void visit(F&& f) const {
        const uint32_t n_round = (n + kThreads - 1) / kThreads * kThreads;
        for (uint32_t i = threadIdx.x; i < n_round; i += kThreads) {
            const bool valid = i < n;
            const uint2 e = valid ? c[i] : make_uint2(0u, 0u);
            f(e.x, static_cast<int32_t>(e.y), valid);
        }
    }
};

// The per-warp candidate regions of the fast path, (raw bits, position):
// each warp visits its own region.
struct RegionSource {
    const uint2* c;  // region 0; region w at c + w * cap
    const uint32_t* wcnt;
    int cap;
    template <class F>
    __device__ __forceinline__ void visit(F&& f) const {
        const int warp = static_cast<int>(threadIdx.x >> 5);
        const uint2* r = c + warp * cap;
        const uint32_t n = min(wcnt[warp], static_cast<uint32_t>(cap));
        const uint32_t n_round = (n + 31u) & ~31u;
        for (uint32_t i = lane_id(); i < n_round; i += 32) {
            const bool valid = i < n;
            const uint2 e = valid ? r[i] : make_uint2(0u, 0u);
            f(bits_key(e.x), static_cast<int32_t>(e.y), valid);
        }
    }
};

// Vectors [jb, je) of the aligned window from a base (global or shared).
template <bool kGlobal>
struct VecSource {
    const float4* vbase;
    int jb, je, rem, len;
    template <class F>
    __device__ __forceinline__ void visit(F&& f) const {
        for (int j0 = jb; j0 < je; j0 += kTileVecs * kThreads) {
            int4 v[kTileVecs];
#pragma unroll
            for (int u = 0; u < kTileVecs; ++u) {
                const int j = j0 + u * kThreads + static_cast<int>(threadIdx.x);
                v[u] = j >= je ? make_int4(0, 0, 0, 0)
                       : kGlobal ? load_stream_bits(vbase + j)
                                 : reinterpret_cast<const int4*>(vbase)[j];
            }
#pragma unroll
            for (int u = 0; u < kTileVecs; ++u) {
                const int j = j0 + u * kThreads + static_cast<int>(threadIdx.x);
                const int p0 = 4 * j - rem;
                const int e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int p = p0 + c;
                    f(bits_key(static_cast<uint32_t>(e[c])), p,
                      j < je && static_cast<unsigned>(p) < static_cast<unsigned>(len));
                }
            }
        }
    }
};
using GlobalSource = VecSource<true>;

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

// Key levels first..last_key, then (det) the position levels, stopping once
// exact. A key level also counts, in the word after its bins, the elements
// of the current group with any key bit below its digit set; when the merged
// count is 0 every such bit is 0 throughout the group (scores rounded to bf16
// or coarser), so the key is settled and the remaining key levels are skipped.
template <class Merge, class Src>
__device__ void run_levels(SelState& st, int first, int last_key, bool det, const Src& src, const Shared& sh,
                           const Merge& mg) {
    int lvl = first;
    while (!st.exact) {
        if (lvl > last_key && lvl < kLvlPos) lvl = kLvlPos;
        if (lvl > kLvlPosLast || (lvl >= kLvlPos && !det)) break;
        const int nb = level_bins(lvl);
        const int shift = level_shift(lvl);
        uint32_t* hist = sh.lvl;
        const uint32_t digit = static_cast<uint32_t>(nb - 1);
        const bool key_level = lvl < kLvlPos;
        const int words = key_level ? nb + 4 : nb;
        clear_words(sh.lvl, words);
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
        if (settled) {
            st.mask |= static_cast<uint64_t>(below) << 32;  // those bits are 0 in the prefix too
            lvl = kLvlPos;
        } else {
            ++lvl;
        }
    }
}

// Output transform of one selected position.
template <bool kPaged>
struct Emitter {
    int32_t* out;
    int32_t* out_raw;
    const int32_t* pt_row;     // the row's page-table row (packed rows: its request's)
    const int32_t* pt_cached;  // page-table entries from pt_first on, in shared memory, or null
    int32_t token0;            // page-table token of position 0 (0 unless packed)
    int32_t pt_first;          // first page-table entry held in pt_cached
    int32_t pt_count;          // entries held in pt_cached
    int32_t page_bits;
    int32_t offset;
    uint32_t k;
    uint32_t* flags;  // device flags word of the workspace
    uint32_t* stats;  // the workspace's count of rows finished on the exact path
    __device__ __forceinline__ int32_t value(int32_t pos) const {
        if (!kPaged) return pos + offset;
        const int32_t t = pos + token0;
        const int32_t q = t >> page_bits;
        const uint32_t c = static_cast<uint32_t>(q - pt_first);
        const int32_t page = (pt_cached && c < static_cast<uint32_t>(pt_count)) ? pt_cached[c] : __ldg(pt_row + q);
        return (page << page_bits) | (t & ((1 << page_bits) - 1));
    }
    __device__ __forceinline__ void write(uint32_t slot, int32_t pos) const {
        if (slot >= k) {  // never taken when the selection is consistent
            atomicOr(flags, TOPK_DEVICE_FLAG_INTERNAL);
            return;
        }
        out[slot] = value(pos);
        if (out_raw) out_raw[slot] = pos;
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
    const uint32_t need = st.need;
    const bool exact = st.exact;
    const bool key_only = static_cast<uint32_t>(st.mask) == 0;  // only key levels ran
    const uint32_t pfx = static_cast<uint32_t>(st.prefix >> 32);
    const uint64_t prefix = st.prefix, mask = st.mask;
    // with a top-aligned mask, "masked key above the prefix" is a plain
    // compare against the prefix (exact) or tau
    auto classify = [&](uint32_t key, int32_t pos, bool valid, bool& def, bool& grp) {
        if (key_only) {
            const uint32_t hk = key & static_cast<uint32_t>(mask >> 32);
            def = valid && (exact ? hk >= pfx : hk > pfx);
            grp = valid && !exact && hk == pfx;
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
        sh.red()[warp] = xd;
        sh.red()[kWarps + warp] = xg;
    }
    __syncthreads();
    uint32_t bd = xd - nd, bg = xg - ng, td = 0, tg = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t rd = sh.red()[w], rg = sh.red()[kWarps + w];
        bd += w < warp ? rd : 0u;
        bg += w < warp ? rg : 0u;
        td += rd;
        tg += rg;
    }
    if (!Merge::kSolo) {  // this CTA's share of the cluster-wide slot ranges
        __syncthreads();
        if (threadIdx.x == 0) {
            sh.red()[0] = td ? atomicAdd(mg.counter(sh, 1), td) : 0u;
            sh.red()[1] = tg ? atomicAdd(mg.counter(sh, 2), tg) : 0u;
        }
        __syncthreads();
        bd += sh.red()[0];
        bg += sh.red()[1];
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

template <bool kPaged>
__device__ void trivial_row(int32_t len, uint32_t k, const Emitter<kPaged>& em, bool pad_out = true) {
    for (uint32_t t = threadIdx.x; t < k; t += kThreads) {
        if (static_cast<int32_t>(t) < len) {
            em.write(t, static_cast<int32_t>(t));
        } else {
            if (pad_out) em.out[t] = -1;  // (the SWA combine's tail fills these slots instead)
            if (em.out_raw) em.out_raw[t] = -1;
        }
    }
}

// The SWA combine's tail of row b (p.positions set): slots [topk_len, width)
// of the output row, topk_len = min(k, len) the row's selected entries, hold
// the window's tokens pos - w + 1 .. pos plus the row's SWA offset, w =
// min(window, pos + 1) (none for pos < 0), then -1 (the PR #30255 page's
// combine_topk_swa_indices, topk_len = min((pos + 1) // COMPRESS_RATIO,
// top_k), in the reading of the library's header). All threads of the CTA.
__device__ __forceinline__ void swa_tail(const Params& p, int b, int32_t len) {
    const int32_t topk_len = min(max(len, 0), p.k);
    const int32_t pos = p.positions[b];
    const int32_t w = pos < 0 ? 0 : min(p.swa_window, pos + 1);
    const int32_t first = pos - w + 1 + (p.swa_offsets ? p.swa_offsets[b] : 0);
    int32_t* row = p.out + static_cast<int64_t>(b) * p.out_stride + topk_len;
    for (int32_t i = static_cast<int32_t>(threadIdx.x); i < p.out_stride - topk_len; i += kThreads)
        row[i] = i < w ? first + i : -1;
}

// Ranks the threshold bin's members, n <= kThreads of them in tkey/tpos
// (16-byte aligned, room for n rounded up to 4): the rank of an element is
// the number of members whose composite (key, ~position) is larger, and the
// ones ranked below `need` take slots k - need + rank: put(slot, pos) stores
// each one. This settles every remaining key and position digit at once
// (ties go to the lowest position). Up to 32 members are ranked by one warp
// through shuffles. Longer lists are padded to a multiple of 4 with entries
// that rank below everything; each element is compared by kThreads / m
// threads (m = n rounded up to a power of two), each over one segment, and the
// partial ranks meet in the shared-memory counters `rank` (n words). A
// caller's barrier must make the lists visible first; the function ends
// without one.
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

// The tie list of the threshold bin (a CTA's `ties` area).
struct TieList {
    uint32_t* key;
    int32_t* pos;
    uint32_t* rank;
};
__device__ __forceinline__ TieList tie_list(uint32_t* ties) {
    constexpr int kPad = kMaxRankTies + 4;
    return TieList{ties, reinterpret_cast<int32_t*>(ties + kPad), ties + 2 * kPad};
}

// ----------------------------------------------------------------------------
// fast path: register tiles, the filter, the sample bound
// ----------------------------------------------------------------------------

// Raw bits of one tile: kTileVecs vectors per thread from vector j0 (vectors
// at or past je read as zero bits and are never in the window).
__device__ __forceinline__ void load_bits(int4 (&v)[kTileVecs], const float4* vbase, int j0, int je) {
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
        const int j = j0 + u * kThreads + static_cast<int>(threadIdx.x);
        v[u] = j < je ? load_stream_bits(vbase + j) : make_int4(0, 0, 0, 0);
    }
}

// The same from a shared-memory chunk: vectors [0, n) of `chunk`.
__device__ __forceinline__ void load_bits_smem(int4 (&v)[kTileVecs], const float4* chunk, int n) {
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
        const int j = u * kThreads + static_cast<int>(threadIdx.x);
        v[u] = j < n ? reinterpret_cast<const int4*>(chunk)[j] : make_int4(0, 0, 0, 0);
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

// Whether every element of the tile at vector j0 lies in the window.
__device__ __forceinline__ bool tile_interior(int j0, int je, int rem, int len) {
    constexpr int T = kTileVecs * kThreads;
    return 4 * j0 - rem >= 0 && 4 * (j0 + T) - rem <= len && j0 + T <= je;
}

// key >= bound_key as one compare of the raw bits: for a non-negative bound
// (bound_key >= 2^31) key >= bound_key <=> bits >= bound_key ^ 2^31 as signed
// integers; below it, key >= bound_key <=> bits <= ~bound_key as unsigned
// ones. thr is that right-hand side.
template <bool kNonNeg>
__device__ __forceinline__ bool passes(int32_t b, uint32_t thr) {
    return kNonNeg ? b >= static_cast<int32_t>(thr) : static_cast<uint32_t>(b) <= thr;
}
__device__ __forceinline__ uint32_t pass_threshold(uint32_t bound_key) {
    return bound_key >= 0x80000000u ? (bound_key ^ 0x80000000u) : ~bound_key;
}

// Stores (bits, p0 + kOff) at shared address a and advances a by one entry
// when bits pass the bound (thr: see passes); with kMasked only when bit kBit
// of `valid` is set too. One compare, one predicated store, one predicated
// add; the position is formed inside, so no position is kept in a register.
template <bool kNonNeg, bool kMasked, int kOff, int kBit>
__device__ __forceinline__ void append_if(uint32_t& a, int32_t bits, uint32_t thr, int32_t p0, uint32_t valid) {
    if (kMasked) {
        if (kNonNeg)
            asm volatile(
                "{\n\t.reg .pred v, q;\n\t.reg .b32 t;\n\tand.b32 t, %4, %6;\n\tsetp.ne.b32 v, t, 0;\n\t"
                "setp.ge.and.s32 q, %1, %2, v;\n\tadd.s32 t, %3, %5;\n\t"
                "@q st.shared.v2.b32 [%0], {%1, t};\n\t@q add.u32 %0, %0, 8;\n\t}"
                : "+r"(a)
                : "r"(bits), "r"(thr), "r"(p0), "r"(valid), "n"(kOff), "n"(1 << kBit)
                : "memory");
        else
            asm volatile(
                "{\n\t.reg .pred v, q;\n\t.reg .b32 t;\n\tand.b32 t, %4, %6;\n\tsetp.ne.b32 v, t, 0;\n\t"
                "setp.le.and.u32 q, %1, %2, v;\n\tadd.s32 t, %3, %5;\n\t"
                "@q st.shared.v2.b32 [%0], {%1, t};\n\t@q add.u32 %0, %0, 8;\n\t}"
                : "+r"(a)
                : "r"(bits), "r"(thr), "r"(p0), "r"(valid), "n"(kOff), "n"(1 << kBit)
                : "memory");
    } else {
        if (kNonNeg)
            asm volatile(
                "{\n\t.reg .pred q;\n\t.reg .b32 t;\n\tsetp.ge.s32 q, %1, %2;\n\tadd.s32 t, %3, %4;\n\t"
                "@q st.shared.v2.b32 [%0], {%1, t};\n\t@q add.u32 %0, %0, 8;\n\t}"
                : "+r"(a)
                : "r"(bits), "r"(thr), "r"(p0), "n"(kOff)
                : "memory");
        else
            asm volatile(
                "{\n\t.reg .pred q;\n\t.reg .b32 t;\n\tsetp.le.u32 q, %1, %2;\n\tadd.s32 t, %3, %4;\n\t"
                "@q st.shared.v2.b32 [%0], {%1, t};\n\t@q add.u32 %0, %0, 8;\n\t}"
                : "+r"(a)
                : "r"(bits), "r"(thr), "r"(p0), "n"(kOff)
                : "memory");
    }
}

// Adds 1 to c when bits pass the bound (and, with kMasked, bit kBit of valid
// is set).
template <bool kNonNeg, bool kMasked, int kBit>
__device__ __forceinline__ void count_if(uint32_t& c, int32_t bits, uint32_t thr, uint32_t valid) {
    if (kMasked) {
        if (kNonNeg)
            asm("{\n\t.reg .pred v, q;\n\t.reg .b32 t;\n\tand.b32 t, %2, %4;\n\tsetp.ne.b32 v, t, 0;\n\t"
                "setp.ge.and.s32 q, %1, %3, v;\n\t@q add.u32 %0, %0, 1;\n\t}"
                : "+r"(c) : "r"(bits), "r"(valid), "r"(thr), "n"(1 << kBit));
        else
            asm("{\n\t.reg .pred v, q;\n\t.reg .b32 t;\n\tand.b32 t, %2, %4;\n\tsetp.ne.b32 v, t, 0;\n\t"
                "setp.le.and.u32 q, %1, %3, v;\n\t@q add.u32 %0, %0, 1;\n\t}"
                : "+r"(c) : "r"(bits), "r"(valid), "r"(thr), "n"(1 << kBit));
    } else {
        if (kNonNeg)
            asm("{\n\t.reg .pred q;\n\tsetp.ge.s32 q, %1, %2;\n\t@q add.u32 %0, %0, 1;\n\t}"
                : "+r"(c) : "r"(bits), "r"(thr));
        else
            asm("{\n\t.reg .pred q;\n\tsetp.le.u32 q, %1, %2;\n\t@q add.u32 %0, %0, 1;\n\t}"
                : "+r"(c) : "r"(bits), "r"(thr));
    }
}

// Compile-time loop over the tile's elements: f(integral_constant<e>).
template <int E, class F>
__device__ __forceinline__ void for_each_elem(F&& f) {
    if constexpr (E < kTileElems) {
        f(std::integral_constant<int, E>{});
        for_each_elem<E + 1>(f);
    }
}

// The filter: appends the tile's in-window elements whose key is at least
// the bound to this warp's candidate region (shared address `region`) as
// (raw bits, position). Straight-line code: every element is compared, one
// warp scan of the per-thread counts gives each thread its first slot, the
// stores are predicated (no branch per element, no shared atomic). `wcount`
// is the warp's running count (warp-uniform); a region that would overflow
// takes no more entries and sets `ovf` (the row then finishes on the exact
// path). Element e of the tile sits at position p0 + (e / 4) * 4 * kThreads
// + e % 4.
template <bool kNonNeg, bool kMasked>
__device__ __forceinline__ void filter_tile(const int4 (&v)[kTileVecs], uint32_t thr, uint32_t valid, int p0,
                                            uint32_t region, uint32_t& wcount, uint32_t cap, bool& ovf) {
    uint32_t c = 0;
    for_each_elem<0>([&](auto ec) {
        constexpr int e = decltype(ec)::value;
        count_if<kNonNeg, kMasked, e>(c, tile_elem(v, e), thr, valid);
    });
    const uint32_t incl = warp_inclusive_scan(c);
    const uint32_t total = __shfl_sync(kFull, incl, 31);
    uint32_t a = region + (wcount + incl - c) * 8u;
    wcount += total;
    if (wcount > cap) {  // warp-uniform
        ovf = true;
        return;
    }
    for_each_elem<0>([&](auto ec) {
        constexpr int e = decltype(ec)::value;
        append_if<kNonNeg, kMasked, (e >> 2) * (4 * kThreads) + (e & 3), e>(a, tile_elem(v, e), thr, p0, valid);
    });
}

// filter_tile for the tile at vector j0 of a window of vectors [.., je).
template <bool kNonNeg>
__device__ __forceinline__ void filter_at(const int4 (&v)[kTileVecs], uint32_t thr, int j0, int je, int rem, int len,
                                          uint32_t region, uint32_t& wcount, uint32_t cap, bool& ovf) {
    const int p0 = 4 * (j0 + static_cast<int>(threadIdx.x)) - rem;
    if (tile_interior(j0, je, rem, len))
        filter_tile<kNonNeg, false>(v, thr, 0xFFFFu, p0, region, wcount, cap, ovf);
    else
        filter_tile<kNonNeg, true>(v, thr, tile_valid(j0, je, rem, len), p0, region, wcount, cap, ovf);
}

// Lower bound on the threshold from a sample of n_s of the window's len keys
// (this thread's in skey[j] where bit j of vmask is set): the 16-bit key
// prefix at which the count from the top first reaches the sample's expected
// share of the top-k plus four standard deviations plus 2, found by two
// 256-bin levels (the top 8 key bits, then the next 8) in the two halves of
// shist (zero on entry; every thread calls this). Returns the prefix's lowest
// key. Four barriers; warp 0 searches.
template <int N>
__device__ uint32_t sample_bound(const uint32_t (&skey)[N], uint32_t vmask, uint32_t n_s, int len, uint32_t k,
                                 const Shared& sh) {
    const float expect = static_cast<float>(k) * static_cast<float>(n_s) / static_cast<float>(len);
    const float tgt = fminf(ceilf(expect + 4.0f * sqrtf(expect) + 2.0f), static_cast<float>(n_s));
    const uint32_t target = max(static_cast<uint32_t>(tgt), 1u);
    const uint32_t h1 = saddr(sh.shist()), h2 = saddr(sh.shist() + kSmallWords);
#pragma unroll
    for (int j = 0; j < N; ++j)
        if ((vmask >> j) & 1u) red_add_shared(h1 + (skey[j] >> 24) * 4u, 1u);
    __syncthreads();
    const Threshold t1 = find_threshold(sh.shist(), kSmall, target, sh);
#pragma unroll
    for (int j = 0; j < N; ++j)
        if (((vmask >> j) & 1u) && (skey[j] >> 24) == t1.bin) red_add_shared(h2 + ((skey[j] >> 16) & 255u) * 4u, 1u);
    __syncthreads();
    const Threshold t2 = find_threshold(sh.shist() + kSmallWords, kSmall, target - t1.above, sh);
    return ((t1.bin << 8) | t2.bin) << 16;
}

// The spread sample of a streamed window: 128 pieces of 4 consecutive
// 16-byte vectors, each a whole 64-byte-aligned block of memory. With v0 the
// first vector of the aligned span on such a boundary and nq the whole blocks
// from there inside the span, piece i is the block v0 + 4 * floor(i * nq /
// 128), so the pieces cover the whole row; 4 consecutive threads load a piece,
// one vector each (kSpreadLoads vectors per thread). 2048 elements in all,
// less the few lanes outside the window. (Twice the sample gives a bound
// nearer the threshold, 25 instead of 36 % above k on the extend rows, but
// costs more than the smaller finish saves.)
#ifndef TOPK_SPREAD_LOG_PIECES
#define TOPK_SPREAD_LOG_PIECES 7
#endif
constexpr int kSpreadLogPieces = TOPK_SPREAD_LOG_PIECES;
constexpr int kSpreadPieces = 1 << kSpreadLogPieces;
constexpr int kSpreadLoads = kSpreadPieces * 4 / kThreads;
static_assert(kSpreadLoads * kThreads == 4 * kSpreadPieces && 4 * kSpreadLoads <= 32, "spread sample shape");
constexpr int kSpreadBins1 = 2048;  // level 1: key bits 31..21
constexpr int kSpreadBins2 = 256;   // level 2: key bits 20..13 inside the level-1 bin
static_assert(kWarps * kSmall >= kSpreadBins1, "level 1 fits the per-warp histograms");

struct SpreadSample {
    int4 v[kSpreadLoads];
    uint32_t valid;  // bit 4u + c: lane c of vector u lies in the window
};

__device__ __forceinline__ int spread_v0(const float4* vbase) {
    return static_cast<int>((4u - ((static_cast<uint32_t>(reinterpret_cast<uintptr_t>(vbase)) >> 4) & 3u)) & 3u);
}
__device__ __forceinline__ int spread_vec(int u, int v0, uint64_t nq) {
    const uint64_t piece = static_cast<uint64_t>(u * (kThreads / 4) + static_cast<int>(threadIdx.x >> 2));
    return v0 + 4 * static_cast<int>((piece * nq) >> kSpreadLogPieces) + static_cast<int>(threadIdx.x & 3u);
}

// Loads this thread's share of the spread sample (nv > 1024).
__device__ __forceinline__ SpreadSample spread_load(const float4* vbase, int nv, int rem, int len) {
    SpreadSample s;
    const int v0 = spread_v0(vbase);
    const uint64_t nq = static_cast<uint32_t>(nv - v0) >> 2;  // >= 255
    s.valid = 0xFFFFFFFFu >> (32 - 4 * kSpreadLoads);
#pragma unroll
    for (int u = 0; u < kSpreadLoads; ++u) {
        const int j = spread_vec(u, v0, nq);  // < v0 + 4 * nq <= nv
        s.v[u] = load_stream_bits(vbase + j);
        const int p0 = 4 * j - rem;
        if (p0 < 0 || p0 + 4 > len) {  // only vector 0 and vector nv - 1 have lanes outside the window
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (p0 + c < 0 || p0 + c >= len) s.valid &= ~(1u << (4 * u + c));
        }
    }
    return s;
}

// The elements of the spread sample: every sampled lane but the `rem`
// before the window (vector 0 is sampled exactly when v0 = 0) and those after
// it (in vector nv - 1, when sampled).
__device__ __forceinline__ uint32_t spread_count(const float4* vbase, int nv, int rem, int len) {
    const int v0 = spread_v0(vbase);
    const uint64_t nq = static_cast<uint32_t>(nv - v0) >> 2;
    const int last = v0 + 4 * static_cast<int>((static_cast<uint64_t>(kSpreadPieces - 1) * nq) >> kSpreadLogPieces) + 3;
    return static_cast<uint32_t>(16 * kSpreadPieces - (v0 == 0 ? rem : 0) - (last == nv - 1 ? 4 * nv - rem - len : 0));
}

// The threshold bound from the spread sample (every thread calls): the
// sample's expected share of the top k plus four standard deviations plus 2,
// located in a 2048-bin histogram of the top 11 key bits (sh.whist()) and
// then a 256-bin one of the next 8 (sh.hist()); both zero on entry and on
// return. Returns a key whose 13 low bits are zero. arrived() runs once this
// thread's sample is in (so that traffic it starts queues behind the sample).
template <class Arrived>
__device__ uint32_t spread_bound(const SpreadSample& s, uint32_t n_s, int len, uint32_t k, const Shared& sh,
                                 Arrived&& arrived) {
    uint32_t* h1 = sh.whist();
    uint32_t* h2 = sh.hist();
#pragma unroll
    for (int u = 0; u < kSpreadLoads; ++u) {
        const int32_t e[4] = {s.v[u].x, s.v[u].y, s.v[u].z, s.v[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if ((s.valid >> (4 * u + c)) & 1u) atomicAdd(&h1[bits_key(static_cast<uint32_t>(e[c])) >> 21], 1u);
    }
    arrived();
    const float expect = static_cast<float>(k) * static_cast<float>(n_s) / static_cast<float>(len);
    const float tgt = fminf(ceilf(expect + 4.0f * sqrtf(expect) + 2.0f), static_cast<float>(n_s));
    const uint32_t target = max(static_cast<uint32_t>(tgt), 1u);
    __syncthreads();
    const Threshold t1 = find_threshold(h1, kSpreadBins1, target, sh);
#pragma unroll
    for (int u = 0; u < kSpreadLoads; ++u) {
        const int32_t e[4] = {s.v[u].x, s.v[u].y, s.v[u].z, s.v[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint32_t key = bits_key(static_cast<uint32_t>(e[c]));
            if (((s.valid >> (4 * u + c)) & 1u) && (key >> 21) == t1.bin) atomicAdd(&h2[(key >> 13) & 255u], 1u);
        }
    }
    __syncthreads();
    const Threshold t2 = find_threshold(h2, kSpreadBins2, target - t1.above, sh);
    clear_words(h1, kSpreadBins1);  // (the searches' last barrier is behind every read of the bins)
    clear_words(h2, kSpreadBins2);
    __syncthreads();
    return t1.found && t2.found ? (t1.bin << 21) | (t2.bin << 13) : 0u;
}

// ----------------------------------------------------------------------------
// fast path: the finish over the candidates
// ----------------------------------------------------------------------------

// Bin of a candidate key in the 256-bin histogram of 16-bit key prefixes
// based at base16 (the bound's prefix); keys 255 or more prefixes above share
// the top bin.
__device__ __forceinline__ uint32_t fine_bin(uint32_t key, uint32_t base16) {
    return min((key >> 16) - base16, static_cast<uint32_t>(kSmall - 1));
}

// A window of 16-bit key prefixes over the candidates, once the threshold
// lies past the first one (see rebin_regions): bin 0 below lo, bin 1 + i the
// prefixes lo + (i << shift) .., bin 255 the rest above.
struct PrefixWindow {
    uint32_t lo, shift;
    __device__ __forceinline__ uint32_t operator()(uint32_t key) const {
        const uint32_t p = key >> 16;
        return p < lo ? 0u : 1u + min((p - lo) >> shift, static_cast<uint32_t>(kSmall - 2));
    }
};

// The first window: the 256 prefixes from the bound's (fine_bin).
struct BoundWindow {
    uint32_t base16;
    __device__ __forceinline__ uint32_t operator()(uint32_t key) const { return fine_bin(key, base16); }
};

// Counts this warp's n candidates (region at shared address `region`) into
// its own histogram at shared address `whist`, binned by `bin_of`.
template <class BinOf>
__device__ __forceinline__ void count_candidates(uint32_t region, uint32_t n, BinOf bin_of, uint32_t whist) {
    for (uint32_t i = lane_id(); i < n; i += 32)
        red_add_shared(whist + bin_of(bits_key(ld_shared_u32(region + i * 8u))) * 4u, 1u);
}

// Thread t < kSmall: bin t summed over the warps' histograms (after a barrier
// that completes them).
__device__ __forceinline__ uint32_t sum_warp_bins(const Shared& sh) {
    uint32_t c = 0;
    const uint32_t* w = sh.whist() + threadIdx.x;
#pragma unroll
    for (int q = 0; q < kWarps; ++q) c += w[q * kSmall];
    return c;
}

// This warp's count of definite candidates (bins above tau, and tau itself
// when exact) and of threshold-bin members, from its own histogram; every
// lane gets both.
__device__ __forceinline__ void warp_counts(const Shared& sh, uint32_t tau, bool exact, uint32_t& def, uint32_t& tie) {
    const uint32_t* h = sh.whist() + (threadIdx.x >> 5) * kSmall + 8 * lane_id();
    const uint4 a = *reinterpret_cast<const uint4*>(h), b = *reinterpret_cast<const uint4*>(h + 4);
    const uint32_t v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t d = 0, t = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t bin = 8 * lane_id() + static_cast<uint32_t>(i);
        d += (bin > tau || (exact && bin == tau)) ? v[i] : 0u;
        t += (!exact && bin == tau) ? v[i] : 0u;
    }
    def = __reduce_add_sync(kFull, d);
    tie = __reduce_add_sync(kFull, t);
}

// The classify-and-write pass over this warp's n candidates once the
// threshold bin tau is known: candidates above it (at or above it when
// exact) take output slots def_base, def_base + 1, ... in order; members of
// the bin take tie-list entries tie_base, ... for ranking (the list may be
// another CTA's). The bases come from the warps' counts, so the pass needs
// no atomics.
template <bool kPaged, class BinOf>
__device__ __forceinline__ void classify_write(uint32_t region, uint32_t n, BinOf bin_of, uint32_t tau,
                                               bool exact, uint32_t def_base, uint32_t tie_base,
                                               const TieList& ties, const Emitter<kPaged>& em) {
    const uint32_t n_round = (n + 31u) & ~31u;
    const uint32_t lt = lanemask_lt();
    for (uint32_t i = lane_id(); i < n_round; i += 32) {
        const bool valid = i < n;
        const uint2 e = valid ? ld_shared_v2(region + i * 8u) : make_uint2(0u, 0u);
        const uint32_t key = bits_key(e.x);
        const uint32_t bin = bin_of(key);
        const bool def = valid && (bin > tau || (exact && bin == tau));
        const uint32_t m = __ballot_sync(kFull, def);
        if (def) em.write(def_base + static_cast<uint32_t>(__popc(m & lt)), static_cast<int32_t>(e.y));
        def_base += static_cast<uint32_t>(__popc(m));
        if (!exact) {
            const bool tie = valid && bin == tau;
            const uint32_t mt = __ballot_sync(kFull, tie);
            if (tie) {
                const uint32_t t = tie_base + static_cast<uint32_t>(__popc(mt & lt));
                if (t < static_cast<uint32_t>(kMaxRankTies)) {
                    ties.key[t] = key;
                    ties.pos[t] = static_cast<int32_t>(e.y);
                }
            }
            tie_base += static_cast<uint32_t>(__popc(mt));
        }
    }
}

// Outcome of the fast finish.
enum FinishResult { kFinished = 0, kNeedLevels = 1, kNeedExact = 2 };

// The per-warp-region finish when the threshold lies past the first window of
// 255 prefixes over the bound (as rebin_top for the compact lists, with the
// candidates' full keys at hand): windows narrow from one spanning every top-
// bin member onto the threshold, until its bin is one prefix wide or holds at
// most kMaxRankTies candidates. On return `win` is the last window and the
// per-warp histograms hold its counts. Every thread calls.
__device__ Threshold rebin_regions(uint32_t region, uint32_t n, uint32_t base16, uint32_t k, PrefixWindow& win,
                                   const Shared& sh) {
    constexpr uint32_t kTop = kSmall - 1, kWide = kSmall - 2;
    uint32_t hi = 0;
    for (uint32_t i = lane_id(); i < n; i += 32) hi = max(hi, bits_key(ld_shared_u32(region + i * 8u)) >> 16);
    hi = __reduce_max_sync(kFull, hi);
    if (lane_id() == 0) atomicMax(&sh.cnt()[4], hi);
    __syncthreads();
    win = PrefixWindow{base16 + kTop, 0u};
    uint32_t span = sh.cnt()[4] - win.lo;  // every top-bin member's prefix lies in [lo, lo + span]
    while ((span >> win.shift) >= kWide) ++win.shift;
    const uint32_t whist = saddr(sh.whist() + (threadIdx.x >> 5) * kSmall);
    Threshold t{0u, 0u, 0u, false};
    for (int pass = 0; pass < 4; ++pass) {
        clear_words(sh.whist(), kWarps * kSmall);
        __syncthreads();
        count_candidates(region, n, win, whist);
        __syncthreads();
        if (threadIdx.x < kSmall) sh.hist()[threadIdx.x] = sum_warp_bins(sh);
        __syncthreads();
        t = find_threshold(sh.hist(), kSmall, k, sh);
        if (!t.found || t.bin == 0u || t.bin == kTop) break;  // (cannot happen: the members number at least k)
        if (win.shift == 0u || t.count <= static_cast<uint32_t>(kMaxRankTies)) return t;
        win.lo += (t.bin - 1u) << win.shift;
        span = (1u << win.shift) - 1u;
        win.shift = 0;
        while ((span >> win.shift) >= kWide) ++win.shift;
    }
    t.found = false;
    return t;
}

// The end of the per-warp-region finish once the threshold bin t (in the
// bins of `bin_of`) is known and the per-warp histograms hold their counts:
// slots for the candidates above it, the bin's members ranked.
template <bool kPaged, class BinOf>
__device__ __forceinline__ void finish_classify(uint32_t region, uint32_t n, BinOf bin_of, const Threshold& t,
                                                uint32_t k, const Shared& sh, const Emitter<kPaged>& em) {
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const uint32_t need = k - t.above;
    const bool exact = t.count == need;
    uint32_t def, tie;
    warp_counts(sh, t.bin, exact, def, tie);
    if (lane_id() == 0) {
        sh.red()[warp] = def;
        sh.red()[kWarps + warp] = tie;
    }
    __syncthreads();
    uint32_t def_base = 0, tie_base = 0;
#pragma unroll
    for (int q = 0; q < kWarps; ++q) {
        def_base += q < warp ? sh.red()[q] : 0u;
        tie_base += q < warp ? sh.red()[kWarps + q] : 0u;
    }
    const TieList ties = tie_list(sh.ties());
    classify_write<kPaged>(region, n, bin_of, t.bin, exact, def_base, tie_base, ties, em);
    if (!exact) {
        __syncthreads();
        rank_threshold_bin(t.count, need, k, ties.key, ties.pos, ties.rank,
                           [&](uint32_t s, int32_t pos) { em.write(s, pos); });
    }
}

// The fast finish of a single-CTA row (every candidate of the row in this
// CTA's regions, `ovf` this warp's overflow flag). kNeedExact: nothing was
// written, the caller runs the exact path from scratch. kNeedLevels: the
// threshold bin is too full to rank; st then holds its 16-bit prefix and the
// caller continues with the low-16-bit radix levels over the regions.
template <bool kPaged>
__device__ FinishResult finish_solo(uint32_t bound_key, uint32_t wcount, bool ovf, uint32_t k, SelState& st,
                                    uint32_t cap, const Shared& sh, const Emitter<kPaged>& em) {
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const uint32_t region = saddr(sh.cand) + static_cast<uint32_t>(warp) * cap * 8u;
    const uint32_t n = min(wcount, cap);
    const uint32_t base16 = bound_key >> 16;
    if (lane_id() == 0) {
        sh.wcnt()[warp] = n;
        if (ovf) atomicOr(&sh.cnt()[3], 1u);
    }
    if (!ovf) count_candidates(region, n, BoundWindow{base16}, saddr(sh.whist() + warp * kSmall));
    if (kPaged) asm volatile("cp.async.wait_all;" ::: "memory");  // page-table entries, published below
    __syncthreads();
    if (sh.cnt()[3] != 0u) return kNeedExact;
    if (threadIdx.x < kSmall) sh.hist()[threadIdx.x] = sum_warp_bins(sh);
    __syncthreads();
    Threshold t = find_threshold(sh.hist(), kSmall, k, sh);
    // the threshold past the first window: re-bin (the 512-thread build; the
    // 256-thread one, at its 64-register cap, sends such rows to the exact
    // path, which keeps its common path's code as it was: 0.7 % on the extend
    // chunks otherwise)
    bool windowed = false;
    PrefixWindow win{0u, 0u};
    if constexpr (kThreads == 512) {
        windowed = t.found && t.bin == static_cast<uint32_t>(kSmall - 1);
        if (windowed) t = rebin_regions(region, n, base16, k, win, sh);
    }
    if (!t.found || t.bin == static_cast<uint32_t>(kSmall - 1)) return kNeedExact;
    const uint32_t need = k - t.above;
    const bool exact = t.count == need;
    if (!exact && t.count > static_cast<uint32_t>(kMaxRankTies)) {
        if (windowed) return kNeedExact;
        st = SelState{static_cast<uint64_t>(base16 + t.bin) << 48, 0xFFFFull << 48, need, false};
        return kNeedLevels;
    }
    if (windowed) finish_classify<kPaged>(region, n, win, t, k, sh, em);
    else finish_classify<kPaged>(region, n, BoundWindow{base16}, t, k, sh, em);
    return kFinished;
}

// ----------------------------------------------------------------------------
// exact paths (used when the fast path's self-check fails)
// ----------------------------------------------------------------------------

// Appends every in-window element of the tile whose key is at least the bound
// (thr = pass_threshold(bound)) to the contiguous list of (key, position)
// `list`, counted in sh.cnt()[0] (one shared atomic per warp); entries past
// `cap` are dropped (callers count first).
template <bool kNonNeg>
__device__ void collect_tile(const int4 (&v)[kTileVecs], uint32_t thr, int j0, int je, int rem, int len,
                             const Shared& sh, uint2* list, int cap) {
    const uint32_t valid = tile_valid(j0, je, rem, len);
    uint32_t c = 0;
#pragma unroll
    for (int e = 0; e < kTileElems; ++e) c += (passes<kNonNeg>(tile_elem(v, e), thr) && ((valid >> e) & 1u)) ? 1u : 0u;
    const uint32_t incl = warp_inclusive_scan(c);
    const uint32_t total = __shfl_sync(kFull, incl, 31);
    if (total == 0) return;
    uint32_t base = 0;
    if (lane_id() == 31) base = atomicAdd(&sh.cnt()[0], total);
    uint32_t idx = __shfl_sync(kFull, base, 31) + incl - c;
    const int p0 = 4 * (j0 + static_cast<int>(threadIdx.x)) - rem;
#pragma unroll
    for (int e = 0; e < kTileElems; ++e) {
        const int32_t b = tile_elem(v, e);
        if (passes<kNonNeg>(b, thr) && ((valid >> e) & 1u)) {
            if (idx < static_cast<uint32_t>(cap))
                list[idx] = make_uint2(bits_key(static_cast<uint32_t>(b)),
                                          static_cast<uint32_t>(p0 + (e >> 2) * (4 * kThreads) + (e & 3)));
            ++idx;
        }
    }
}

// The exact path of a single-CTA row read from global memory: a full level-1
// histogram pass; then, when the elements at or above its threshold bin fit
// the candidate buffer, one more pass collects them and the remaining levels
// run on the buffer, else the levels re-read the row.
template <bool kPaged>
__device__ __noinline__ void exact_row_global(const float4* vbase, int nv, int rem, int len, uint32_t k, bool det,
                                 const Shared& sh0, const Emitter<kPaged>& em) {
    constexpr int T = kTileVecs * kThreads;
    const Shared sh = exact_view(sh0, false);
    if (threadIdx.x == 0) atomicAdd(em.stats, 1u);
    uint2* list = exact_list(sh);
    const SoloMerge mg;
    const GlobalSource all{vbase, 0, nv, rem, len};
    clear_words(sh.lvl, kBins);
    __syncthreads();
    uint32_t* hist = sh.lvl;
    all.visit([&](uint32_t kk, int32_t, bool valid) {
        if (valid) atomicAdd(&hist[kk >> 20], 1u);
    });
    const Threshold t1 = find_threshold(mg.merge(sh, kBins), kBins, k, sh);
    SelState st{0ull, 0ull, k, false};
    apply_level(st, kLvlKey12, t1);
    if (!st.exact && count_from(sh.lvl, kBins, t1.bin, sh) <= static_cast<uint32_t>(kXListCap)) {
        if (threadIdx.x == 0) sh.cnt()[0] = 0;
        __syncthreads();
        const uint32_t bound = t1.bin << 20, thr = pass_threshold(bound);
        for (int j0 = 0; j0 < nv; j0 += T) {
            int4 v[kTileVecs];
            load_bits(v, vbase, j0, nv);
            if (bound >= 0x80000000u) collect_tile<true>(v, thr, j0, nv, rem, len, sh, list, kXListCap);
            else collect_tile<false>(v, thr, j0, nv, rem, len, sh, list, kXListCap);
        }
        __syncthreads();
        const CandSource src{list, min(sh.cnt()[0], static_cast<uint32_t>(kXListCap))};
        run_levels(st, kLvlKey12 + 1, kLvlKeyLast, det, src, sh, mg);
        emit_selected<kPaged>(st, k, src, sh, mg, em);
    } else {
        run_levels(st, kLvlKey12 + 1, kLvlKeyLast, det, all, sh, mg);
        emit_selected<kPaged>(st, k, all, sh, mg, em);
    }
}

// ----------------------------------------------------------------------------
// routes of a single-CTA row
// ----------------------------------------------------------------------------

// Per-row inputs, after the data-error checks.
struct RowInfo {
    int32_t len, start, offset, table_row, token0;
};

__device__ __forceinline__ void park_row(const RowInfo& r, const Shared& sh) {
    if (threadIdx.x == 0) {
        int32_t* d = sh.row();
        d[0] = r.len, d[1] = r.start, d[2] = r.offset, d[3] = r.table_row, d[4] = r.token0;
    }
}
__device__ __forceinline__ RowInfo load_row(const Shared& sh) {
    const int32_t* d = sh.row();
    return RowInfo{d[0], d[1], d[2], d[3], d[4]};
}

// The page-table entries [first, first + n) of a row's table that window
// positions [p_lo, p_hi) map to (tokens token0 + p).
struct PageSpan {
    int32_t first;
    int n;
};
__device__ __forceinline__ PageSpan page_span(int32_t token0, int32_t page_bits, int32_t p_lo, int32_t p_hi) {
    const int32_t first = (token0 + p_lo) >> page_bits;
    return PageSpan{first, ((token0 + p_hi - 1) >> page_bits) - first + 1};
}

// PAGED: starts asynchronous copies into shared memory of the page-table
// entries that positions [p_lo, p_hi) map to, when they fit `cap` entries;
// the finish waits for them (cp.async.wait_all, then a barrier). Other
// lookups read global memory.
template <bool kPaged>
__device__ __forceinline__ void prefetch_pages(const Params& p, const RowInfo& r, int32_t p_lo, int32_t p_hi, int cap,
                                               const Shared& sh) {
    if (!kPaged || p_hi <= p_lo) return;
    const PageSpan ps = page_span(r.token0, p.page_bits, p_lo, p_hi);
    if (ps.n > cap) return;
    const int32_t* pt_row = p.page_table + static_cast<int64_t>(r.table_row) * p.page_table_stride + ps.first;
    for (int i = threadIdx.x; i < ps.n; i += kThreads) {
        const uint32_t dst = saddr(sh.pages + i);
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(pt_row + i) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <bool kPaged>
__device__ __forceinline__ Emitter<kPaged> make_emitter(const Params& p, int b, const RowInfo& r) {
    Emitter<kPaged> em;
    em.out = p.out + static_cast<int64_t>(b) * p.out_stride;
    em.out_raw = p.out_raw ? p.out_raw + static_cast<int64_t>(b) * p.k : nullptr;
    em.pt_row = kPaged ? p.page_table + static_cast<int64_t>(r.table_row) * p.page_table_stride : nullptr;
    em.pt_cached = nullptr;
    em.token0 = r.token0;
    em.pt_first = 0;
    em.pt_count = 0;
    em.page_bits = p.page_bits;
    em.offset = r.offset;
    em.k = static_cast<uint32_t>(p.k);
    em.flags = &p.hdr->flags;
    em.stats = &p.hdr->exact_rows;
    return em;
}

// The emitter of a row whose page-table entries for positions [p_lo, p_hi)
// were prefetched (prefetch_pages with the same arguments). Built after the
// filter, so none of it is live during the score pass.
template <bool kPaged>
__device__ __forceinline__ Emitter<kPaged> row_emitter(const Params& p, int b, const RowInfo& r, int32_t p_lo,
                                                       int32_t p_hi, int cap, const Shared& sh) {
    Emitter<kPaged> em = make_emitter<kPaged>(p, b, r);
    if (kPaged && p_hi > p_lo) {
        const PageSpan ps = page_span(r.token0, p.page_bits, p_lo, p_hi);
        if (ps.n <= cap) {
            em.pt_cached = sh.pages;
            em.pt_first = ps.first;
            em.pt_count = ps.n;
        }
    }
    return em;
}

// The rest of a row after the fast finish declined to rank its threshold
// bin (see finish_solo): the low-16-bit radix levels over the regions.
template <bool kPaged>
__device__ __noinline__ void finish_levels(SelState st, uint32_t k, bool det, const Shared sh,
                                           const Emitter<kPaged> em) {
    const RegionSource src{sh.cand, sh.wcnt(), kWarpCap};
    run_levels(st, kLvlLow16, kLvlLow16Last, det, src, sh, SoloMerge{});
    emit_selected<kPaged>(st, k, src, sh, SoloMerge{}, em);
}

// The exact path of a register-route row, from its registers.
template <bool kPaged>
__device__ __noinline__ void exact_row_registers(const int4 (&v)[kTileVecs], int rem, int len, uint32_t k, bool det,
                                                 const Shared sh0, const Emitter<kPaged> em) {
    const Shared sh = exact_view(sh0, false);
    if (threadIdx.x == 0) atomicAdd(em.stats, 1u);
    SelState st{0ull, 0ull, k, false};
    const RegSource src{v, rem, len};
    run_levels(st, kLvlKey12, kLvlKeyLast, det, src, sh, SoloMerge{});
    emit_selected<kPaged>(st, k, src, sh, SoloMerge{}, em);
}

// Register route: the whole aligned window (nv <= kTileVecs * kThreads
// vectors) is one register tile. The sample is every fourth position
// (positions 4j: lane `rem` of vector j), read from the registers.
template <bool kPaged, int kLay>
__device__ void register_row(const Params& p, int b, const float4* vbase, int nv, int rem, int len) {
    const uint32_t k = static_cast<uint32_t>(p.k);
    int4 v[kTileVecs];
    load_bits(v, vbase, 0, nv);
    uint32_t skey[kTileVecs];
    uint32_t vmask = 0;
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) {
        const int j = u * kThreads + static_cast<int>(threadIdx.x);
        const int32_t b = rem == 0 ? v[u].x : rem == 1 ? v[u].y : rem == 2 ? v[u].z : v[u].w;
        skey[u] = bits_key(static_cast<uint32_t>(b));
        vmask |= (4 * j < len ? 1u : 0u) << u;
    }
    const uint32_t bound_key =
        sample_bound<kTileVecs>(skey, vmask, static_cast<uint32_t>((len + 3) / 4), len, k, layout<kLay>());
    const uint32_t thr = pass_threshold(bound_key);
    const uint32_t valid = tile_valid(0, nv, rem, len);
    const int p0 = 4 * static_cast<int>(threadIdx.x) - rem;
    const uint32_t region = saddr(layout<kLay>().cand) + (threadIdx.x >> 5) * (kWarpCap * 8u);
    uint32_t wcount = 0;
    bool ovf = false;
    if (bound_key >= 0x80000000u) filter_tile<true, true>(v, thr, valid, p0, region, wcount, kWarpCap, ovf);
    else filter_tile<false, true>(v, thr, valid, p0, region, wcount, kWarpCap, ovf);
    const Shared sh = layout<kLay>();
    const RowInfo ri = load_row(sh);
    const bool det = (p.flags & TOPK_DETERMINISTIC) != 0;
    const Emitter<kPaged> em = row_emitter<kPaged>(p, b, ri, 0, len, kPageCache, sh);
    SelState st;
    const FinishResult r = finish_solo<kPaged>(bound_key, wcount, ovf, k, st, kWarpCap, sh, em);
    if (r == kFinished) return;
    if (r == kNeedLevels) {
        finish_levels<kPaged>(st, k, det, sh, em);
        return;
    }
    exact_row_registers<kPaged>(v, rem, len, k, det, sh, em);
}

// Asks the memory system to bring tile t of the window (vectors
// [t * T, min((t + 1) * T, nv))) into L2 ahead of its loads: one 1-D bulk
// prefetch (16-byte aligned start and size), issued by one thread, costing
// no registers while the bytes are in flight.
__device__ __forceinline__ void prefetch_tile_l2(const float4* vbase, int t, int nv) {
    constexpr int T = kTileVecs * kThreads;
    const int j = t * T;
    if (j >= nv) return;
    const uint32_t bytes = static_cast<uint32_t>(min(T, nv - j)) * 16u;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vbase + j), "r"(bytes) : "memory");
}
// Tiles requested into L2 beyond the two register tiles. 0: each register
// tile's bytes are asked for by one bulk prefetch a step before its loads
// (one 16 KB request instead of thousands of 16-byte ones), and no further;
// deeper prefetching was slower on the 1024-row extend chunk, where about
// 600 rows stream at once and L2 is no larger than the bytes in flight.
#ifndef TOPK_PREFETCH_TILES
#define TOPK_PREFETCH_TILES 0
#endif
constexpr int kPrefetchTiles = TOPK_PREFETCH_TILES;

// Streaming route (nv > kTileVecs * kThreads vectors): two register tiles in
// turn, one loading while the other is filtered, and the kPrefetchTiles
// tiles after those on their way into L2; the sample is read from global
// memory (spread over the whole window).
template <bool kNonNeg>
__device__ __forceinline__ void stream_filter(int4 (&cur)[kTileVecs], int4 (&nxt)[kTileVecs], const float4* vbase,
                                              int nv, int rem, int len, uint32_t thr, uint32_t region,
                                              uint32_t& wcount, bool& ovf) {
    constexpr int T = kTileVecs * kThreads;
    int j0 = 0;
    for (int t = 0;; t += 2) {
        if (threadIdx.x == 0) {  // tiles t + 2 + kPrefetchTiles, t + 3 + kPrefetchTiles into L2
            prefetch_tile_l2(vbase, t + 2 + kPrefetchTiles, nv);
            prefetch_tile_l2(vbase, t + 3 + kPrefetchTiles, nv);
        }
        filter_at<kNonNeg>(cur, thr, j0, nv, rem, len, region, wcount, kWarpCap, ovf);
        j0 += T;
        if (j0 >= nv) break;
        if (j0 + T < nv) load_bits(cur, vbase, j0 + T, nv);
        filter_at<kNonNeg>(nxt, thr, j0, nv, rem, len, region, wcount, kWarpCap, ovf);
        j0 += T;
        if (j0 >= nv) break;
        if (j0 + T < nv) load_bits(nxt, vbase, j0 + T, nv);
    }
}

// ----------------------------------------------------------------------------
// streamed rows: compact per-thread candidate lists
// ----------------------------------------------------------------------------
//
// Each thread appends its candidates to a list of its own: entry s of thread
// t is word s * kThreads + t of the candidate buffer (interleaved, so a
// warp's lanes storing their s-th entries hit 32 different banks). An entry
// packs the top 16 bits of the score's fp32 pattern (all the finish's
// histogram needs) with the element's 16-bit index l in the thread's share of
// the row: l = 16 * tile + 4 * u + c for lane c of the thread's vector u of a
// tile, so position = 4 * (tile * T + u * kThreads + t) + c - rem. The filter
// then needs no per-tile count and no warp scan: per element one compare, one
// add, one byte permute, one predicated store and one predicated add. The
// few members of the threshold bin, which need their full keys, are read
// again from global memory (L2).

constexpr int kListCap = kCandBytes / (kThreads * 4);  // entries per thread
constexpr uint32_t kListStride = kThreads * 4u;        // bytes between a thread's entries
constexpr int kListMaxTiles = 4096;                    // tiles a 16-bit index covers
static_assert(kTileVecs == 4 && kListCap >= 24, "list layout");

#define TOPK_LA_HEAD "{\n\t.reg .pred q, v, r;\n\t.reg .b32 t;\n\t"
#define TOPK_LA_GE "setp.ge.s32 q, %1, %2;\n\t"
#define TOPK_LA_LE "setp.le.u32 q, %1, %2;\n\t"
#define TOPK_LA_MASK "and.b32 t, %4, %7;\n\tsetp.ne.b32 v, t, 0;\n\t"
#define TOPK_LA_GE_M "setp.ge.and.s32 q, %1, %2, v;\n\t"
#define TOPK_LA_LE_M "setp.le.and.u32 q, %1, %2, v;\n\t"
#define TOPK_LA_ENTRY "add.u32 t, %3, %6;\n\tprmt.b32 t, t, %1, 0x7610;\n\t"
#define TOPK_LA_STORE "@q st.shared.u32 [%0], t;\n\t@q add.u32 %0, %0, %8;\n\t}"
#define TOPK_LA_STORE_CHK "setp.lt.and.u32 r, %0, %5, q;\n\t@r st.shared.u32 [%0], t;\n\t@q add.u32 %0, %0, %8;\n\t}"
#define TOPK_LA_ARGS                                                                                       \
    : "+r"(a) : "r"(bits), "r"(thr), "r"(lb), "r"(valid), "r"(lim), "n"(kOff), "n"(1 << kBit), "n"(kListStride) \
    : "memory"

// Appends the entry of element kOff of the tile (bits, index lb + kOff) at
// shared address a and advances a by one list stride when the bits pass the
// bound (thr: see passes); kMasked: only if bit kBit of `valid` is set;
// kChecked: the store is skipped at or past `lim` (a still advances, so a
// final a > lim reports the overflow).
template <bool kNonNeg, bool kMasked, bool kChecked, int kOff, int kBit>
__device__ __forceinline__ void list_append(uint32_t& a, int32_t bits, uint32_t thr, uint32_t lb, uint32_t valid,
                                            uint32_t lim) {
    if constexpr (!kMasked && !kChecked) {
        if constexpr (kNonNeg) asm volatile(TOPK_LA_HEAD TOPK_LA_GE TOPK_LA_ENTRY TOPK_LA_STORE TOPK_LA_ARGS);
        else asm volatile(TOPK_LA_HEAD TOPK_LA_LE TOPK_LA_ENTRY TOPK_LA_STORE TOPK_LA_ARGS);
    } else if constexpr (!kMasked) {
        if constexpr (kNonNeg) asm volatile(TOPK_LA_HEAD TOPK_LA_GE TOPK_LA_ENTRY TOPK_LA_STORE_CHK TOPK_LA_ARGS);
        else asm volatile(TOPK_LA_HEAD TOPK_LA_LE TOPK_LA_ENTRY TOPK_LA_STORE_CHK TOPK_LA_ARGS);
    } else {
        static_assert(kChecked, "masked tiles are always checked");
        if constexpr (kNonNeg)
            asm volatile(TOPK_LA_HEAD TOPK_LA_MASK TOPK_LA_GE_M TOPK_LA_ENTRY TOPK_LA_STORE_CHK TOPK_LA_ARGS);
        else asm volatile(TOPK_LA_HEAD TOPK_LA_MASK TOPK_LA_LE_M TOPK_LA_ENTRY TOPK_LA_STORE_CHK TOPK_LA_ARGS);
    }
}
#undef TOPK_LA_HEAD
#undef TOPK_LA_GE
#undef TOPK_LA_LE
#undef TOPK_LA_MASK
#undef TOPK_LA_GE_M
#undef TOPK_LA_LE_M
#undef TOPK_LA_ENTRY
#undef TOPK_LA_STORE
#undef TOPK_LA_STORE_CHK
#undef TOPK_LA_ARGS

template <bool kNonNeg, bool kMasked, bool kChecked>
__device__ __forceinline__ void list_tile(const int4 (&v)[kTileVecs], uint32_t thr, uint32_t lb, uint32_t valid,
                                          uint32_t& a, uint32_t lim) {
    for_each_elem<0>([&](auto ec) {
        constexpr int e = decltype(ec)::value;
        list_append<kNonNeg, kMasked, kChecked, e, e>(a, tile_elem(v, e), thr, lb, valid, lim);
    });
}

// Loads tile j0 (vectors j0 + u * kThreads + t) without bounds checks: for
// tiles wholly inside the aligned span.
__device__ __forceinline__ void load_bits_full(int4 (&v)[kTileVecs], const float4* vbase, int j0) {
    const float4* q = vbase + j0 + static_cast<int>(threadIdx.x);
#pragma unroll
    for (int u = 0; u < kTileVecs; ++u) v[u] = load_stream_bits(q + u * kThreads);
}

// One step of the streamed filter: tile tt (in v) into the lists, then the
// load of tile tt + kDist into v. Tiles [t_lo, t_hi) lie wholly inside the window
// (no masks, unchecked loads); a warp with a lane within one tile of its
// list's end takes the checked appends.
template <bool kNonNeg, int kDist>
__device__ __forceinline__ void list_step(int4 (&v)[kTileVecs], int tt, int t_lo, int t_hi, int n_tiles,
                                          const float4* vbase, int nv, int rem, int len, uint32_t thr,
                                          uint32_t& a, uint32_t lim) {
    constexpr int T = kTileVecs * kThreads;
    const uint32_t lb = static_cast<uint32_t>(tt) * kTileElems;
    if (tt >= t_lo && tt < t_hi) {
        if (__any_sync(kFull, a + static_cast<uint32_t>(kTileElems) * kListStride > lim))
            list_tile<kNonNeg, false, true>(v, thr, lb, 0xFFFFu, a, lim);
        else
            list_tile<kNonNeg, false, false>(v, thr, lb, 0xFFFFu, a, lim);
    } else {
        list_tile<kNonNeg, true, true>(v, thr, lb, tile_valid(tt * T, nv, rem, len), a, lim);
    }
    const int tn = tt + kDist;
    if (tn < t_hi) load_bits_full(v, vbase, tn * T);
    else if (tn < n_tiles) load_bits(v, vbase, tn * T, nv);
}

// The streamed window (nv <= kListMaxTiles tiles) into the lists: one
// register tile (tile 0 loaded by the caller), each tile's successor loaded
// right after it is filtered and asked into L2 by one bulk prefetch a step
// earlier, so its loads mostly hit L2 (a second register tile in flight was
// slower: the registers it holds cost more than the latency it hides with
// 32 warps per SM). a: this thread's list cursor (shared address), lim: its
// end.
template <bool kNonNeg>
__device__ __forceinline__ void stream_list(int4 (&cur)[kTileVecs], const float4* vbase, int nv, int rem, int len,
                                            uint32_t thr, uint32_t& a, uint32_t lim) {
    constexpr int T = kTileVecs * kThreads;
    const int n_tiles = (nv + T - 1) / T;
    const int t_lo = rem == 0 ? 0 : 1;     // tile 0 holds the rem lanes before the window
    const int t_hi = (len + rem) / (4 * T);  // tiles below it end inside the window
    for (int t = 0;; ++t) {
        if (threadIdx.x == 0) prefetch_tile_l2(vbase, t + 2, nv);
        list_step<kNonNeg, 1>(cur, t, t_lo, t_hi, n_tiles, vbase, nv, rem, len, thr, a, lim);
        if (t + 1 >= n_tiles) break;
    }
}

// Bits 31..16 of an entry's key (the order-preserving map of its top 16 bits).
__device__ __forceinline__ uint32_t entry_key16(uint32_t e) {
    return (e >> 16) ^ ((static_cast<uint32_t>(static_cast<int32_t>(e) >> 31) & 0x7FFFu) | 0x8000u);
}
// The window position of this thread's entry e: with l its low 16 bits,
// 4 * (tile * T + u * kThreads + t) + c - rem = ((l & ~3) << log2(kThreads))
// + (l & 3) + tbase, tbase = 4 * t - rem.
constexpr int kLogThreads = kThreads == 512 ? 9 : kThreads == 256 ? 8 : kThreads == 128 ? 7 : -1;
static_assert(kLogThreads > 0 && (1 << kLogThreads) == kThreads, "power-of-two teams");
__device__ __forceinline__ int32_t entry_pos(uint32_t e, int32_t tbase) {
    const uint32_t l = e & 0xFFFFu;
    return static_cast<int32_t>(((l & ~3u) << kLogThreads) + (l & 3u)) + tbase;
}
__device__ __forceinline__ uint32_t fine_bin16(uint32_t key16, uint32_t base16) {
    return min(key16 - base16, static_cast<uint32_t>(kSmall - 1));
}

// The compact finish when the threshold lies above the count pass's window
// of 255 prefixes over the bound (the bound many 16-bit prefix steps below
// the k-th score, as when the scores straddle zero or span many octaves):
// every winner is then a member of the top bin. The members' keys are read
// back from global memory (L2) and their 16-bit prefixes kept in the entries
// (the other entries get prefix 0; every member's is at least base16 + 255).
// Windows then narrow onto the threshold: bin 0 below `lo`, bin 1 + i the
// prefixes lo + (i << sh) .., bin 255 the rest above. The first window spans
// every member; each next one spans the previous threshold bin, until that
// bin is one prefix wide or holds at most kMaxRankTies members (the tie
// ranking reads full keys). On return the entries hold their bins and the
// per-warp histograms the last window's counts, as after the count pass.
// Every thread calls (the caller's condition is the same on every thread).
__device__ Threshold rebin_top(uint32_t* lp, uint32_t n, uint32_t base16, uint32_t k, int32_t tbase, const float* w,
                               uint32_t* whw, const Shared& sh) {
    const uint32_t* const wbits = reinterpret_cast<const uint32_t*>(w);
    constexpr uint32_t kTop = kSmall - 1, kWide = kSmall - 2;
    uint32_t hi = 0;
    for (uint32_t s = 0; s < n; ++s) {
        uint32_t e = lp[s * kThreads];
        if ((e >> 16) == kTop) {
            const uint32_t p16 = bits_key(__ldg(wbits + entry_pos(e, tbase))) >> 16;
            hi = max(hi, p16);
            e = (p16 << 16) | (e & 0xFFFFu);
        } else {
            e &= 0xFFFFu;
        }
        lp[s * kThreads] = e;
    }
    hi = __reduce_max_sync(kFull, hi);
    if (lane_id() == 0) atomicMax(&sh.cnt()[4], hi);
    __syncthreads();
    uint32_t lo = base16 + kTop;
    uint32_t span = sh.cnt()[4] - lo;  // the members' prefixes lie in [lo, lo + span]
    uint32_t shift = 0;
    while ((span >> shift) >= kWide) ++shift;
    Threshold t{0u, 0u, 0u, false};
    for (int pass = 0; pass < 4; ++pass) {
        clear_words(sh.whist(), kWarps * kSmall);
        __syncthreads();
        for (uint32_t s = 0; s < n; ++s) {
            const uint32_t p16 = lp[s * kThreads] >> 16;
            if (p16 >= lo) atomicAdd(&whw[1u + min((p16 - lo) >> shift, kWide)], 1u);
        }
        __syncthreads();
        if (threadIdx.x < kSmall) sh.hist()[threadIdx.x] = sum_warp_bins(sh);
        __syncthreads();
        t = find_threshold(sh.hist(), kSmall, k, sh);
        if (!t.found || t.bin == 0u || t.bin == kTop) {  // (cannot happen: the members number at least k)
            t.found = false;
            return t;
        }
        if (shift == 0u || t.count <= static_cast<uint32_t>(kMaxRankTies)) break;
        lo += (t.bin - 1u) << shift;
        span = (1u << shift) - 1u;
        shift = 0;
        while ((span >> shift) >= kWide) ++shift;
    }
    if (shift != 0u && t.count > static_cast<uint32_t>(kMaxRankTies)) t.found = false;
    for (uint32_t s = 0; s < n; ++s) {
        const uint32_t e = lp[s * kThreads];
        const uint32_t p16 = e >> 16;
        const uint32_t bin = p16 >= lo ? 1u + min((p16 - lo) >> shift, kWide) : 0u;
        lp[s * kThreads] = (bin << 16) | (e & 0xFFFFu);
    }
    return t;
}

// The fast finish over the compact lists (n_raw: this thread's appends, more
// than kListCap meaning its list overflowed); w: the window's scores, for
// the threshold bin's full keys. As finish_solo, except that a threshold bin
// too full to rank also sends the row to the exact path, that the count pass
// writes each entry's bin over its top 16 bits for the classify pass, and
// that the selected positions are first gathered in shared memory (the
// per-warp histograms' space, free by then; a warp's definite entries of one
// list depth take consecutive slots, threshold-bin members go to the tie list
// through a shared counter) and then written out slot by slot, so that every
// global store is coalesced. kNeedExact: nothing was written.
template <bool kPaged>
__device__ __forceinline__ FinishResult finish_list(uint32_t bound_key, uint32_t n_raw, uint32_t k, int rem, const float* w,
                                    const Shared& sh, const Emitter<kPaged>& em) {
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const bool ovf = n_raw > static_cast<uint32_t>(kListCap);
    const uint32_t n = min(n_raw, static_cast<uint32_t>(kListCap));
    const uint32_t nmax = __reduce_max_sync(kFull, n);
    const uint32_t base16 = bound_key >> 16;
    uint32_t* const lp = reinterpret_cast<uint32_t*>(sh.cand) + threadIdx.x;  // entry s at lp[s * kThreads]
    uint32_t* const whw = sh.whist() + warp * kSmall;
    auto count_pass = [&](auto nonneg) {
        // a non-negative bound leaves only non-negative scores: key16 = top16 | 0x8000
        constexpr bool kNN = decltype(nonneg)::value;
        const uint32_t d16 = base16 - 0x8000u;
#pragma unroll 2
        for (uint32_t s = 0; s < nmax; ++s) {
            if (s < n) {
                const uint32_t e = lp[s * kThreads];
                const uint32_t bin = kNN ? min((e >> 16) - d16, static_cast<uint32_t>(kSmall - 1))
                                         : fine_bin16(entry_key16(e), base16);
                atomicAdd(&whw[bin], 1u);
                lp[s * kThreads] = __byte_perm(e, bin, 0x5410);  // (bin << 16) | (e & 0xFFFF)
            }
        }
    };
    if (bound_key >= 0x80000000u) count_pass(std::true_type{});
    else count_pass(std::false_type{});
    if (kPaged) asm volatile("cp.async.wait_all;" ::: "memory");  // page-table entries, published below
    if (__syncthreads_or(ovf)) return kNeedExact;
    if (threadIdx.x < kSmall) sh.hist()[threadIdx.x] = sum_warp_bins(sh);
    __syncthreads();
    Threshold t = find_threshold(sh.hist(), kSmall, k, sh);
    const int32_t tbase = 4 * static_cast<int32_t>(threadIdx.x) - rem;
    if (t.found && t.bin == static_cast<uint32_t>(kSmall - 1)) t = rebin_top(lp, n, base16, k, tbase, w, whw, sh);
    if (!t.found || t.bin == static_cast<uint32_t>(kSmall - 1)) return kNeedExact;
    const uint32_t need = k - t.above;
    const bool exact = t.count == need;
    if (!exact && t.count > static_cast<uint32_t>(kMaxRankTies)) return kNeedExact;
    uint32_t def, tie;
    warp_counts(sh, t.bin, exact, def, tie);
    if (lane_id() == 0) sh.red()[warp] = def;
    const uint32_t tau = t.bin;
    // bins above the threshold bin, and the threshold bin itself when exact
    const uint32_t lowest = exact ? tau : tau + 1u;
    const TieList ties = tie_list(sh.ties());
    __syncthreads();  // the warps' counts
    uint32_t slot = 0;
#pragma unroll
    for (int q = 0; q < kWarps; ++q) slot += q < warp ? sh.red()[q] : 0u;
    const uint32_t lt = lanemask_lt();
    static_assert(kWarps * kSmall >= TOPK_MAX_K, "the gathered slots fit the per-warp histograms");
    int32_t* const stage = reinterpret_cast<int32_t*>(sh.whist());  // slot -> position
    uint32_t* const n_ties = &sh.cnt()[2];
#pragma unroll 2
    for (uint32_t s = 0; s < nmax; ++s) {
        const bool valid = s < n;
        const uint32_t e = valid ? lp[s * kThreads] : 0u;
        const uint32_t bin = e >> 16;
        const bool d = valid && bin >= lowest;
        const uint32_t m = __ballot_sync(kFull, d);
        const uint32_t sl = slot + static_cast<uint32_t>(__popc(m & lt));
        if (d && sl < k) stage[sl] = entry_pos(e, tbase);  // (sl < k always holds when consistent)
        slot += static_cast<uint32_t>(__popc(m));
        if (!exact && valid && bin == tau)  // a threshold-bin member (few per row)
            ties.pos[atomicAdd(n_ties, 1u)] = entry_pos(e, tbase);
    }
    if (!exact) {
        __syncthreads();  // the members' positions; their keys are read in one round trip
        if (threadIdx.x < t.count)
            ties.key[threadIdx.x] = bits_key(__ldg(reinterpret_cast<const uint32_t*>(w) + ties.pos[threadIdx.x]));
        __syncthreads();
        rank_threshold_bin(t.count, need, k, ties.key, ties.pos, ties.rank, [&](uint32_t s, int32_t pos) {
            if (s < k) stage[s] = pos;
        });
    }
    __syncthreads();  // every slot gathered
    const bool vec = (k & 3u) == 0u && ((reinterpret_cast<uintptr_t>(em.out) | reinterpret_cast<uintptr_t>(em.out_raw)) & 15u) == 0u;
    if (vec) {  // 16-byte rows: four slots per store
        const int4* st4 = reinterpret_cast<const int4*>(stage);
        for (uint32_t i = threadIdx.x; i < k / 4u; i += kThreads) {
            const int4 q = st4[i];
            reinterpret_cast<int4*>(em.out)[i] = make_int4(em.value(q.x), em.value(q.y), em.value(q.z), em.value(q.w));
            if (em.out_raw) reinterpret_cast<int4*>(em.out_raw)[i] = q;
        }
    } else {
        for (uint32_t i = threadIdx.x; i < k; i += kThreads) em.write(i, stage[i]);
    }
    return kFinished;
}

// Streaming route (nv > kTileVecs * kThreads vectors): the bound comes from
// the row's spread sample, taken first while the head tiles travel into L2.
template <bool kPaged, int kLay>
__device__ void stream_row(const Params& p, int b, const float* w, const float4* vbase, int nv, int rem, int len) {
    const uint32_t k = static_cast<uint32_t>(p.k);
    constexpr int T = kTileVecs * kThreads;
    int4 cur[kTileVecs], nxt[kTileVecs];
    // the spread sample first; once it is in, the head tiles travel into L2
    // while the bound is searched
    const SpreadSample ss = spread_load(vbase, nv, rem, len);  // nv > T >= 1024
    const uint32_t bound_key = spread_bound(ss, spread_count(vbase, nv, rem, len), len, k, layout<kLay>(), [&] {
        if (threadIdx.x == 0)
            for (int t = 0; t < 2 + kPrefetchTiles; ++t) prefetch_tile_l2(vbase, t, nv);
    });
    load_bits(cur, vbase, 0, nv);
    const uint32_t thr = pass_threshold(bound_key);
#if TOPK_COMPACT_LISTS
    if (nv <= kListMaxTiles * T) {
        const uint32_t a0 = saddr(layout<kLay>().cand) + threadIdx.x * 4u;
        const uint32_t lim = a0 + static_cast<uint32_t>(kListCap) * kListStride;
        uint32_t a = a0;
        if (bound_key >= 0x80000000u) stream_list<true>(cur, vbase, nv, rem, len, thr, a, lim);
        else stream_list<false>(cur, vbase, nv, rem, len, thr, a, lim);
        const Shared sh = layout<kLay>();
        const RowInfo ri = load_row(sh);
        const Emitter<kPaged> em = row_emitter<kPaged>(p, b, ri, 0, len, kPageCache, sh);
        if (finish_list<kPaged>(bound_key, (a - a0) / kListStride, k, rem, w, sh, em) == kFinished) return;
        exact_row_global<kPaged>(vbase, nv, rem, len, k, (p.flags & TOPK_DETERMINISTIC) != 0, sh, em);
        return;
    }
#endif
    // rows beyond the lists' 16-bit index (more than kListMaxTiles tiles):
    // per-warp regions of (bits, position), two register tiles in turn
    load_bits(nxt, vbase, T, nv);
    const uint32_t region = saddr(layout<kLay>().cand) + (threadIdx.x >> 5) * (kWarpCap * 8u);
    uint32_t wcount = 0;
    bool ovf = false;
    if (bound_key >= 0x80000000u) stream_filter<true>(cur, nxt, vbase, nv, rem, len, thr, region, wcount, ovf);
    else stream_filter<false>(cur, nxt, vbase, nv, rem, len, thr, region, wcount, ovf);
    const Shared sh = layout<kLay>();
    const RowInfo ri = load_row(sh);
    const bool det = (p.flags & TOPK_DETERMINISTIC) != 0;
    const Emitter<kPaged> em = row_emitter<kPaged>(p, b, ri, 0, len, kPageCache, sh);
    SelState st;
    const FinishResult r = finish_solo<kPaged>(bound_key, wcount, ovf, k, st, kWarpCap, sh, em);
    if (r == kFinished) return;
    if (r == kNeedLevels) {
        finish_levels<kPaged>(st, k, det, sh, em);
        return;
    }
    exact_row_global<kPaged>(vbase, nv, rem, len, k, det, sh, em);
}

// ----------------------------------------------------------------------------
// kernels
// ----------------------------------------------------------------------------


// Reads row b's inputs; a negative length, start or packed page-table start
// makes the row empty and is counted (seq_len < 0 already by the plan when
// `planned`).
__device__ __forceinline__ RowInfo row_info(const Params& p, int b, bool kPagedMode) {
    RowInfo r;
    r.len = p.seq_lens[b];
    r.start = p.row_starts ? p.row_starts[b] : 0;
    r.offset = kPagedMode ? 0 : p.out_offsets[b];
    r.table_row = (kPagedMode && p.row_to_batch) ? p.row_to_batch[b] : b;
    r.token0 = (kPagedMode && p.pt_row_starts) ? p.pt_row_starts[b] : 0;
    return r;
}

__device__ __forceinline__ void check_row(RowInfo& r, bool planned, bool counter_thread, const Params& p) {
    if (r.len < 0 || r.start < 0 || r.token0 < 0) {
        if (counter_thread && (!planned || r.len >= 0)) atomicAdd(&p.hdr->error_rows, 1u);
        r.len = 0;
        r.token0 = 0;
        r.start = 0;
    }
}

// One row on one CTA (trivial, register or streaming route); the shared
// counters and histograms must be zero.
template <bool kPaged, int kLay>
__device__ void solo_row(const Params& p, int b, const RowInfo& r) {
    if (p.positions) swa_tail(p, b, r.len);
    const uint32_t k = static_cast<uint32_t>(p.k);
    if (r.len <= p.k) {
        trivial_row<kPaged>(r.len, k, make_emitter<kPaged>(p, b, r), p.positions == nullptr);
        return;
    }
    prefetch_pages<kPaged>(p, r, 0, r.len, kPageCache, layout<kLay>());
    park_row(r, layout<kLay>());  // read back after the score pass (published by its barriers)
    const int rem = r.start & 3;
    const float* w = p.scores + static_cast<int64_t>(b) * p.score_stride + r.start;
    const float4* vbase = reinterpret_cast<const float4*>(w - rem);
    const int nv = (r.len + rem + 3) >> 2;
    if (nv <= kTileVecs * kThreads) register_row<kPaged, kLay>(p, b, vbase, nv, rem, r.len);
    else stream_row<kPaged, kLay>(p, b, w, vbase, nv, rem, r.len);
}

// Zeroes the shared state one row needs (histograms, counters). No barrier.
__device__ __forceinline__ void clear_row_state(const Shared& sh) {
    clear_words(sh.shist(), 2 * kSmallWords);
    clear_words(sh.hist(), 2 * kSmallWords + kWarps * kSmall);  // hist, mhist, whist
    if (threadIdx.x < 48) sh.res()[threadIdx.x] = 0;  // res, cnt, wcnt (not the parked row)
}

// One CTA per row; rows come from the plan's order (longest first), rows the
// plan gave to the cluster path are skipped (their CTAs exit at once).
// kMinBlocks: CTAs per SM the register budget is sized for.
template <bool kPaged, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) topk_rows_kernel(const __grid_constant__ Params p) {
    clear_row_state(layout<kLayRows>());  // shared memory only: before the grid dependency
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
    const RowInfo r0 = row_info(p, b0, kPaged);
    const bool planned = magic == kPlanMagic && h_batch == p.batch && h_k == p.k;
    int b = b0;
    if (planned) {
        if (b0 >= n_order) return;
        b = ord;
    } else if (blockIdx.x == 0 && threadIdx.x == 0) {
        atomicOr(&p.hdr->flags, TOPK_DEVICE_FLAG_PLAN_MISMATCH);
    }
    RowInfo r = b == b0 ? r0 : row_info(p, b, kPaged);
    check_row(r, planned, threadIdx.x == 0, p);
    __syncthreads();  // the cleared state is visible
    solo_row<kPaged, kLayRows>(p, b, r);
}

#if TOPK_WITH_CLUSTER
// ----------------------------------------------------------------------------
// cluster route: bulk-copy staging, the cluster finish
// ----------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* m, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(m)), "r"(count) : "memory");
}

// One arrival plus the byte count the bulk copies completing on `m` will bring.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* m, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(m)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* m, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(m)), "r"(parity)
        : "memory");
    return ok != 0u;
}

// Waits for phase `parity` of `m` to complete, at most kWaitCycles; past that
// it flags TOPK_DEVICE_FLAG_TIMEOUT and returns (the caller goes on, so no
// barrier is left unmatched; the result is then flagged as unreliable).
__device__ void mbar_wait(uint64_t* m, uint32_t parity, uint32_t* flags) {
    if (mbar_try_wait(m, parity)) return;
    const long long t0 = clock64();
    while (!mbar_try_wait(m, parity)) {
        if (clock64() - t0 > kWaitCycles) {
            if (lane_id() == 0) atomicOr(flags, TOPK_DEVICE_FLAG_TIMEOUT);
            return;
        }
    }
}

// Chunk c of this CTA's slice, vectors [jb + c * kStageVecs, ...) of the
// aligned window, into stage c % kStages by one 1-D bulk copy (16-byte
// aligned source, destination and size), completing on that stage's
// mbarrier. One thread issues it.
__device__ __forceinline__ void issue_chunk(const Shared& sh, const float4* vbase, int jb, int je, int c) {
    const int s = c % kStages;
    const int j = jb + c * kStageVecs;
    const uint32_t bytes = static_cast<uint32_t>(min(kStageVecs, je - j)) * 16u;
    mbar_expect_tx(&sh.mbar()[s], bytes);
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_addr(sh.stage + s * kStageVecs)),
                 "l"(vbase + j), "r"(bytes), "r"(smem_addr(&sh.mbar()[s]))
                 : "memory");
}

// The exact radix path over this CTA's slice (levels merged over the
// cluster), from the staged copy when it is whole, else from global memory.
// Ends with a cluster barrier (no CTA reads another's histograms after it).
template <bool kPaged>
__device__ __noinline__ void exact_slice(const float4* vbase, const float4* staged, int jb, int je, int rem, int len, uint32_t k,
                            bool det, const Shared& sh0, const Emitter<kPaged>& em) {
    const Shared sh = exact_view(sh0, true);
    if (threadIdx.x == 0) atomicAdd(em.stats, 1u);
    SelState st{0ull, 0ull, k, false};
    const ClusterMerge mg;
    if (staged) {
        const VecSource<false> src{staged - jb, jb, je, rem, len};
        run_levels(st, kLvlKey12, kLvlKeyLast, det, src, sh, mg);
        emit_selected<kPaged>(st, k, src, sh, mg, em);
    } else {
        const GlobalSource src{vbase, jb, je, rem, len};
        run_levels(st, kLvlKey12, kLvlKeyLast, det, src, sh, mg);
        emit_selected<kPaged>(st, k, src, sh, mg, em);
    }
    cg::this_cluster().sync();
}

// The cluster finish when the threshold lies past the first window of 255
// prefixes over the bound (as rebin_regions, with the windows' histograms
// merged into every CTA's mhist): every decision comes from the merged
// histograms, which are the same in every CTA, so every CTA takes the same
// number of cluster barriers. On return `win` is the last window and this
// CTA's per-warp histograms hold its counts. Every thread of the cluster calls.
__device__ Threshold rebin_cluster(uint32_t region, uint32_t n, uint32_t base16, uint32_t k, PrefixWindow& win,
                                   const Shared& sh, cg::cluster_group& cluster) {
    constexpr uint32_t kTop = kSmall - 1, kWide = kSmall - 2;
    uint32_t hi = 0;
    for (uint32_t i = lane_id(); i < n; i += 32) hi = max(hi, bits_key(ld_shared_u32(region + i * 8u)) >> 16);
    hi = __reduce_max_sync(kFull, hi);
    if (lane_id() == 0 && hi != 0u) atomicMax(cluster.map_shared_rank(&sh.cnt()[4], 0), hi);
    cluster.sync();  // every CTA's largest prefix is in the leader's word
    win = PrefixWindow{base16 + kTop, 0u};
    uint32_t span = *cluster.map_shared_rank(&sh.cnt()[4], 0) - win.lo;  // the members' prefixes: [lo, lo + span]
    while ((span >> win.shift) >= kWide) ++win.shift;
    const uint32_t whist = saddr(sh.whist() + (threadIdx.x >> 5) * kSmall);
    Threshold t{0u, 0u, 0u, false};
    for (int pass = 0; pass < 4; ++pass) {
        clear_words(sh.whist(), kWarps * kSmall);
        clear_words(sh.mhist(), kSmallWords);
        cluster.sync();  // every CTA's merged histogram is clear before any counts arrive
        count_candidates(region, n, win, whist);
        __syncthreads();
        if (threadIdx.x < kSmall) {
            const uint32_t c = sum_warp_bins(sh);
            if (c != 0u)
                for (int q = 0; q < kClusterSize; ++q) atomicAdd(cluster.map_shared_rank(sh.mhist(), q) + threadIdx.x, c);
        }
        cluster.sync();  // every CTA's counts are in every CTA's mhist
        t = find_threshold(sh.mhist(), kSmall, k, sh);
        if (!t.found || t.bin == 0u || t.bin == kTop) break;  // (cannot happen: the members number at least k)
        if (win.shift == 0u || t.count <= static_cast<uint32_t>(kMaxRankTies)) return t;
        win.lo += (t.bin - 1u) << win.shift;
        span = (1u << win.shift) - 1u;
        win.shift = 0;
        while ((span >> win.shift) >= kWide) ++win.shift;
    }
    t.found = false;
    return t;
}

// One long row on the cluster: CTA `rank` takes the slice of vectors
// [jb, je) of the aligned window. Every CTA draws the same sample of the
// whole row, so every CTA computes the same bound; each filters its staged
// slice into its candidate regions and counts them in its own 256-bin
// histogram, which it then adds into every CTA's `mhist` with
// distributed-shared-memory reductions (so each CTA searches an identical
// copy); definite slots come from the leader's counter, and the threshold
// bin's members are gathered in the leader's tie list and ranked there.
// Ends with a cluster barrier after which the CTA's state is clean again
// (the leader resets its counters after it).
template <bool kPaged>
__device__ void cluster_row(const Params& p, int b, const Shared& sh, uint32_t& phase) {
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const uint32_t k = static_cast<uint32_t>(p.k);
    RowInfo r = row_info(p, b, kPaged);
    check_row(r, true, rank == 0 && threadIdx.x == 0, p);
    if (p.positions && rank == 0) swa_tail(p, b, r.len);
    if (r.len <= p.k) {  // only a data error (an emptied row) makes a cluster row this short
        if (rank == 0) trivial_row<kPaged>(r.len, k, make_emitter<kPaged>(p, b, r), p.positions == nullptr);
    } else {
        const int rem = r.start & 3;
        const float* w = p.scores + static_cast<int64_t>(b) * p.score_stride + r.start;
        const float4* vbase = reinterpret_cast<const float4*>(w - rem);
        const int nv = (r.len + rem + 3) >> 2;
        const int per = (nv + kClusterSize - 1) / kClusterSize;
        const int jb = min(nv, rank * per);
        const int je = min(nv, jb + per);
        const int n_chunks = (je - jb + kStageVecs - 1) / kStageVecs;
        const bool det = (p.flags & TOPK_DETERMINISTIC) != 0;
        const SpreadSample ss = spread_load(vbase, nv, rem, r.len);  // the same sample of the whole row in every CTA
        if (threadIdx.x == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of the stages come first
            for (int c = 0; c < min(n_chunks, kStages); ++c) issue_chunk(sh, vbase, jb, je, c);
        }
        const int32_t p_lo = max(4 * jb - rem, 0), p_hi = min(4 * je - rem, r.len);
        prefetch_pages<kPaged>(p, r, p_lo, p_hi, kClusterPageCache, sh);
        const uint32_t bound_key = spread_bound(ss, spread_count(vbase, nv, rem, r.len), r.len, k, sh, [] {});
        const uint32_t thr = pass_threshold(bound_key);
        const int warp = static_cast<int>(threadIdx.x >> 5);
        const uint32_t region = saddr(sh.cand) + static_cast<uint32_t>(warp) * (kClusterWarpCap * 8u);
        uint32_t wcount = 0;
        bool ovf = false;
        auto filter_slice = [&](auto nonneg) {
            constexpr bool kNN = decltype(nonneg)::value;
            for (int c = 0; c < n_chunks; ++c) {
                const int s = c % kStages;
                mbar_wait(&sh.mbar()[s], (phase >> s) & 1u, &p.hdr->flags);
                phase ^= 1u << s;
                const int j0 = jb + c * kStageVecs;
                int4 v[kTileVecs];
                load_bits_smem(v, sh.stage + s * kStageVecs, min(kStageVecs, je - j0));
                filter_at<kNN>(v, thr, j0, je, rem, r.len, region, wcount, kClusterWarpCap, ovf);
                if (c + kStages < n_chunks) {
                    __syncthreads();  // every thread is done with stage s
                    if (threadIdx.x == 0) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue_chunk(sh, vbase, jb, je, c + kStages);
                    }
                }
            }
        };
        if (bound_key >= 0x80000000u) filter_slice(std::true_type{});
        else filter_slice(std::false_type{});

        // the cluster finish
        const Emitter<kPaged> em = row_emitter<kPaged>(p, b, r, p_lo, p_hi, kClusterPageCache, sh);
        const uint32_t n = min(wcount, static_cast<uint32_t>(kClusterWarpCap));
        const uint32_t base16 = bound_key >> 16;
        if (lane_id() == 0) {
            sh.wcnt()[warp] = n;
            if (ovf)
                for (int q = 0; q < kClusterSize; ++q) atomicOr(cluster.map_shared_rank(&sh.cnt()[3], q), 1u);
        }
        if (!ovf) count_candidates(region, n, BoundWindow{base16}, saddr(sh.whist() + warp * kSmall));
        __syncthreads();  // this CTA's warp histograms are complete
        if (threadIdx.x < kSmall) {
            const uint32_t c = sum_warp_bins(sh);
            if (c != 0u)
                for (int q = 0; q < kClusterSize; ++q) atomicAdd(cluster.map_shared_rank(sh.mhist(), q) + threadIdx.x, c);
        }
        if (kPaged) asm volatile("cp.async.wait_all;" ::: "memory");
        cluster.sync();  // every CTA's counts are in every CTA's mhist, every flag is set
        bool done = false;
        if (sh.cnt()[3] == 0u) {  // the same in every CTA, like mhist
            Threshold t = find_threshold(sh.mhist(), kSmall, k, sh);
            PrefixWindow win{0u, 0u};
            const bool windowed = t.found && t.bin == static_cast<uint32_t>(kSmall - 1);
            if (windowed) t = rebin_cluster(region, n, base16, k, win, sh, cluster);
            const bool ranked = !windowed || t.count == k - t.above ||
                                t.count <= static_cast<uint32_t>(kMaxRankTies);  // else the exact slice path
            if (t.found && t.bin != static_cast<uint32_t>(kSmall - 1) && ranked) {
                const uint32_t need = k - t.above;
                const bool exact = t.count == need;
                if (!exact && t.count > static_cast<uint32_t>(kMaxRankTies)) {
                    SelState st{static_cast<uint64_t>(base16 + t.bin) << 48, 0xFFFFull << 48, need, false};
                    const RegionSource src{sh.cand, sh.wcnt(), kClusterWarpCap};
                    run_levels(st, kLvlLow16, kLvlLow16Last, det, src, sh, ClusterMerge{});
                    emit_selected<kPaged>(st, k, src, sh, ClusterMerge{}, em);
                    cluster.sync();  // no CTA reads another's level bins after this
                } else {
                    // slot bases: this warp's place in the CTA, the CTA's in the row (one
                    // atomic per CTA on the leader's counters)
                    uint32_t def, tie;
                    warp_counts(sh, t.bin, exact, def, tie);
                    if (lane_id() == 0) {
                        sh.red()[warp] = def;
                        sh.red()[kWarps + warp] = tie;
                    }
                    __syncthreads();
                    uint32_t def_base = 0, tie_base = 0, cta_def = 0, cta_tie = 0;
#pragma unroll
                    for (int q = 0; q < kWarps; ++q) {
                        const uint32_t dq = sh.red()[q], tq = sh.red()[kWarps + q];
                        def_base += q < warp ? dq : 0u;
                        tie_base += q < warp ? tq : 0u;
                        cta_def += dq;
                        cta_tie += tq;
                    }
                    if (threadIdx.x == 0) {
                        sh.res()[8] = cta_def ? atomicAdd(cluster.map_shared_rank(&sh.cnt()[1], 0), cta_def) : 0u;
                        sh.res()[9] = cta_tie ? atomicAdd(cluster.map_shared_rank(&sh.cnt()[2], 0), cta_tie) : 0u;
                    }
                    __syncthreads();
                    def_base += sh.res()[8];
                    tie_base += sh.res()[9];
                    const TieList leader_ties = tie_list(cluster.map_shared_rank(sh.ties(), 0));
                    if (windowed)
                        classify_write<kPaged>(region, n, win, t.bin, exact, def_base, tie_base, leader_ties, em);
                    else
                        classify_write<kPaged>(region, n, BoundWindow{base16}, t.bin, exact, def_base, tie_base,
                                               leader_ties, em);
                    if (!exact) {
                        cluster.sync();  // the tie list is complete
                        if (rank == 0) {
                            const TieList ties = tie_list(sh.ties());
                            rank_threshold_bin(t.count, need, k, ties.key, ties.pos, ties.rank,
                                               [&](uint32_t s, int32_t pos) { em.write(s, pos); });
                        }
                    }
                }
                done = true;
            }
        }
        if (!done)
            exact_slice<kPaged>(vbase, n_chunks <= kStages ? sh.stage : nullptr, jb, je, rem, r.len, k, det, sh, em);
    }
    __syncthreads();  // every local use of this row's state is done
    if (threadIdx.x == 0) sh.cnt()[3] = 0;
    clear_words(sh.hist(), 2 * kSmallWords + kWarps * kSmall);  // hist, mhist, whist
    clear_words(sh.shist(), 2 * kSmallWords);
    cluster.sync();  // the row is done in every CTA; no CTA touches another's state for it any more
    if (rank == 0 && threadIdx.x == 0) {
        sh.cnt()[1] = 0;
        sh.cnt()[2] = 0;
        sh.cnt()[4] = 0;
    }
}


// One thread-block cluster per long row, looping over the plan's cluster list.
// With all_rows set the same launch also takes every other row of the batch
// (after the cluster rows of its slot): rank 0 of a cluster runs it as a
// single-CTA row and the other CTAs of that cluster are done.
template <bool kPaged>
__global__ void __cluster_dims__(kClusterSize, 1, 1) __launch_bounds__(kThreads, 1)
    topk_cluster_kernel(const __grid_constant__ Params p, int all_rows) {
    const Shared sh = layout<kLayCluster>();
    clear_row_state(sh);  // shared memory only: before the grid dependency
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&sh.mbar()[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dependency_wait();
    allow_dependents();
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const PlanHeader* hdr = p.hdr;
    const bool planned = hdr->magic == kPlanMagic && hdr->batch == p.batch && hdr->k == p.k;
    const int n_cluster = planned ? hdr->n_cluster : 0;
    const int n_rest = !all_rows ? 0 : planned ? hdr->n_order : p.batch;
    if (all_rows && !planned && blockIdx.x == 0 && threadIdx.x == 0)
        atomicOr(&p.hdr->flags, TOPK_DEVICE_FLAG_PLAN_MISMATCH);
    const int n_slots = static_cast<int>(gridDim.x) / kClusterSize;
    const int slot = static_cast<int>(blockIdx.x) / kClusterSize;
    __syncthreads();  // the cleared state and the mbarriers are ready
    if (slot < n_cluster) cluster.sync();  // every CTA of the cluster runs before any reaches into another
    uint32_t phase = 0;
    for (int i = slot; i < n_cluster + n_rest; i += n_slots) {
        if (i < n_cluster) {
            cluster_row<kPaged>(p, p.cluster_rows[i], sh, phase);
            continue;
        }
        if (rank != 0) return;  // rows of the rest come after every cluster row of this slot
        const int b = planned ? p.order[i - n_cluster] : i - n_cluster;
        RowInfo r = row_info(p, b, kPaged);
        check_row(r, planned, threadIdx.x == 0, p);
        __syncthreads();
        clear_row_state(sh);
        __syncthreads();
        solo_row<kPaged, kLayClusterSolo>(p, b, r);
    }
}

#endif  // TOPK_WITH_CLUSTER

}  // namespace
}  // namespace TOPK_NS
}  // namespace topk_impl
