// Threshold bounds for the long rows of a large batch, computed ahead of the
// rows kernel: one CTA per row reads a sample spread over the row's window
// and writes a key that is, with overwhelming probability, at most the key
// of the row's k-th largest score. The rows kernel then starts filtering its
// row at once instead of sampling it first; on a busy SM that sample (a
// round trip to loaded memory, two histogram levels and their barriers) was
// the longest serial stretch of a row.
//
// The bound is only a hint. The rows kernel collects every element whose key
// is at least the bound and checks that it has at least k of them (and that
// they fit its buffers), else it finishes the row on its exact path, so any
// value here gives the right output; a poor one only costs time.
//
// The method is that of the rows kernel's own sample (a radix digit of the
// key histogrammed, as the 12-bit first digit of the PR #36684 page, "Feature
// and motivation", but on a sample): the sample's expected share of the
// top-k plus four standard deviations plus 2 is located in a 2048-bin
// histogram of the top 11 key bits and then in a 256-bin histogram of the
// next 8 bits, so the bound has 19 resolved bits.

#include <cuda_runtime.h>

#include <cstdint>

#include "topk_common.cuh"

namespace topk_impl {
namespace bound {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPieces = 128;                    // 64-byte pieces (4 vectors) of one row's sample
constexpr int kLogPieces = 7;
constexpr int kLoads = kPieces * 4 / kThreads;  // 16-byte vectors per thread
constexpr int kBins1 = 2048;                    // level 1: key bits 31..21
constexpr int kShift1 = 21;
constexpr int kRun = kBins1 / kThreads;         // level-1 bins per thread
constexpr int kBins2 = 256;                     // level 2: key bits 20..13 inside the level-1 bin
constexpr int kShift2 = 13;
static_assert(kLoads * kThreads == 4 * kPieces && (1 << kLogPieces) == kPieces, "shape");
static_assert(kRun % 4 == 0 && kBins2 == kThreads && kShift1 + 11 == 32 && kShift2 + 8 == kShift1, "shape");

// Order-preserving fp32 bits -> uint32 (negatives: all bits flipped;
// non-negatives: sign bit set).
__device__ __forceinline__ uint32_t bits_key(uint32_t b) {
    return b ^ (static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u);
}

// 16 bytes of scores as integer bits, not kept in L1; the lines stay in L2,
// where the rows kernel finds them again.
__device__ __forceinline__ int4 load_bits(const float4* p) {
    int4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void red_add_shared(uint32_t* a, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(a))), "r"(v)
                 : "memory");
}

// Row b's bound, for rows the rows kernel streams: seq_len > k and more than
// min_nv 16-byte vectors in the window's aligned span (shorter rows, and rows
// with a negative start or length, get no bound and the rows kernel reads
// none for them). The sample is 128 pieces of 4 consecutive vectors, each a
// whole 64-byte-aligned block of memory: with v0 the first vector of the span
// on such a boundary and nq the whole blocks from there inside the span,
// piece i is the block v0 + 4 * floor(i * nq / 128), so the pieces cover the
// whole row; 4 lanes load a piece, one vector each. Lanes outside the window
// are left out.
__global__ void __launch_bounds__(kThreads) topk_bound_kernel(const float* __restrict__ scores, int64_t stride,
                                                               const int32_t* __restrict__ row_starts,
                                                               const int32_t* __restrict__ seq_lens, int32_t k,
                                                               int32_t min_nv, uint32_t* __restrict__ bounds) {
    __shared__ __align__(16) uint32_t h1[kBins1];
    __shared__ __align__(16) uint32_t h2[kBins2];
    __shared__ uint32_t wtot[kWarps];
    __shared__ uint32_t res[2];
    const int tid = static_cast<int>(threadIdx.x);
    const uint32_t lane = threadIdx.x & 31u;
    const int warp = tid >> 5;
#pragma unroll
    for (int i = 0; i < kRun / 4; ++i) reinterpret_cast<uint4*>(h1)[i * kThreads + tid] = make_uint4(0u, 0u, 0u, 0u);
    h2[tid] = 0u;
    if (tid == 0) res[0] = res[1] = 0u;  // (always overwritten: the target is at most the sample size)
    grid_dependency_wait();
    allow_dependents();
    const int b = static_cast<int>(blockIdx.x);
    const int32_t len = seq_lens[b];
    const int32_t start = row_starts ? row_starts[b] : 0;
    if (len <= k || start < 0) return;  // CTA-uniform
    const int rem = start & 3;
    const int nv = (len + rem + 3) >> 2;
    if (nv <= min_nv) return;
    const float4* vbase = reinterpret_cast<const float4*>(scores + static_cast<int64_t>(b) * stride + (start - rem));
    const int v0 = static_cast<int>((4u - ((static_cast<uint32_t>(reinterpret_cast<uintptr_t>(vbase)) >> 4) & 3u)) & 3u);
    const uint64_t nq = static_cast<uint32_t>(nv - v0) >> 2;  // whole blocks, >= 255 (nv >= 1024)

    int j[kLoads];
    int4 v[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
        const uint64_t piece = static_cast<uint64_t>(u * (kThreads / 4) + (tid >> 2));
        j[u] = v0 + 4 * static_cast<int>((piece * nq) >> kLogPieces) + (tid & 3);  // < v0 + 4 * nq <= nv
        v[u] = load_bits(vbase + j[u]);
    }
    __syncthreads();  // the cleared histograms are visible
    uint32_t key[4 * kLoads];
    uint32_t valid = 0;
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
        const int32_t e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int p = 4 * j[u] - rem + c;
            key[4 * u + c] = bits_key(static_cast<uint32_t>(e[c]));
            if (p >= 0 && p < len) {
                valid |= 1u << (4 * u + c);
                red_add_shared(&h1[key[4 * u + c] >> kShift1], 1u);
            }
        }
    }
    __syncthreads();

    // Level 1: thread t holds bins kRun*t .. kRun*t + kRun - 1; the count
    // above its run comes from a warp-shuffle suffix sum and the warp totals.
    uint32_t bin[kRun];
#pragma unroll
    for (int q = 0; q < kRun / 4; ++q) {
        const uint4 w = reinterpret_cast<const uint4*>(h1)[(kRun / 4) * tid + q];
        bin[4 * q] = w.x, bin[4 * q + 1] = w.y, bin[4 * q + 2] = w.z, bin[4 * q + 3] = w.w;
    }
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < kRun; ++i) s += bin[i];
    uint32_t x = s;  // sum over this warp's lanes >= this lane
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, x, off);
        if (lane + off < 32u) x += y;
    }
    if (lane == 0) wtot[warp] = x;
    __syncthreads();
    uint32_t total = 0, above = x - s;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        total += wtot[w];
        above += w > warp ? wtot[w] : 0u;
    }
    // n_s = total sampled elements; the target is the sample's expected share
    // of the top k plus four standard deviations plus 2, at most n_s
    const float expect = static_cast<float>(k) * static_cast<float>(total) / static_cast<float>(len);
    const float tgt = fminf(ceilf(expect + 4.0f * sqrtf(expect) + 2.0f), static_cast<float>(total));
    const uint32_t target = max(static_cast<uint32_t>(tgt), 1u);
    if (above < target && above + s >= target) {  // exactly one thread: its run holds the target
        uint32_t acc = above;
#pragma unroll
        for (int i = kRun - 1; i >= 0; --i) {
            if (acc + bin[i] >= target) {
                res[0] = static_cast<uint32_t>(kRun * tid + i);
                res[1] = acc;
                break;
            }
            acc += bin[i];
        }
    }
    __syncthreads();
    const uint32_t b1 = res[0], above1 = res[1];

    // Level 2 over the sample elements in bin b1.
#pragma unroll
    for (int e = 0; e < 4 * kLoads; ++e)
        if (((valid >> e) & 1u) && (key[e] >> kShift1) == b1) red_add_shared(&h2[(key[e] >> kShift2) & 255u], 1u);
    __syncthreads();
    if (warp == 0) {  // lane l holds bins 8l .. 8l + 7
        const uint4 lo = reinterpret_cast<const uint4*>(h2)[2 * lane];
        const uint4 hi = reinterpret_cast<const uint4*>(h2)[2 * lane + 1];
        const uint32_t c[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
        uint32_t s2 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) s2 += c[i];
        uint32_t x2 = s2;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint32_t y = __shfl_down_sync(kFull, x2, off);
            if (lane + off < 32u) x2 += y;
        }
        const uint32_t target2 = target - above1;  // >= 1, at most the count of bin b1
        uint32_t acc = x2 - s2;
        const bool mine = acc < target2 && acc + s2 >= target2;
        if (__ballot_sync(kFull, mine) == 0u) {  // cannot happen; a bound of 0 sends the row to the exact path
            if (lane == 0) bounds[b] = 0u;
        } else if (mine) {
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (acc + c[i] >= target2) {
                    bounds[b] = (b1 << kShift1) | ((8u * lane + static_cast<uint32_t>(i)) << kShift2);
                    break;
                }
                acc += c[i];
            }
        }
    }
}

}  // namespace

cudaError_t launch(const Params& p, uint32_t* bounds, int min_nv, cudaStream_t stream) {
    return launch_pdl(topk_bound_kernel, p.batch, kThreads, 0, stream, p.scores, p.score_stride, p.row_starts,
                      p.seq_lens, p.k, static_cast<int32_t>(min_nv), bounds);
}

}  // namespace bound
}  // namespace topk_impl
