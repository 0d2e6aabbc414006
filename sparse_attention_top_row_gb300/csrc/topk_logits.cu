// The indexer-logits producer upstream of the top-k, on the 5th-generation
// tensor cores of sm_103a (tcgen05 MMAs with TMEM accumulators, operands
// staged by TMA):
//
//   logits[t][s] = kv_scale[s] * sum_h w[t][h] * max(0, q[t][h] . kv[s])
//   for ks[t] <= s < ke[t]
//
// with q [n_q, 64, 128] and kv [n_kv, 128] FP8 E4M3, w [n_q, 64] and
// kv_scale [n_kv] fp32. This is the reading of the FP8 MQA-logits producer
// that the PR #35175 page (PR body: the contiguous-KV indexer writes logit
// columns at absolute positions of the batch-flattened KV) and the PR #36684
// page ("Key source snippets", server_args.py: the v2 path needs tcgen05 and
// TMEM) put upstream of the top-k; row t of the result is the RAGGED
// transform's window at row_start = ks[t], seq_len = ke[t] - ks[t].
//
// Mapping. A work unit is a group of kGroup = 4 consecutive queries and a
// contiguous share of the group's key tiles (the host splits each group into
// `parts` shares so that the units fill the persistent CTAs, one per SM,
// evenly). The unit's 4 x 64 head vectors (256 rows of 128 bytes) are the
// MMA's B operand, loaded once per unit (double-buffered: the next unit's
// while this one's keys stream); the keys stream through a ring of kStages
// shared-memory stages, 128 keys (16 KB) a stage, as the A operand. One tile
// D = KV_tile . Q^T has M = 128 keys (TMEM lanes), N = 256 (query, head)
// columns and K = 128 (four kind::f8f6f4 MMAs of K = 32), so each epilogue
// thread owns one key and finds all 64 heads of a query in its own TMEM
// lane: the head sum needs no exchange between threads. Two accumulators
// (2 x 256 TMEM columns) let the MMAs of tile j + 1 run while tile j is read
// out. Shared memory (about 163 KB) keeps one CTA per SM, so the CTA's
// 512-column TMEM allocation never waits.
//
// Warp roles (10 warps): one thread of warp 0 walks the CTA's units, hands
// each to the others as a record in shared memory and issues the TMA loads
// (query tile, head weights, key tiles); warp 1
// owns the TMEM allocation and one of its threads issues the MMAs (a single
// thread issuing both was the bottleneck: each step of its loop waits);
// warps 2..9 read the accumulators out. A warp reaches TMEM lanes
// 32 * (warp % 4) .. + 31: warps 2..5 take the even tiles (accumulator 0),
// warps 6..9 the odd ones (accumulator 1), all four queries each, in two
// 128-column loads; the accumulator goes back to the MMAs once the second is
// in. On every SM sub-partition one warp of each group runs, so one computes
// while the other waits for its tile.
//
// Every wait on an mbarrier is bounded: past about a second the kernel ORs
// TOPK_DEVICE_FLAG_TIMEOUT into the caller's flag word and goes on, so no
// barrier is left unmatched and the TMEM allocation is always released.

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "topk.h"
#include "topk_common.cuh"

namespace topk_impl {
namespace {

constexpr int kHeads = TOPK_INDEXER_HEADS;  // 64
constexpr int kDim = TOPK_INDEXER_DIM;      // 128 (bytes of one FP8 row)
constexpr int kGroup = 4;                   // queries per CTA
constexpr int kN = kGroup * kHeads;         // 256: MMA N (query, head) columns
constexpr int kM = 128;                     // keys per tile: MMA M, TMEM lanes
constexpr int kMmaK = 32;                   // K of one kind::f8f6f4 MMA
constexpr int kStages = 6;                  // key tiles in flight
constexpr int kEpiWarps = 8;
constexpr int kThreadsL = 32 * (2 + kEpiWarps);
constexpr uint32_t kTmemCols = 2 * kN;      // two accumulators
constexpr uint32_t kQBytes = kN * kDim;     // 32 KB
constexpr uint32_t kTileBytes = kM * kDim;  // 16 KB
constexpr uint32_t kWBytes = kN * 4;       // a group's head weights, fp32
constexpr uint32_t kKvOff = 2 * kQBytes;   // two query tiles (this unit's and the next)
constexpr uint32_t kWOff = kKvOff + kStages * kTileBytes;
constexpr uint32_t kRecOff = kWOff + 2 * kWBytes;  // two unit records (UnitRec)
constexpr uint32_t kBarOff = kRecOff + 2 * 64;
constexpr int kBars = 2 * kStages + 2 + 2 + 2 + 2;  // full, empty, q full, q free, tmem full, tmem empty
constexpr uint32_t kSlotOff = kBarOff + kBars * 8;
constexpr size_t kSmemLogits = kSlotOff + 16 + 1024;  // + alignment slack (tiles on 1024 B)
static_assert(kSmemLogits > 114 * 1024, "one CTA per SM (its TMEM allocation is the whole TMEM)");
static_assert(kSmemLogits <= 227 * 1024, "shared memory per CTA");
constexpr long long kLogitsWaitCycles = 1ll << 31;  // about a second

// Instruction descriptor of tcgen05.mma kind::f8f6f4: D fp32 (bits 4-5 = 1),
// A and B E4M3 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(kN >> 3) << 17) | (static_cast<uint32_t>(kM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile of 128-byte rows in the
// 128-byte swizzle (what a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes):
// start address >> 4 (bits 0-13), leading offset unused for this layout (1),
// stride offset 1024 B between 8-row groups (bits 32-45), version 1 (bits
// 46-47), base offset 0 (tiles on 1024-byte boundaries), layout 2 = 128-byte
// swizzle (bits 61-63). Stepping K by 32 bytes inside the swizzled row adds
// 2 to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (static_cast<uint64_t>(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ uint32_t cvta_smem(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool bar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}
// Waits for the phase of `bar` with this parity to complete, at most
// kLogitsWaitCycles; past that it flags the timeout and returns.
__device__ __forceinline__ void bar_wait(uint32_t bar, uint32_t parity, uint32_t* flags) {
    if (bar_try_wait(bar, parity)) return;
    const long long t0 = clock64();
    while (!bar_try_wait(bar, parity)) {
        if (clock64() - t0 > kLogitsWaitCycles) {
            atomicOr(flags, TOPK_DEVICE_FLAG_TIMEOUT);
            return;
        }
    }
}

// 2-D TMA tile load (x: byte column, a multiple of 16; y: row) completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D (TMEM) = A . B^T (+ D when acc): A, B from shared memory by descriptor.
__device__ __forceinline__ void mma_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}
// `bar` gets one arrival once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// This warp's 32 TMEM lanes, 128 consecutive fp32 columns from `taddr`
// (thread i: lane base + i), waited for inside the same statement so that
// no use of the registers can be scheduled before the data are in.
__device__ __forceinline__ void tmem_load128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
        "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
        "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
        "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127"
        "}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        :
          "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
          "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
          "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
          "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
          "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
          "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]),
          "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]),
          "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]),
          "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
}

// Four consecutive fp32 words of shared memory (a broadcast when every lane
// reads the same address).
__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}

struct LogitsParams {
    const float* kv_scale;
    const float* weights;
    const int32_t* ks;
    const int32_t* ke;
    float* logits;
    int64_t stride;
    int32_t n_q;
    int32_t n_kv;
    int32_t parts;  // work units per query group, each a contiguous share of the group's key tiles
    int32_t units;  // query groups x parts
    uint32_t* flags;
};

// One work unit: queries t0 .. t0 + 3 over key tiles kbase + 128 j, j < n_tiles.
struct Unit {
    int t0, kbase, n_tiles;
};

// A unit as the producer hands it to the MMA issuer and the readout warps
// (in shared memory, next to the unit's query tile): n_tiles == 0 ends the
// sequence; lo/hi: each query's window clamped to [0, n_kv) (empty past n_q).
struct UnitRec {
    int t0, kbase, n_tiles, pad;
    int lo[kGroup], hi[kGroup];
};
static_assert(sizeof(UnitRec) <= 64, "unit record");

// Unit u: query group u / parts, share u % parts of the group's key span
// (the union of its queries' windows, from the tile holding its first key).
__device__ __forceinline__ Unit unit_of(const LogitsParams& p, int u) {
    const int group = u / p.parts, part = u % p.parts;
    const int t0 = group * kGroup;
    int lo = INT_MAX, hi = 0;
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
        const int t = t0 + i;
        if (t < p.n_q) {
            const int a = max(__ldg(p.ks + t), 0), b = min(__ldg(p.ke + t), p.n_kv);
            if (a < b) {
                lo = min(lo, a);
                hi = max(hi, b);
            }
        }
    }
    const int kbase0 = lo & ~(kM - 1);
    const int group_tiles = lo < hi ? (hi - kbase0 + kM - 1) / kM : 0;
    const int per_part = (group_tiles + p.parts - 1) / p.parts;
    return Unit{t0, kbase0 + part * per_part * kM, max(0, min(per_part, group_tiles - part * per_part))};
}

// Persistent: CTA c takes units c, c + gridDim.x, ... in turn (every role
// walks the same sequence and skips the same empty units). Tiles are counted
// over the CTA's whole sequence, so the stage ring and the two accumulators
// run on across units; the query tile and head weights are double-buffered
// by unit, the next unit's loaded while this one's keys stream.
__global__ void __launch_bounds__(kThreadsL, 1)
    topk_indexer_logits_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tkv,
                               const __grid_constant__ LogitsParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = cvta_smem(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* const sm = smem_raw + (base - raw);
    const uint32_t bars = base + kBarOff;
    auto full = [&](int s) { return bars + 8u * static_cast<uint32_t>(s); };
    auto empty = [&](int s) { return bars + 8u * static_cast<uint32_t>(kStages + s); };
    auto qfull = [&](int q) { return bars + 8u * static_cast<uint32_t>(2 * kStages + q); };
    auto qfree = [&](int q) { return bars + 8u * static_cast<uint32_t>(2 * kStages + 2 + q); };
    auto tfull = [&](int b) { return bars + 8u * static_cast<uint32_t>(2 * kStages + 4 + b); };
    auto tempty = [&](int b) { return bars + 8u * static_cast<uint32_t>(2 * kStages + 6 + b); };
    auto qtile = [&](int q) { return base + static_cast<uint32_t>(q) * kQBytes; };
    auto wtile = [&](int q) { return base + kWOff + static_cast<uint32_t>(q) * kWBytes; };
    uint32_t* const slot = reinterpret_cast<uint32_t*>(sm + kSlotOff);

    const int warp = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31u);
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            bar_init(full(s), 1);
            bar_init(empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(qfull(b), 1);
            bar_init(qfree(b), kEpiWarps);
            bar_init(tfull(b), 1);
            bar_init(tempty(b), kEpiWarps / 2);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        __syncwarp();
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(cvta_smem(slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const int u0 = static_cast<int>(blockIdx.x), du = static_cast<int>(gridDim.x);

    if (warp == 0) {
        if (lane == 0) {  // TMA producer: per unit its record, query tile and weights, then its key tiles
            int g = 0, nu = 0;
            for (int u = u0;; u += du) {
                const Unit un = u < p.units ? unit_of(p, u) : Unit{0, 0, 0};
                if (u < p.units && un.n_tiles == 0) continue;
                const int q = nu & 1;
                if (nu >= 2) bar_wait(qfree(q), static_cast<uint32_t>((nu >> 1) & 1) ^ 1u, p.flags);
                UnitRec* const rec = reinterpret_cast<UnitRec*>(sm + kRecOff) + q;
                rec->t0 = un.t0;
                rec->kbase = un.kbase;
                rec->n_tiles = un.n_tiles;
#pragma unroll
                for (int i = 0; i < kGroup; ++i) {
                    const int t = un.t0 + i;
                    const bool v = un.n_tiles > 0 && t < p.n_q;
                    rec->lo[i] = v ? max(__ldg(p.ks + t), 0) : 0;
                    rec->hi[i] = v ? min(__ldg(p.ke + t), p.n_kv) : 0;
                }
                if (un.n_tiles == 0) {  // the end: the record alone (the arrival publishes it)
                    bar_arrive(qfull(q));
                    break;
                }
                const uint32_t wbytes = static_cast<uint32_t>(min(kGroup, p.n_q - un.t0)) * (kHeads * 4);
                bar_expect_tx(qfull(q), kQBytes + wbytes);  // (its arrival publishes the record)
                tma_load_2d(qtile(q), &tq, 0, un.t0 * kHeads, qfull(q));
                asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                                 wtile(q)),
                             "l"(p.weights + static_cast<int64_t>(un.t0) * kHeads), "r"(wbytes), "r"(qfull(q))
                             : "memory");
                for (int j = 0; j < un.n_tiles; ++j, ++g) {
                    const int s = g % kStages;
                    if (g >= kStages) bar_wait(empty(s), static_cast<uint32_t>((g / kStages) & 1) ^ 1u, p.flags);
                    bar_expect_tx(full(s), kTileBytes);
                    tma_load_2d(base + kKvOff + static_cast<uint32_t>(s) * kTileBytes, &tkv, 0, un.kbase + j * kM, full(s));
                }
                ++nu;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            int g = 0;
            for (int nu = 0;; ++nu) {
                const int q = nu & 1;
                bar_wait(qfull(q), static_cast<uint32_t>((nu >> 1) & 1), p.flags);
                const int n_tiles = reinterpret_cast<const volatile UnitRec*>(sm + kRecOff)[q].n_tiles;
                if (n_tiles == 0) break;
                const uint64_t bdesc = sw128_desc(qtile(q));
                for (int j = 0; j < n_tiles; ++j, ++g) {
                    const int s = g % kStages, b = g & 1;
                    bar_wait(full(s), static_cast<uint32_t>((g / kStages) & 1), p.flags);
                    if (g >= 2) bar_wait(tempty(b), static_cast<uint32_t>((g >> 1) & 1) ^ 1u, p.flags);
                    tc_fence_after();
                    const uint64_t adesc = sw128_desc(base + kKvOff + static_cast<uint32_t>(s) * kTileBytes);
                    const uint32_t d = tmem + static_cast<uint32_t>(b * kN);
#pragma unroll
                    for (int kk = 0; kk < kDim / kMmaK; ++kk)
                        mma_f8(d, adesc + static_cast<uint64_t>(2 * kk), bdesc + static_cast<uint64_t>(2 * kk),
                               kk > 0 ? 1u : 0u);
                    mma_commit(empty(s));
                    mma_commit(tfull(b));
                }
            }
            // the last tile's MMAs are complete before the TMEM is released
            if (g > 0) bar_wait(tfull((g - 1) & 1), static_cast<uint32_t>(((g - 1) >> 1) & 1), p.flags);
        }
        __syncwarp();
    } else {  // epilogue: one key per thread, the four queries of every other tile
        const int quarter = warp & 3;
        const int eg = (warp - 2) >> 2;  // epilogue group: tiles g with g % 2 == eg, accumulator eg
        const int row = quarter * 32 + lane;
        const uint32_t acc_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(eg * kN);
        int g = 0;
        for (int nu = 0;; ++nu) {
            const int q = nu & 1;
            bar_wait(qfull(q), static_cast<uint32_t>((nu >> 1) & 1), p.flags);  // the unit's record and weights
            __syncwarp();
            const UnitRec un = reinterpret_cast<const UnitRec*>(sm + kRecOff)[q];
            if (un.n_tiles == 0) break;
            const int* const lo_t = un.lo;
            const int* const hi_t = un.hi;
            float* const out0 = p.logits + static_cast<int64_t>(un.t0) * p.stride;
            const uint32_t w_addr = wtile(q);
            for (int j = 0; j < un.n_tiles; ++j, ++g) {
                if ((g & 1) != eg) continue;
                const int s = un.kbase + j * kM + row;
                const float scale = s < p.n_kv ? __ldg(p.kv_scale + s) : 0.0f;
                bar_wait(tfull(eg), static_cast<uint32_t>((g >> 1) & 1), p.flags);
                __syncwarp();  // the TMEM loads below are warp-collective
                tc_fence_after();
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t r[2 * kHeads];  // two queries, all heads, in one load
                    tmem_load128(acc_addr + static_cast<uint32_t>(half * 2 * kHeads), r);
                    if (half == 1) {  // the accumulator is in registers: hand it back to the MMAs
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) bar_arrive(tempty(eg));
                    }
                    // packed fp32 pairs, w * max(d, 0) two heads an instruction, both
                    // queries interleaved (four independent accumulator chains)
                    float2 acc[2][2] = {{make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)},
                                        {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)}};
#pragma unroll
                    for (int e = 0; e < kHeads; e += 4) {
#pragma unroll
                        for (int i = 0; i < 2; ++i) {
                            const int qi = 2 * half + i;
                            const float4 w4 = lds_f4(w_addr + static_cast<uint32_t>((qi * kHeads + e) * 4));
                            const uint32_t* d = r + i * kHeads + e;
                            // even heads: max(x, 0) (ALU pipe); odd heads: x + |x| = 2 max(x, 0),
                            // exactly, on the FMA pipe (their sums are halved at the end): the
                            // two pipes share the ReLUs
                            const float a1 = __uint_as_float(d[1]), a3 = __uint_as_float(d[3]);
                            const float2 x0 = make_float2(fmaxf(__uint_as_float(d[0]), 0.0f), a1 + fabsf(a1));
                            const float2 x1 = make_float2(fmaxf(__uint_as_float(d[2]), 0.0f), a3 + fabsf(a3));
                            acc[i][0] = __ffma2_rn(make_float2(w4.x, w4.y), x0, acc[i][0]);
                            acc[i][1] = __ffma2_rn(make_float2(w4.z, w4.w), x1, acc[i][1]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int qi = 2 * half + i;
                        if (s >= lo_t[qi] && s < hi_t[qi])
                            out0[static_cast<int64_t>(qi) * p.stride + s] =
                                ((acc[i][0].x + 0.5f * acc[i][0].y) + (acc[i][1].x + 0.5f * acc[i][1].y)) * scale;
                    }
                }
            }
            __syncwarp();  // this warp is done with the unit's record and weights (and its MMAs are done)
            if (lane == 0) bar_arrive(qfree(q));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    allow_dependents();
}

PFN_cuTensorMapEncodeTiled_v12000 encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A 2-D map over `rows` rows of 128 bytes, tiles of box_rows rows, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint32_t box_rows) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = encode_tiled();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDim)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kDim), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxDevicesL = 64;
bool g_logits_ready[kMaxDevicesL];
int g_logits_sms[kMaxDevicesL];
std::mutex g_logits_mutex;

// Work units per query group: the groups' key tiles split into `parts`
// contiguous shares so that the persistent CTAs (one per SM, each taking
// every SM-count-th unit) end together: the fewest parts (at most 16, and
// none shorter than about 8 tiles of the longest possible span) whose units
// fill the CTAs' last round to 97 %, else the fullest. (A unit costs one more
// 32 KB query tile, loaded while the previous unit's keys stream.)
int logits_parts(int groups, int n_kv) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesL) return 1;
    const int slots = max(g_logits_sms[dev], 1);
    const int max_parts = max(1, min(16, n_kv / (8 * kM)));
    int best = 1;
    double best_fill = 0.0;
    for (int parts = 1; parts <= max_parts; ++parts) {
        const double rounds = static_cast<double>(groups) * parts / slots;
        const double fill = rounds / std::ceil(rounds);
        if (fill >= 0.97) return parts;
        if (fill > best_fill) {
            best_fill = fill;
            best = parts;
        }
    }
    return best;
}

cudaError_t prepare_logits() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevicesL) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_logits_mutex);
    if (!g_logits_ready[dev]) {
        e = cudaFuncSetAttribute(topk_indexer_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(kSmemLogits));
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&g_logits_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_logits_ready[dev] = true;
    }
    return cudaSuccess;
}

}  // namespace
}  // namespace topk_impl

using namespace topk_impl;

extern "C" int topk_indexer_logits(const uint8_t* q, const uint8_t* kv, const float* kv_scale, const float* weights,
                                   const int32_t* ks, const int32_t* ke, int32_t n_q, int32_t n_kv, float* logits,
                                   int64_t logits_stride, uint32_t* device_flags, topk_stream_t stream) {
    if (n_q < 0 || n_kv < 0 || n_q > TOPK_INDEXER_MAX_QUERIES || n_kv > TOPK_INDEXER_MAX_KEYS || logits_stride < 0)
        return TOPK_ERR_ARG;
    if (n_q == 0 || n_kv == 0) return TOPK_OK;
    if (!q || !kv || !kv_scale || !weights || !ks || !ke || !logits || !device_flags) return TOPK_ERR_ARG;
    if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) | reinterpret_cast<uintptr_t>(weights)) &
         15u) != 0)
        return TOPK_ERR_ALIGN;
    if (prepare_logits() != cudaSuccess) return TOPK_ERR_CUDA;
    CUtensorMap tq, tkv;
    if (!make_map(&tq, q, static_cast<uint64_t>(n_q) * kHeads, kN) ||
        !make_map(&tkv, kv, static_cast<uint64_t>(n_kv), kM))
        return TOPK_ERR_CUDA;
    LogitsParams prm;
    prm.kv_scale = kv_scale;
    prm.weights = weights;
    prm.ks = ks;
    prm.ke = ke;
    prm.logits = logits;
    prm.stride = logits_stride;
    prm.n_q = n_q;
    prm.n_kv = n_kv;
    prm.flags = device_flags;
    const int groups = (n_q + kGroup - 1) / kGroup;
    prm.parts = logits_parts(groups, n_kv);
    prm.units = groups * prm.parts;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return TOPK_ERR_CUDA;
    const int grid = min(prm.units, max(g_logits_sms[dev], 1));  // one persistent CTA per SM
    const cudaError_t e = launch_pdl(topk_indexer_logits_kernel, grid, kThreadsL, kSmemLogits,
                                     reinterpret_cast<cudaStream_t>(stream), tq, tkv, prm);
    return e == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
}
