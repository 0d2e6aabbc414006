// Shared by the selection builds and the plan/host code of the indexer top-k
// library (topk.cu): the plan workspace header, the launch parameters, the
// cluster-path limits, warp helpers, the programmatic-dependent-launch
// helpers, and the entry points of the two builds of the selection kernels
// (512 threads per row; 256 threads per row for large batches).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "topk.h"

namespace topk_impl {

constexpr int32_t kClusterFloor = 32768;  // rows longer than this may use the cluster path
constexpr int32_t kClusterMaxBatch = 64;  // ... when the batch is at most this
constexpr int kClusterSize = 4;           // CTAs per long row on the cluster path
constexpr uint32_t kFull = 0xFFFFFFFFu;

struct alignas(64) PlanHeader {
    uint32_t magic;
    int32_t batch;
    int32_t k;
    int32_t n_order;      // rows listed in order[] (all rows not on the cluster path)
    int32_t n_cluster;    // rows listed in cluster_rows[]
    uint32_t error_rows;  // device-side data errors
    uint32_t flags;       // TOPK_DEVICE_FLAG_*
    uint32_t exact_rows;  // rows (slices) the transform finished on the exact path (statistics)
    int32_t reserved[8];
};
static_assert(sizeof(PlanHeader) == 64, "header layout");
constexpr uint32_t kPlanMagic = 0x6E616C50u;

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
    int32_t out_stride;            // elements between output rows (k, or the SWA combine's width)
    const int32_t* positions;      // SWA combine: each row's query position, or null (no combine)
    int32_t swa_window;            // SWA combine: the window's size in tokens
    const int32_t* swa_offsets;    // SWA combine: each row's window offset, or null (0)
};

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

// Programmatic dependent launch. Every kernel here is launched so that it may
// be scheduled while the previous kernel on the stream is still running, and
// reads or writes no global memory before grid_dependency_wait(), which
// returns once the previous kernels have completed and their writes are
// visible: stream order is kept, only the launch latency is hidden.
// allow_dependents() lets the next kernel on the stream be scheduled early
// under the same rule (a kernel launched without the attribute is unaffected).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

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

// The 512-thread build (topk_select512.cu): the rows kernel (one or two CTAs
// per SM) and the cluster kernel. prepare() sets the kernels' shared-memory
// limits on the current device and returns how many clusters fit at once.
namespace t512 {
cudaError_t prepare(int* max_clusters);
cudaError_t launch_rows(bool paged, bool one_per_sm, const Params& p, cudaStream_t stream);
cudaError_t launch_cluster(bool paged, int clusters, int all_rows, const Params& p, cudaStream_t stream);
}  // namespace t512

// The 256-thread build (topk_select256.cu): the rows kernel, four CTAs per SM.
namespace t256 {
cudaError_t prepare();
cudaError_t launch_rows(bool paged, const Params& p, cudaStream_t stream);
}  // namespace t256

}  // namespace topk_impl
