// Sparse-attention indexer top-k + output transform for GB300 (sm_103a): the
// plan kernel, the host-side launch plan and the C ABI declared in
// include/topk.h. The selection kernels live in topk_select.cuh, compiled
// for 512 threads per row (topk_select512.cu) and 256 threads per row
// (topk_select256.cu); topk_common.cuh holds what the translation units
// share. The indexer-logits kernel and its entry point live in
// topk_logits.cu.
//
// The plan -> transform split follows the "#26788 [JIT Kernel] DeepSeek-V4 DSA
// indexer: faster top-k + page-table transform (runtime k <= 2048)" page
// ("Implementation breakdown": a plan kernel whose metadata the transform
// dispatches on). Every kernel is launched with programmatic dependent launch
// and waits (griddepcontrol.wait) before touching global memory.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "topk.h"
#include "topk_common.cuh"

using std::max;
using std::min;

namespace topk_impl {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kBandTrivial = 32;              // plan bands: 0..31 by length, then these two
constexpr int kBandCluster = 33;
constexpr int kBands = 34;


// Workspace: the plan header, order[batch] and cluster_rows[batch].
size_t workspace_bytes_for(int32_t batch) {
    if (batch < 0) return 0;
    size_t bytes = sizeof(PlanHeader) + 2 * sizeof(int32_t) * static_cast<size_t>(batch);
    return (bytes + 255) / 256 * 256;
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
            hdr->exact_rows = 0;
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
    int max_clusters = 0;  // co-resident clusters of the cluster kernel (one CTA per SM)
    int sms = 0;           // streaming multiprocessors
};

constexpr int kMaxDevices = 64;
DeviceState g_devices[kMaxDevices];
std::mutex g_mutex;

cudaError_t device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& st = g_devices[dev];
    if (!st.ready) {
        int mc = 0;
        e = t512::prepare(&mc);
        if (e == cudaSuccess) e = t256::prepare();
        if (e != cudaSuccess) return e;
        st.max_clusters = mc;
        e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        st.ready = true;
    }
    *out = &st;
    return cudaSuccess;
}

bool valid_k(int32_t k) { return k >= 1 && k <= TOPK_MAX_K; }

// Kernels one transform of `batch` rows launches: a batch whose every row can
// have a cluster of its own runs in the cluster kernel alone (its cluster rows
// split, the others on one CTA each); a larger batch of at most
// kClusterMaxBatch rows adds the cluster kernel to the rows kernel; above that
// the rows kernel alone.
int transform_launches(const DeviceState& ds, int32_t batch) {
    if (batch <= 0) return 0;
    if (batch <= kClusterMaxBatch && batch <= ds.max_clusters) return 1;
    return batch <= kClusterMaxBatch ? 2 : 1;
}

// The launch plan of a transform:
//   batch <= kClusterMaxBatch and <= the co-resident clusters: the cluster
//     kernel alone (512 threads per CTA);
//   batch <= SMs: the 512-thread rows kernel, one CTA per SM (plus the
//     cluster kernel for the long rows of batches up to kClusterMaxBatch);
//   larger batches: the 256-thread rows kernel, four CTAs per SM.
template <bool kPaged>
int launch_transform(const Params& prm, cudaStream_t stream) {
    DeviceState* ds = nullptr;
    if (device_state(&ds) != cudaSuccess) return TOPK_ERR_CUDA;
    const int B = prm.batch;
    if (B <= kClusterMaxBatch && B <= ds->max_clusters)
        return t512::launch_cluster(kPaged, B, 1, prm, stream) == cudaSuccess ? TOPK_OK : TOPK_ERR_CUDA;
    const cudaError_t le = B <= ds->sms ? t512::launch_rows(kPaged, true, prm, stream)
                                        : t256::launch_rows(kPaged, prm, stream);
    if (le != cudaSuccess) return TOPK_ERR_CUDA;
    if (B <= kClusterMaxBatch &&
        t512::launch_cluster(kPaged, min(B, ds->max_clusters), 0, prm, stream) != cudaSuccess)
        return TOPK_ERR_CUDA;
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
    p.out_stride = k;
    p.hdr = static_cast<PlanHeader*>(workspace);
    p.order = reinterpret_cast<const int32_t*>(static_cast<uint8_t*>(workspace) + sizeof(PlanHeader));
    p.cluster_rows = p.order + batch;
    return p;
}
}  // namespace
}  // namespace topk_impl

using namespace topk_impl;

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

int topk_transform_ragged_swa(const float* scores, int64_t score_stride, const int32_t* row_starts,
                              const int32_t* seq_lens, const int32_t* out_offsets, int32_t batch, int32_t k,
                              void* workspace, size_t workspace_bytes, const int32_t* positions,
                              int32_t window_size, const int32_t* swa_offsets, int32_t out_width, int32_t* out,
                              int32_t* out_raw, uint32_t flags, topk_stream_t stream) {
    const int st = common_checks(scores, score_stride, seq_lens, batch, k, workspace, workspace_bytes, out, flags);
    if (st != TOPK_OK) return st;
    if (window_size < 0 || window_size > TOPK_MAX_SWA_WINDOW) return TOPK_ERR_ARG;
    if (static_cast<int64_t>(out_width) < static_cast<int64_t>(k) + window_size) return TOPK_ERR_ARG;
    if (batch > 0 && (out_offsets == nullptr || positions == nullptr)) return TOPK_ERR_ARG;
    if (batch == 0) return TOPK_OK;
    Params p = make_params(scores, score_stride, row_starts, seq_lens, batch, k, workspace, out, out_raw, flags);
    p.out_offsets = out_offsets;
    p.out_stride = out_width;
    p.positions = positions;
    p.swa_window = window_size;
    p.swa_offsets = swa_offsets;
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

int topk_transform_launches(int32_t batch) {
    if (batch <= 0) return 0;
    DeviceState* ds = nullptr;
    if (device_state(&ds) != cudaSuccess) return -1;
    return transform_launches(*ds, batch);
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
