// The 512-thread build of the selection kernels: the rows kernel for batches
// up to one row per SM (one CTA of 512 threads per SM) and the
// thread-block-cluster kernel (few long rows, and whole small batches).
#define TOPK_THREADS 512
#define TOPK_NS t512
#define TOPK_WITH_CLUSTER 1
#include "topk_select.cuh"

namespace topk_impl {
namespace t512 {
namespace {

// Shared-memory limits of one build's kernels and the co-resident cluster
// count of its cluster kernel.
template <bool kPaged>
cudaError_t prepare_mode(int& max_clusters) {
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<kPaged, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemRows));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_cluster_kernel<kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kSmemCluster));
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
    if (cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel<kPaged>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();  // the query is advisory: fall back to a conservative count
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = sms > 2 * kClusterSize ? sms / (2 * kClusterSize) : 1;
    }
    max_clusters = max_clusters == 0 ? n : min(max_clusters, n);
    return cudaSuccess;
}

}  // namespace

cudaError_t prepare(int* max_clusters) {
    int mc = 0;
    cudaError_t e = prepare_mode<true>(mc);
    if (e == cudaSuccess) e = prepare_mode<false>(mc);
    *max_clusters = mc > 0 ? mc : 1;
    return e;
}

cudaError_t launch_rows(bool paged, bool one_per_sm, const Params& p, cudaStream_t stream) {
    (void)one_per_sm;  // this build runs one CTA of 512 threads per SM
    return paged ? launch_pdl(topk_rows_kernel<true, 1>, p.batch, kThreads, kSmemRows, stream, p)
                 : launch_pdl(topk_rows_kernel<false, 1>, p.batch, kThreads, kSmemRows, stream, p);
}

cudaError_t launch_cluster(bool paged, int clusters, int all_rows, const Params& p, cudaStream_t stream) {
    return paged ? launch_pdl(topk_cluster_kernel<true>, kClusterSize * clusters, kThreads, kSmemCluster, stream, p,
                              all_rows)
                 : launch_pdl(topk_cluster_kernel<false>, kClusterSize * clusters, kThreads, kSmemCluster, stream, p,
                              all_rows);
}

}  // namespace t512
}  // namespace topk_impl
