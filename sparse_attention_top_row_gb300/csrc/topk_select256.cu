// The 256-thread build of the selection kernels: the rows kernel for large
// batches (more rows than SMs), four CTAs of 256 threads per SM, so that four
// rows are in flight on every SM and one row's latency-bound finish overlaps
// the others' score streams.
#define TOPK_THREADS 256
#define TOPK_NS t256
#define TOPK_WITH_CLUSTER 0
#ifndef TOPK_CTAS_PER_SM
#define TOPK_CTAS_PER_SM 4
#endif
#ifndef TOPK_WARP_CAP
#define TOPK_WARP_CAP 576
#endif
#ifndef TOPK_PAGE_CACHE
#define TOPK_PAGE_CACHE 1024
#endif
#include "topk_select.cuh"

namespace topk_impl {
namespace t256 {

cudaError_t prepare() {
    cudaError_t e = cudaFuncSetAttribute(topk_rows_kernel<true, TOPK_CTAS_PER_SM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemRows));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(topk_rows_kernel<false, TOPK_CTAS_PER_SM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(kSmemRows));
}

cudaError_t launch_rows(bool paged, const Params& p, cudaStream_t stream) {
    return paged ? launch_pdl(topk_rows_kernel<true, TOPK_CTAS_PER_SM>, p.batch, kThreads, kSmemRows, stream, p)
                 : launch_pdl(topk_rows_kernel<false, TOPK_CTAS_PER_SM>, p.batch, kThreads, kSmemRows, stream, p);
}

}  // namespace t256
}  // namespace topk_impl
