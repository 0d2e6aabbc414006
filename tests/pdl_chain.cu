// Test-only kernels that sit before and after the library's launches on a
// stream, to check its programmatic dependent launch (PDL) behaviour against
// the hazards the "#26788 [JIT Kernel] DeepSeek-V4 DSA indexer" page's review
// notes raise (a producer that lets its dependents start before it has
// written its output; a consumer that starts early).
//
//  * pdl_produce: copies `n` floats src -> dst after a bounded delay. With
//    `trigger` set it executes griddepcontrol.launch_dependents first, so a
//    kernel launched after it with the PDL attribute may be scheduled at once;
//    that kernel must not read dst before griddepcontrol.wait returns.
//  * pdl_consume: launched with the PDL attribute; waits on the grid
//    dependency, then copies `n` ints src -> dst (the library's output).
//
// Every loop is bounded; nothing here waits on a flag.

#include <cuda_runtime.h>

#include <cstdint>

namespace {

__global__ void producer_kernel(const float* src, float* dst, long long n, long long delay_cycles, int trigger) {
    if (trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long t0 = clock64();
    while (clock64() - t0 < delay_cycles) {
    }
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

__global__ void consumer_kernel(const int32_t* src, int32_t* dst, long long n) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<long long>(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

}  // namespace

extern "C" int pdl_produce(const float* src, float* dst, long long n, long long delay_cycles, int trigger,
                           void* stream) {
    producer_kernel<<<148, 256, 0, static_cast<cudaStream_t>(stream)>>>(src, dst, n, delay_cycles, trigger);
    return static_cast<int>(cudaGetLastError());
}

extern "C" int pdl_consume(const int32_t* src, int32_t* dst, long long n, void* stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(148, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return static_cast<int>(cudaLaunchKernelEx(&cfg, consumer_kernel, src, dst, n));
}
