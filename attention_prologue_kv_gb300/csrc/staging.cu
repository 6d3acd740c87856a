// Host staging for kv_rmsnorm_rope_cache_staged without copy-engine
// operations: a kernel reads the step's packed inputs straight from pinned
// (device-mapped) host memory into the device staging buffer, and a one-thread
// kernel writes the status word back to pinned host memory. Both are launched
// with programmatic dependent launch around the KV kernel, so a step is three
// chained kernels instead of DMA-kernel-DMA.
//
// Ordering: every kernel here calls pdl_wait() before touching memory, so the
// copy of step k+1 cannot overwrite the staging buffer while step k's KV
// kernel still reads it, and the status write sees the KV kernel's result.
#include "kvr_internal.cuh"

namespace kvr {

__global__ void __launch_bounds__(256) stage_in_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                       int64_t n16) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) dst[i] = src[i];
}

__global__ void status_out_kernel(volatile int32_t* host_status, const int32_t* dev_status) {
    pdl_wait();
    pdl_launch_dependents();
    *host_status = *reinterpret_cast<const volatile int32_t*>(dev_status);
}

cudaError_t launch_stage_in(void* dst, const void* src, int64_t bytes, cudaStream_t s) {
    const int64_t n16 = bytes / 16;
    const int64_t cap = int64_t(sm_count_current_device()) * 2;
    int64_t grid = (n16 + 255) / 256;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch_pdl(stage_in_kernel, dim3(unsigned(grid)), dim3(256), size_t(0), s, static_cast<uint4*>(dst),
                      static_cast<const uint4*>(src), n16);
}

cudaError_t launch_status_out(int32_t* host_status, const int32_t* dev_status, cudaStream_t s) {
    return launch_pdl(status_out_kernel, dim3(1), dim3(1), size_t(0), s,
                      static_cast<volatile int32_t*>(host_status), dev_status);
}

}  // namespace kvr
