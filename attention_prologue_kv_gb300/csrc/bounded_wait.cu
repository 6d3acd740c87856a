// Exercise of the bounded-wait path the pipeline kernels rely on: a warp
// waits on an mbarrier phase that can never complete (it expects bytes that
// no copy delivers), polling the way mbar_wait does, and gives up when the
// time limit passes or when another warp raises the abort flag. The kernel
// then records KVR_DEVERR_TIMEOUT and returns, leaving the context usable.
// No copy is in flight, so the CTA may exit with the phase pending.
//
// Also here: a late producer of device words, for checking that a kernel
// reads its inputs only after its dependency wait.
#include "kvr_internal.cuh"

namespace kvr {

__global__ void __launch_bounds__(64) bounded_wait_kernel(int32_t* status, uint64_t limit_ns, uint64_t abort_after_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        int ok = 1;
        if (threadIdx.x == 0) {
            mbar_arrive_expect_tx(&bar, 16);   // 16 bytes that will never arrive
            ok = 0;
            const uint64_t t0 = globaltimer_ns();
            for (;;) {
                __nanosleep(64);
                if (mbar_try_wait(&bar, 0)) {
                    ok = 1;
                    break;
                }
                if (abort_flag) break;
                if (globaltimer_ns() - t0 > limit_ns) break;
            }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        if (!ok && threadIdx.x == 0) atomicOr(status, KVR_DEVERR_TIMEOUT);
    } else if (threadIdx.x == 32 && abort_after_ns > 0) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < abort_after_ns) __nanosleep(256);
        abort_flag = 1;
    }
}

cudaError_t launch_bounded_wait(int32_t* status, int64_t limit_ns, int64_t abort_after_ns, cudaStream_t s) {
    bounded_wait_kernel<<<1, 64, 0, s>>>(status, uint64_t(limit_ns), uint64_t(abort_after_ns));
    return cudaGetLastError();
}

// One warp: waits for its own predecessor, lets the next launch start at
// once, spins (bounded by delay_ns) and only then copies src[0..count) to
// dst, so the dependent grid runs its pre-wait code while the old values are
// still there.
__global__ void __launch_bounds__(32) store_after_delay_kernel(int64_t* dst, const int64_t* src, int64_t count,
                                                               uint64_t delay_ns) {
    pdl_wait();
    pdl_launch_dependents();
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < delay_ns) __nanosleep(256);
    for (int64_t i = threadIdx.x; i < count; i += 32) dst[i] = src[i];
}

cudaError_t launch_store_after_delay(int64_t* dst, const int64_t* src, int64_t count, int64_t delay_ns,
                                     cudaStream_t s) {
    return launch_pdl(store_after_delay_kernel, dim3(1), dim3(32), 0, s, dst, src, count, uint64_t(delay_ns));
}

}  // namespace kvr
