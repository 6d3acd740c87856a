// Internal declarations and device helpers shared by the libkvr.so kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvr.h"

namespace kvr {

// ---------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------

// Output element kinds. OUT16 is the 16-bit input type itself (bf16 or f16).
enum OutKind : int { OUT16 = 0, OUT_I8 = 1, OUT_E4M3 = 2, OUT_E5M2 = 3 };

struct BF16 {
    static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
    static __device__ __forceinline__ float hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
    static __device__ __forceinline__ float one(uint16_t u) { return __uint_as_float(uint32_t(u) << 16); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ uint16_t one_out(float v) {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        return *reinterpret_cast<uint16_t*>(&h);
    }
};

struct F16 {
    static __device__ __forceinline__ float lo(uint32_t u) { return __half2float(__ushort_as_half(uint16_t(u & 0xFFFFu))); }
    static __device__ __forceinline__ float hi(uint32_t u) { return __half2float(__ushort_as_half(uint16_t(u >> 16))); }
    static __device__ __forceinline__ float one(uint16_t u) { return __half2float(__ushort_as_half(u)); }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ uint16_t one_out(float v) { return __half_as_ushort(__float2half_rn(v)); }
};

// Two floats -> two 8-bit codes packed in 16 bits (lo in the low byte).
template <int K>
__device__ __forceinline__ uint32_t enc8x2(float lo, float hi) {
    if constexpr (K == OUT_E4M3) {
        uint16_t r;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
        return r;
    } else if constexpr (K == OUT_E5M2) {
        uint16_t r;
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
        return r;
    } else {  // OUT_I8: round half to even, clamp to [-128, 127]
        int a = min(max(__float2int_rn(lo), -128), 127);
        int b = min(max(__float2int_rn(hi), -128), 127);
        return (uint32_t(a) & 0xFFu) | ((uint32_t(b) & 0xFFu) << 8);
    }
}

// Runtime-kind variant for the small k-cache part.
__device__ __forceinline__ uint32_t enc8x2_rt(int kind, float lo, float hi) {
    if (kind == OUT_E4M3) return enc8x2<OUT_E4M3>(lo, hi);
    if (kind == OUT_E5M2) return enc8x2<OUT_E5M2>(lo, hi);
    return enc8x2<OUT_I8>(lo, hi);
}

// ---------------------------------------------------------------------------
// Memory helpers
// ---------------------------------------------------------------------------

// Streaming read-only loads: inputs are read once, keep them out of L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
    uint32_t r;
    asm("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ uint16_t ld_stream_u16(const void* p) {
    uint16_t r;
    asm("ld.global.nc.L1::no_allocate.b16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}
__device__ __forceinline__ int64_t ld_stream_s64(const int64_t* p) {
    int64_t r;
    asm("ld.global.nc.L1::no_allocate.s64 %0, [%1];" : "=l"(r) : "l"(p));
    return r;
}

// ---------------------------------------------------------------------------
// mbarrier, bulk async copy (TMA engine), programmatic dependent launch
// ---------------------------------------------------------------------------

// Longest any wait in these kernels may take before it gives up, raises
// KVR_DEVERR_TIMEOUT and lets the CTA drain and exit (a correct run waits
// for microseconds).
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// try_wait may suspend the thread until the phase completes or, at most,
// the hinted number of nanoseconds pass: waiting warps issue few instructions.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000)
        : "memory");
    return ok != 0;
}
// Wait until the phase with parity `parity` of `bar` has completed. Returns
// false if *abort becomes non-zero (when abort is given) or WAIT_LIMIT_NS passes.
// sleep_ns > 0 backs off between polls (for a lone waiter during a long copy,
// so that it does not take issue slots from warps that are computing).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                          unsigned sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (sleep_ns) __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if (abort != nullptr && *abort) return false;
        if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) return false;
    }
}
// mbar_wait for a whole warp: lane 0 waits, every lane gets its outcome, so
// the warp never diverges on a wait that gives up.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, const volatile int* abort,
                                               unsigned sleep_ns = 0) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, sleep_ns) ? 1 : 0;
    return __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
}

// One bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// An L2 access policy that marks lines for early eviction (data read once),
// and the bulk copy that carries it. KVR_BULK_EVICT_FIRST=0 uses the default
// policy instead.
#ifndef KVR_BULK_EVICT_FIRST
#define KVR_BULK_EVICT_FIRST 1
#endif
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
#if KVR_BULK_EVICT_FIRST
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
#else
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
#endif
    return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// L2 prefetch hints. They move nothing into registers or shared memory and
// L2 is the point of coherence, so they may run before pdl_wait(): a write
// by the preceding grid to a prefetched line still lands in L2 and is what
// the later loads see. Bulk form: 16-byte aligned address, size a multiple of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// Programmatic dependent launch: wait for the preceding grid's results (a
// no-op without the launch attribute), then let the next grid launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Parameter blocks (passed by value to the kernels)
// ---------------------------------------------------------------------------

struct KvParams {
    const void* kv;
    const void* gamma;
    const void* cos;
    const void* sin;
    const int64_t* index;
    void* ckv;
    void* kc;
    const float* ckv_scale;
    const float* k_scale;
    int32_t* status;
    int64_t T;           // token rows
    int64_t Skv;
    int64_t kv_stride;   // elements between consecutive kv rows
    int64_t d0, d1;      // cache leading dims
    int64_t nblk;        // PA_BLK_BSND: index entries per sequence
    int Dv, Dk;
    // bulk (TMA) pipeline layout, set by the host for the pipelined kernel
    int R;               // rows per tile
    int S;               // pipeline stages
    int kv_contig;       // kv rows are dense: one bulk copy per tile
    int idx_bulk;        // the index tile is bulk-copied (else read from global)
    uint32_t stage_bytes, off_cos, off_sin, off_idx, off_consts, off_stages;
    int mode;            // kvr_cache_mode
    int k_kind;          // OutKind of the k cache
    int ckv_scale_per_ch, k_scale_per_ch;
    int params_ready;    // gamma/scales may be read before the dependency wait
    float eps, inv_dv, alpha;
};

struct QsaParams {
    const void* raw;
    void* block_keys;
    const int64_t* key_length;
    const void* cos;
    const void* sin;
    const void* w;
    const void* past_raw;
    const void* past_rope;
    void* next_raw;
    void* next_rope;
    const void* past_bk;  // concat-output form: past block keys [N, Bp, Di], else NULL
    int32_t* status;
    int64_t N, L, Bcap, kbs;
    int64_t nbmax;       // CTAs per sequence for block keys = ceil(L / kbs)
    int64_t Bp;          // rows of past_bk per sequence
    int64_t ncopy;       // CTAs per sequence copying past rows (0 unless past_bk)
    int copy_rows;       // past rows per copy CTA
    int copy_vec;        // the copy may use 16-byte accesses
    int key_length_per_seq;
    int Di, Dr;
    int rope_first;      // rotate channels [0, Dr) instead of [Di-Dr, Di)
    int rope_half;       // rotate-half pairs (x[i], x[i+Dr/2]) instead of (x[2i], x[2i+1])
    int params_ready;    // key_length, tables and weight may be read before the dependency wait
    int key_length_late; // no early key_length hint (the preceding kernel writes it)
    float eps, inv_di, inv_kbs;
};

struct DqParams {
    const void* q;
    int8_t* out;
    float* scale;
    int64_t rows, H, q_stride;
    int exact;           // recompute near-tie codes from the exact rational
};

// Launch with programmatic stream serialisation allowed: the grid may be
// scheduled while the previous kernel on the stream drains; its kernels call
// pdl_wait() before reading global memory (before it they only issue L2
// prefetches, and, when the caller sets params_ready, read the inputs it covers).
template <typename... Args>
cudaError_t launch_pdl(void (*fn)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fn, args...);
}

// Kernel paths of the KV prologue, chosen by the host from shapes and alignment.
enum KvPath : int { KV_GENERIC = 0, KV_VEC = 1, KV_BULK = 2 };

// Launchers (host), defined next to their kernels. Return a CUDA error code.
cudaError_t launch_kv(const KvParams& p, int in_dtype, int ckv_kind, int path, cudaStream_t s);
cudaError_t launch_kv_bulk(const KvParams& p, int in_dtype, int ckv_kind, cudaStream_t s);
cudaError_t launch_qsa(const QsaParams& p, int in_dtype, bool vec, bool bulk, bool warp, cudaStream_t s);
// Shapes with a compiled warp-per-block QSA kernel.
bool qsa_warp_shape(int64_t Di, int64_t kbs);
cudaError_t launch_device_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s);
cudaError_t launch_dq(const DqParams& p, int in_dtype, bool vec, cudaStream_t s);

int sm_count_current_device();

}  // namespace kvr
