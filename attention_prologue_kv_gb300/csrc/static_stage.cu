// kv_rmsnorm_rope_cache_staged_static: the host-staged KV call for callers
// that cannot allocate device memory.
//
// kv_rmsnorm_rope_cache_staged copies a step's packed inputs from host memory
// into a device buffer the caller provides. Some callers have no way to
// provide one: code that runs where cudaMalloc is not allowed (inside a
// custom allocator's own callbacks, under a framework that owns all device
// memory and exposes no allocation hook to plugins, or in a process whose
// allocation budget is already committed). For them this entry point keeps
// the staging area in a file-scope device array instead: the driver sets it
// aside when it loads this library's code on a device, and it stays there
// until the process exits. Nothing here calls cudaMalloc, cudaFree or any
// routine that allocates device memory.
//
// Host code cannot use the array's name as a device address (in host code
// the name denotes a host-side stand-in), so every call looks the address up
// with cudaGetSymbolAddress in the current context and checks the result.
// The lookup allocates nothing; it is redone on every call rather than kept,
// because a kept address goes stale when the device is reset or when the
// caller runs in a context other than the one it was looked up in. The first
// lookup on a device may load this library's device code there. Device code
// could name the array directly; the kernels here receive the looked-up
// address as an ordinary pointer.
#include "kvr_internal.cuh"

// The staging area (KVR_STATIC_STAGE_BYTES, declared in kvr.h).
static __device__ __align__(256) unsigned char kvr_static_stage[KVR_STATIC_STAGE_BYTES];

namespace {

// Device address of the staging area in the current context.
kvr_status static_stage_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, kvr_static_stage) != cudaSuccess || p == nullptr) {
        (void)cudaGetLastError();
        return KVR_ERR_CUDA;
    }
    *out = p;
    return KVR_OK;
}

// [off, off + len) lies inside [0, bytes) and off is a multiple of align.
bool span_inside(int64_t off, int64_t len, int64_t bytes, int64_t align) {
    return off >= 0 && off % align == 0 && off <= bytes && len <= bytes - off;
}

}  // namespace

extern "C" kvr_status kv_rmsnorm_rope_cache_staged_static(const kvr_kv_args* args, const void* host_src,
                                                           int64_t bytes, int64_t kv_offset, int64_t cos_offset,
                                                           int64_t sin_offset, int64_t index_offset,
                                                           int32_t* host_status, cudaStream_t stream) {
    if (args == nullptr) return KVR_ERR_NULL;
    if (bytes < 0 || bytes > KVR_STATIC_STAGE_BYTES) return KVR_ERR_SHAPE;
    int64_t T = 0;
    if (args->Bkv < 0 || args->Skv < 0 || __builtin_mul_overflow(args->Bkv, args->Skv, &T)) return KVR_ERR_SHAPE;
    kvr_kv_args a = *args;
    void* base = nullptr;
    if (T > 0) {
        // Every byte the call reads from the staging area must come from this
        // call's copy: the four inputs have to lie inside [0, bytes).
        if (args->Dv < 1 || args->Dk < 2 || args->Dv > bytes || args->Dk > bytes || T > bytes ||
            args->cache_d1 < 1)
            return KVR_ERR_SHAPE;
        const int64_t D = args->Dv + args->Dk;
        const int64_t stride = args->kv_row_stride == 0 ? D : args->kv_row_stride;
        if (stride < D || stride > bytes) return KVR_ERR_SHAPE;
        const int64_t kv_len = ((T - 1) * stride + D) * 2;
        const int64_t table_len = T * args->Dk * 2;
        const int64_t n_index = args->mode == KVR_CACHE_PA_BLK_BSND
                                    ? args->Bkv * ((args->Skv + args->cache_d1 - 1) / args->cache_d1)
                                    : T;
        if (!span_inside(kv_offset, kv_len, bytes, 2) || !span_inside(cos_offset, table_len, bytes, 2) ||
            !span_inside(sin_offset, table_len, bytes, 2) || !span_inside(index_offset, n_index * 8, bytes, 8))
            return KVR_ERR_SHAPE;
        if (host_src == nullptr) return KVR_ERR_NULL;
        const kvr_status st = static_stage_address(&base);
        if (st != KVR_OK) return st;
        unsigned char* b = static_cast<unsigned char*>(base);
        a.kv = b + kv_offset;
        a.cos = b + cos_offset;
        a.sin = b + sin_offset;
        a.index = reinterpret_cast<const int64_t*>(b + index_offset);
    } else {
        bytes = 0;   // nothing to read: no copy
    }
    return kv_rmsnorm_rope_cache_staged(&a, host_src, base, bytes, host_status, stream);
}
