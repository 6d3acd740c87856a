// Host side of libkvr.so: argument validation, kernel selection, launch.
// Every entry point returns before launching anything when its arguments
// are invalid; see include/kvr.h for the contract.
#include <atomic>
#include <cstdlib>
#include <initializer_list>
#include <mutex>
#include <unordered_set>
#include <vector>

#include <algorithm>

#include "kvr_internal.cuh"

namespace kvr {

int sm_count_current_device() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return 1;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = 1;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

// 16-byte vectorised copy for the in-process bandwidth reference.
__global__ void __launch_bounds__(256) device_copy_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src,
                                                          int64_t n) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) dst[i] = ld_stream_v4(src + i);
}

cudaError_t launch_device_copy(void* dst, const void* src, int64_t bytes, cudaStream_t s) {
    const int64_t n = bytes / 16;
    const int64_t cap = int64_t(sm_count_current_device()) * 8;
    int64_t grid = (n + 255) / 256;
    if (grid > cap) grid = cap;
    device_copy_kernel<<<int(grid), 256, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src), n);
    return cudaGetLastError();
}

// Defined in bounded_wait.cu.
cudaError_t launch_bounded_wait(int32_t* status, int64_t limit_ns, int64_t abort_after_ns, cudaStream_t s);
cudaError_t launch_store_after_delay(int64_t* dst, const int64_t* src, int64_t count, int64_t delay_ns,
                                     cudaStream_t s);
// Defined in staging.cu.
cudaError_t launch_stage_in(void* dst, const void* src, int64_t bytes, cudaStream_t s);
cudaError_t launch_status_out(int32_t* host_status, const int32_t* dev_status, cudaStream_t s);

}  // namespace kvr

using namespace kvr;

// Smallest batch (token rows) that takes the bulk-copy pipeline; smaller
// batches take the register path, whose latency is lower.
#ifndef KVR_BULK_MIN_ROWS
#define KVR_BULK_MIN_ROWS 8192
#endif

namespace {

bool is16(kvr_dtype d) { return d == KVR_BF16 || d == KVR_F16; }
bool is8(kvr_dtype d) { return d == KVR_INT8 || d == KVR_FP8_E4M3FN || d == KVR_FP8_E5M2; }

int out_kind(kvr_dtype d) {
    switch (d) {
        case KVR_INT8: return OUT_I8;
        case KVR_FP8_E4M3FN: return OUT_E4M3;
        case KVR_FP8_E5M2: return OUT_E5M2;
        default: return OUT16;
    }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Do the byte ranges [a, a+na) and [b, b+nb) overlap?
bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
    if (a == nullptr || b == nullptr || na <= 0 || nb <= 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + uintptr_t(nb) && y < x + uintptr_t(na);
}

kvr_status cuda_status(cudaError_t e) { return e == cudaSuccess ? KVR_OK : KVR_ERR_CUDA; }

// True when every factor is nonnegative and their product stays below 2^62,
// so that the element offsets and byte counts derived from it cannot
// overflow int64.
bool product_fits(std::initializer_list<int64_t> factors) {
    int64_t p = 1;
    for (int64_t x : factors) {
        if (x < 0) return false;
        if (x != 0 && p > (int64_t(1) << 62) / x) return false;
        p *= x;
    }
    return true;
}

// Debug validation: -1 until the environment (KVR_DEBUG_VALIDATE=1) has
// been read, then 0 or 1; kvr_set_debug_validate() overrides it.
std::atomic<int> g_debug_validate{-1};

bool debug_validate() {
    int v = g_debug_validate.load();
    if (v < 0) {
        const char* e = std::getenv("KVR_DEBUG_VALIDATE");
        int unset = -1;
        g_debug_validate.compare_exchange_strong(unset, (e != nullptr && e[0] == '1') ? 1 : 0);
        v = g_debug_validate.load();
    }
    return v == 1;
}

// The cache row of every token of a kv_rmsnorm_rope_cache call, read from a
// host copy of its index: what the kernels cannot check (they see one row
// at a time) is that no two tokens name the same cache row, which the index
// restrictions of "aclnnKvRmsNormRopeCache" forbid (within a batch in Norm
// mode, anywhere in the paged modes). Out-of-range entries are reported
// here too. Returns KVR_ERR_INDEX on a violation.
kvr_status check_index_host(const kvr_kv_args* a, const int64_t* idx) {
    const int64_t Bkv = a->Bkv, Skv = a->Skv, d0 = a->cache_d0, d1 = a->cache_d1;
    std::unordered_set<int64_t> rows;
    rows.reserve(size_t(Bkv * Skv));
    if (a->mode == KVR_CACHE_NORM) {
        for (int64_t b = 0; b < Bkv; ++b)
            for (int64_t s = 0; s < Skv; ++s) {
                const int64_t e = idx[b * Skv + s];
                if (e == -1) continue;
                if (e < 0 || e >= d1) return KVR_ERR_INDEX;
                if (!rows.insert(b * d1 + e).second) return KVR_ERR_INDEX;
            }
    } else if (a->mode == KVR_CACHE_PA_BSND) {
        for (int64_t t = 0; t < Bkv * Skv; ++t) {
            const int64_t e = idx[t];
            if (e == -1) continue;
            if (e < 0 || e >= d0 * d1) return KVR_ERR_INDEX;
            if (!rows.insert(e).second) return KVR_ERR_INDEX;
        }
    } else {   // PA_BLK_BSND: one entry per d1 tokens; token s -> entry + s mod d1, inside the entry's block
        const int64_t nblk = (Skv + d1 - 1) / d1;
        for (int64_t b = 0; b < Bkv; ++b)
            for (int64_t q = 0; q < nblk; ++q) {
                const int64_t e = idx[b * nblk + q];
                if (e == -1) continue;
                const int64_t ntok = std::min(d1, Skv - q * d1);
                if (e < 0 || e >= d0 * d1 || e % d1 + ntok > d1) return KVR_ERR_INDEX;
                for (int64_t r = 0; r < ntok; ++r)
                    if (!rows.insert(e + r).second) return KVR_ERR_INDEX;
            }
    }
    return KVR_OK;
}

// Copy the index of a planned call to the host (synchronising `stream`) and
// check it. Skipped while the stream is being captured into a graph (a
// capture cannot synchronise).
kvr_status debug_check_index(const kvr_kv_args* a, cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return KVR_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return KVR_OK;
    const int64_t nblk = (a->Skv + a->cache_d1 - 1) / a->cache_d1;
    const int64_t n = a->mode == KVR_CACHE_PA_BLK_BSND ? a->Bkv * nblk : a->Bkv * a->Skv;
    std::vector<int64_t> idx(static_cast<size_t>(n));
    if (cudaMemcpyAsync(idx.data(), a->index, size_t(n) * sizeof(int64_t), cudaMemcpyDeviceToHost, stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return KVR_ERR_CUDA;
    }
    return check_index_host(a, idx.data());
}

}  // namespace

namespace {

// A validated kv_rmsnorm_rope_cache call, ready to launch.
struct KvPlan {
    KvParams p;
    int path;
    int in_dtype;
    int ckv_kind;
};

// Validate the arguments of kv_rmsnorm_rope_cache and fill the launch plan;
// `*empty` is set when there is nothing to launch (T = 0).
kvr_status kv_plan(const kvr_kv_args* a, KvPlan* plan, bool* empty) {
    *empty = false;
    if (a == nullptr) return KVR_ERR_NULL;
    if (a->Bkv < 0 || a->Skv < 0 || a->Dv < 1 || a->Dk < 2 || (a->Dk & 1) || a->cache_d0 < 1 ||
        a->cache_d1 < 1 || a->Dv > (int64_t(1) << 30) || a->Dk > (int64_t(1) << 30))
        return KVR_ERR_SHAPE;
    if (a->mode != KVR_CACHE_NORM && a->mode != KVR_CACHE_PA_BSND && a->mode != KVR_CACHE_PA_BLK_BSND)
        return KVR_ERR_MODE;
    if (!is16(a->in_dtype)) return KVR_ERR_DTYPE;
    if (!(a->ckv_dtype == a->in_dtype || is8(a->ckv_dtype))) return KVR_ERR_DTYPE;
    if (!(a->k_dtype == a->in_dtype || is8(a->k_dtype))) return KVR_ERR_DTYPE;
    const int64_t D = a->Dv + a->Dk;
    const int64_t stride = a->kv_row_stride == 0 ? D : a->kv_row_stride;
    if (stride < D) return KVR_ERR_SHAPE;
    if (!product_fits({a->Bkv, a->Skv, stride, 2}) || !product_fits({a->Bkv, a->Skv, a->Dk, 4}) ||
        !product_fits({a->cache_d0, a->cache_d1, D, 2}))
        return KVR_ERR_SHAPE;
    if (a->mode == KVR_CACHE_NORM && a->cache_d0 < a->Bkv) return KVR_ERR_SHAPE;
    if (!(a->eps >= 0.f) || !(a->kc_scale == a->kc_scale)) return KVR_ERR_SHAPE;
    const int64_t T = a->Bkv * a->Skv;
    if (T == 0) {   // empty input: caches are not updated
        *empty = true;
        return KVR_OK;
    }
    if (a->kv == nullptr || a->gamma == nullptr || a->cos == nullptr || a->sin == nullptr ||
        a->index == nullptr || a->ckv_cache == nullptr || a->k_cache == nullptr)
        return KVR_ERR_NULL;
    // 8-bit caches need their scale, 16-bit caches take none.
    if (is8(a->ckv_dtype) != (a->ckv_scale != nullptr)) return KVR_ERR_NULL;
    if (is8(a->k_dtype) != (a->k_scale != nullptr)) return KVR_ERR_NULL;
    if (a->ckv_scale != nullptr && a->ckv_scale_len != a->Dv && a->ckv_scale_len != 1) return KVR_ERR_SHAPE;
    if (a->k_scale != nullptr && a->k_scale_len != a->Dk && a->k_scale_len != 1) return KVR_ERR_SHAPE;
    if (!aligned(a->kv, 2) || !aligned(a->gamma, 2) || !aligned(a->cos, 2) || !aligned(a->sin, 2) ||
        !aligned(a->index, 8) || !aligned(a->ckv_scale, 4) || !aligned(a->k_scale, 4) ||
        (is16(a->ckv_dtype) && !aligned(a->ckv_cache, 2)) || (is16(a->k_dtype) && !aligned(a->k_cache, 2)))
        return KVR_ERR_SHAPE;

    const int64_t nblk = (a->Skv + a->cache_d1 - 1) / a->cache_d1;
    const int64_t n_index = a->mode == KVR_CACHE_PA_BLK_BSND ? a->Bkv * nblk : T;
    const int64_t rows = a->cache_d0 * a->cache_d1;
    const int64_t ckv_bytes = rows * a->Dv * (is16(a->ckv_dtype) ? 2 : 1);
    const int64_t k_bytes = rows * a->Dk * (is16(a->k_dtype) ? 2 : 1);
    const int64_t kv_bytes = ((T - 1) * stride + D) * 2;
    const void* ins[] = {a->kv, a->gamma, a->cos, a->sin, a->index, a->ckv_scale, a->k_scale};
    const int64_t in_bytes[] = {kv_bytes, a->Dv * 2, T * a->Dk * 2, T * a->Dk * 2, n_index * 8,
                                a->ckv_scale_len * 4, a->k_scale_len * 4};
    for (int i = 0; i < 7; ++i)
        if (overlap(a->ckv_cache, ckv_bytes, ins[i], in_bytes[i]) || overlap(a->k_cache, k_bytes, ins[i], in_bytes[i]))
            return KVR_ERR_ALIAS;
    if (overlap(a->ckv_cache, ckv_bytes, a->k_cache, k_bytes)) return KVR_ERR_ALIAS;

    KvParams& p = plan->p;
    p = KvParams{};
    p.kv = a->kv;
    p.gamma = a->gamma;
    p.cos = a->cos;
    p.sin = a->sin;
    p.index = a->index;
    p.ckv = a->ckv_cache;
    p.kc = a->k_cache;
    p.ckv_scale = a->ckv_scale;
    p.k_scale = a->k_scale;
    p.status = a->dev_status;
    p.T = T;
    p.Skv = a->Skv;
    p.kv_stride = stride;
    p.d0 = a->cache_d0;
    p.d1 = a->cache_d1;
    p.nblk = nblk;
    p.Dv = int(a->Dv);
    p.Dk = int(a->Dk);
    p.mode = int(a->mode);
    p.k_kind = out_kind(a->k_dtype);
    p.ckv_scale_per_ch = a->ckv_scale_len == a->Dv && a->Dv > 1;
    p.k_scale_per_ch = a->k_scale_len == a->Dk;
    p.eps = a->eps;
    p.inv_dv = 1.0f / float(a->Dv);
    p.alpha = a->kc_scale;
    p.params_ready = a->params_ready != 0;

    // Kernel path: the bulk-copy pipeline and the register path need 16-byte
    // rows (Dv, Dk multiples of 8, 16-byte aligned bases and row stride);
    // anything else takes the element-wise path.
    const bool ckv8 = is8(a->ckv_dtype), k8 = is8(a->k_dtype);
    const bool vec = (a->Dv % 8 == 0) && a->Dv <= 1024 && (a->Dk % 8 == 0) && a->Dk <= 256 && (stride % 8 == 0) &&
                     aligned(a->kv, 16) && aligned(a->gamma, 16) && aligned(a->cos, 16) && aligned(a->sin, 16) &&
                     aligned(a->ckv_cache, ckv8 ? 8 : 16) && aligned(a->k_cache, k8 ? 4 : 8) &&
                     aligned(a->ckv_scale, 16);
    int path = vec ? KV_VEC : KV_GENERIC;
    if (vec && T >= KVR_BULK_MIN_ROWS) {
        path = KV_BULK;
        p.kv_contig = stride == D;
        p.idx_bulk = a->mode != KVR_CACHE_PA_BLK_BSND && aligned(a->index, 16);
    }
    plan->path = path;
    plan->in_dtype = a->in_dtype;
    plan->ckv_kind = out_kind(a->ckv_dtype);
    return KVR_OK;
}


}  // namespace

extern "C" {

int kvr_abi_version(void) { return KVR_ABI_VERSION; }

const char* kvr_status_string(kvr_status s) {
    switch (s) {
        case KVR_OK: return "ok";
        case KVR_ERR_NULL: return "a required pointer is NULL, or an optional pair is half given";
        case KVR_ERR_SHAPE: return "a size is outside its documented range";
        case KVR_ERR_DTYPE: return "an element type is not supported for that argument";
        case KVR_ERR_MODE: return "unknown cache mode";
        case KVR_ERR_ALIAS: return "an output overlaps an input it must not overlap";
        case KVR_ERR_CUDA: return "the CUDA launch failed";
        case KVR_ERR_INDEX: return "debug validation: an index entry is out of range or names a cache row another entry names";
    }
    return "unknown status";
}

void kvr_set_debug_validate(int on) { g_debug_validate.store(on ? 1 : 0); }

kvr_status kv_rmsnorm_rope_cache(const kvr_kv_args* a, cudaStream_t stream) {
    KvPlan plan;
    bool empty;
    const kvr_status st = kv_plan(a, &plan, &empty);
    if (st != KVR_OK || empty) return st;
    if (debug_validate()) {
        const kvr_status v = debug_check_index(a, stream);
        if (v != KVR_OK) return v;
    }
    (void)cudaGetLastError();
    return cuda_status(launch_kv(plan.p, plan.in_dtype, plan.ckv_kind, plan.path, stream));
}

// Device address of pinned (page-locked, device-mapped) host memory, or NULL
// for anything else (pageable or unknown memory keeps the copy-engine path).
static void* mapped_host_ptr(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return at.type == cudaMemoryTypeHost ? at.devicePointer : nullptr;
}

#ifndef KVR_STAGE_WITH_KERNELS
#define KVR_STAGE_WITH_KERNELS 1
#endif

kvr_status kv_rmsnorm_rope_cache_staged(const kvr_kv_args* a, const void* host_src, void* dev_dst, int64_t bytes,
                                        int32_t* host_status, cudaStream_t stream) {
    if (a == nullptr) return KVR_ERR_NULL;
    if (bytes < 0) return KVR_ERR_SHAPE;
    if (bytes > 0 && (host_src == nullptr || dev_dst == nullptr)) return KVR_ERR_NULL;
    if (host_status != nullptr && a->dev_status == nullptr) return KVR_ERR_NULL;
    KvPlan plan;
    bool empty;
    const kvr_status st = kv_plan(a, &plan, &empty);
    if (st != KVR_OK) return st;
    // Pinned inputs in whole 16-byte units go through a copy kernel chained
    // with the KV kernel; anything else through a copy-engine operation.
    const void* src_dev = (KVR_STAGE_WITH_KERNELS && bytes > 0 && bytes % 16 == 0 && aligned(host_src, 16) &&
                           aligned(dev_dst, 16))
                              ? mapped_host_ptr(host_src)
                              : nullptr;
    int32_t* status_dev = (KVR_STAGE_WITH_KERNELS && host_status != nullptr && aligned(host_status, 4))
                              ? static_cast<int32_t*>(mapped_host_ptr(host_status))
                              : nullptr;
    (void)cudaGetLastError();
    if (bytes > 0) {
        const cudaError_t e = src_dev != nullptr
                                  ? launch_stage_in(dev_dst, src_dev, bytes, stream)
                                  : cudaMemcpyAsync(dev_dst, host_src, size_t(bytes), cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return KVR_ERR_CUDA;
    }
    if (!empty && debug_validate()) {   // after the copy: the index may be part of the staged inputs
        const kvr_status v = debug_check_index(a, stream);
        if (v != KVR_OK) return v;
    }
    if (!empty) {
        const cudaError_t e = launch_kv(plan.p, plan.in_dtype, plan.ckv_kind, plan.path, stream);
        if (e != cudaSuccess) return KVR_ERR_CUDA;
    }
    if (host_status != nullptr) {
        const cudaError_t e =
            status_dev != nullptr
                ? launch_status_out(status_dev, a->dev_status, stream)
                : cudaMemcpyAsync(host_status, a->dev_status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
        if (e != cudaSuccess) return KVR_ERR_CUDA;
    }
    return KVR_OK;
}

kvr_status qsa_prepare(const kvr_qsa_args* a, cudaStream_t stream) {
    if (a == nullptr) return KVR_ERR_NULL;
    if (!is16(a->in_dtype)) return KVR_ERR_DTYPE;
    if (a->rope_layout < KVR_QSA_ROPE_INTERLEAVE_LAST || a->rope_layout > KVR_QSA_ROPE_HALF_FIRST)
        return KVR_ERR_MODE;
    // With no new tokens (L = 0) the tables are never read and may be NULL:
    // the rotation is then on iff the carried cos/sin is given.
    const bool rope = a->rope_cos != nullptr || a->rope_sin != nullptr ||
                      (a->L == 0 && a->past_incomplete_rope != nullptr);
    if (a->N < 0 || a->L < 0 || a->Di < 1 || a->Di > 4096 || a->Bcap < 1 || a->key_block_size < 2 ||
        a->Bp < 0 || (a->key_length_len != 1 && a->key_length_len != a->N))
        return KVR_ERR_SHAPE;
    if (rope && (a->Dr < 2 || (a->Dr & 1) || a->Dr > a->Di)) return KVR_ERR_SHAPE;
    if (!(a->eps >= 0.f)) return KVR_ERR_SHAPE;
    if (!product_fits({a->N, a->L, a->Di, 2}) || !product_fits({a->N, a->Bcap, a->Di, 2}) ||
        !product_fits({a->N, a->Bp, a->Di, 2}) || !product_fits({a->N, a->key_block_size, a->Di, 2}) ||
        !product_fits({a->key_length_len, 8}))
        return KVR_ERR_SHAPE;
    // Concat-output form: the past block keys come from a separate buffer.
    const bool concat = a->past_block_index_keys != nullptr && a->past_block_index_keys != a->block_keys;
    // Without new tokens only the carry outputs and the past-row copy remain.
    if (a->N == 0 ||
        (a->L == 0 && !concat && a->next_incomplete_raw_keys == nullptr && a->next_incomplete_rope == nullptr))
        return KVR_OK;
    if ((a->L > 0 && a->raw_index_keys == nullptr) || a->block_keys == nullptr || a->key_length == nullptr ||
        a->past_incomplete_raw_keys == nullptr)
        return KVR_ERR_NULL;
    if (rope && a->past_incomplete_rope == nullptr) return KVR_ERR_NULL;
    if (rope && a->L > 0 && (a->rope_cos == nullptr || a->rope_sin == nullptr)) return KVR_ERR_NULL;
    if (!rope && a->past_incomplete_rope != nullptr) return KVR_ERR_NULL;
    if (!rope && a->next_incomplete_rope != nullptr) return KVR_ERR_NULL;
    const int64_t kbs = a->key_block_size;
    const int64_t nbmax = (a->L + kbs - 1) / kbs;
    const int64_t Dr = rope ? a->Dr : 0;
    const bool vec = (a->Di % 8 == 0) && aligned(a->raw_index_keys, 16) && aligned(a->past_incomplete_raw_keys, 16);
    const bool bulk = vec && (Dr % 8 == 0) && aligned(a->rope_cos, 16) && aligned(a->rope_sin, 16) &&
                      aligned(a->past_incomplete_rope, 16) && aligned(a->k_norm_weight, 16);
    const bool warp = bulk && qsa_warp_shape(a->Di, kbs);
    // Past rows copied per CTA in the concat form: about 16 KB (4 KB per
    // warp in the warp-per-block kernel).
    const int64_t copy_bytes = warp ? 4096 : 16384;
    const int64_t copy_rows = a->Di * 2 >= copy_bytes ? 1 : copy_bytes / (a->Di * 2);
    const int64_t ncopy = concat ? (std::min(a->Bp, a->Bcap) + copy_rows - 1) / copy_rows : 0;
    if (a->N * (nbmax + 1 + ncopy) > 0x7FFFFFFFLL) return KVR_ERR_SHAPE;
    const void* ptrs[] = {a->raw_index_keys, a->block_keys, a->rope_cos, a->rope_sin, a->k_norm_weight,
                          a->past_incomplete_raw_keys, a->past_incomplete_rope, a->next_incomplete_raw_keys,
                          a->next_incomplete_rope, a->past_block_index_keys};
    for (const void* q : ptrs)
        if (!aligned(q, 2)) return KVR_ERR_SHAPE;
    if (!aligned(a->key_length, 8)) return KVR_ERR_SHAPE;

    const int64_t nr_bytes = a->N * (kbs - 1) * a->Di * 2;
    const int64_t nrope_bytes = a->N * 2 * Dr * 2;
    const void* ins[] = {a->raw_index_keys, a->block_keys, a->rope_cos, a->rope_sin, a->k_norm_weight,
                         a->past_incomplete_raw_keys, a->past_incomplete_rope, a->key_length,
                         concat ? a->past_block_index_keys : nullptr};
    const int64_t in_bytes[] = {a->N * a->L * a->Di * 2, a->N * a->Bcap * a->Di * 2, a->N * a->L * Dr * 2,
                                a->N * a->L * Dr * 2, a->Di * 2, nr_bytes, nrope_bytes, a->key_length_len * 8,
                                a->N * a->Bp * a->Di * 2};
    constexpr int n_ins = sizeof(ins) / sizeof(ins[0]);
    for (int i = 0; i < n_ins; ++i)
        if (overlap(a->next_incomplete_raw_keys, nr_bytes, ins[i], in_bytes[i]) ||
            overlap(a->next_incomplete_rope, nrope_bytes, ins[i], in_bytes[i]))
            return KVR_ERR_ALIAS;
    if (overlap(a->next_incomplete_raw_keys, nr_bytes, a->next_incomplete_rope, nrope_bytes)) return KVR_ERR_ALIAS;
    for (int i = 0; i < n_ins; ++i)
        if (i != 1 && overlap(a->block_keys, in_bytes[1], ins[i], in_bytes[i])) return KVR_ERR_ALIAS;

    QsaParams p;
    p.raw = a->raw_index_keys;
    p.block_keys = a->block_keys;
    p.key_length = a->key_length;
    p.cos = a->rope_cos;
    p.sin = a->rope_sin;
    p.w = a->k_norm_weight;
    p.past_raw = a->past_incomplete_raw_keys;
    p.past_rope = a->past_incomplete_rope;
    p.next_raw = a->next_incomplete_raw_keys;
    p.next_rope = a->next_incomplete_rope;
    p.past_bk = concat ? a->past_block_index_keys : nullptr;
    p.status = a->dev_status;
    p.N = a->N;
    p.L = a->L;
    p.Bcap = a->Bcap;
    p.kbs = kbs;
    p.nbmax = nbmax;
    p.Bp = a->Bp;
    p.ncopy = ncopy;
    p.copy_rows = int(copy_rows);
    p.copy_vec = concat && a->Di % 8 == 0 && aligned(a->past_block_index_keys, 16) && aligned(a->block_keys, 16);
    p.key_length_per_seq = a->key_length_len == a->N && a->N > 1;
    p.Di = int(a->Di);
    p.Dr = int(Dr);
    p.rope_first = a->rope_layout == KVR_QSA_ROPE_INTERLEAVE_FIRST || a->rope_layout == KVR_QSA_ROPE_HALF_FIRST;
    p.rope_half = a->rope_layout == KVR_QSA_ROPE_HALF_LAST || a->rope_layout == KVR_QSA_ROPE_HALF_FIRST;
    p.params_ready = a->params_ready != 0;
    p.key_length_late = a->key_length_late != 0;
    p.eps = a->eps;
    p.inv_di = 1.0f / float(a->Di);
    p.inv_kbs = 1.0f / float(kbs);

    (void)cudaGetLastError();
    return cuda_status(launch_qsa(p, a->in_dtype, vec, bulk, warp, stream));
}

kvr_status kvr_check_bounded_wait(int32_t* dev_status, int64_t limit_ns, int64_t abort_after_ns,
                                  cudaStream_t stream) {
    if (dev_status == nullptr) return KVR_ERR_NULL;
    if (limit_ns < 1000 || limit_ns > 1000000000 || abort_after_ns < 0 || abort_after_ns > limit_ns)
        return KVR_ERR_SHAPE;
    (void)cudaGetLastError();
    return cuda_status(launch_bounded_wait(dev_status, limit_ns, abort_after_ns, stream));
}

kvr_status kvr_store_after_delay(int64_t* dst, const int64_t* src, int64_t count, int64_t delay_ns,
                                 cudaStream_t stream) {
    if (count < 0 || count > (int64_t(1) << 20) || delay_ns < 0 || delay_ns > 100000000) return KVR_ERR_SHAPE;
    if (count == 0) return KVR_OK;
    if (dst == nullptr || src == nullptr) return KVR_ERR_NULL;
    if (!aligned(dst, 8) || !aligned(src, 8)) return KVR_ERR_SHAPE;
    if (overlap(dst, count * 8, src, count * 8)) return KVR_ERR_ALIAS;
    (void)cudaGetLastError();
    return cuda_status(launch_store_after_delay(dst, src, count, delay_ns, stream));
}

kvr_status dynamic_quant(const kvr_dq_args* a, cudaStream_t stream) {
    if (a == nullptr) return KVR_ERR_NULL;
    if (!is16(a->in_dtype)) return KVR_ERR_DTYPE;
    const int64_t stride = a->q_row_stride == 0 ? a->Hckv : a->q_row_stride;
    if (a->rows < 0 || a->Hckv < 1 || stride < a->Hckv || !product_fits({a->rows, stride, 2}))
        return KVR_ERR_SHAPE;
    if (a->rows == 0) return KVR_OK;
    if (a->q_nope == nullptr || a->q_out == nullptr || a->dequant_scale == nullptr) return KVR_ERR_NULL;
    if (!aligned(a->q_nope, 2) || !aligned(a->dequant_scale, 4)) return KVR_ERR_SHAPE;
    const int64_t in_bytes = ((a->rows - 1) * stride + a->Hckv) * 2;
    if (overlap(a->q_out, a->rows * a->Hckv, a->q_nope, in_bytes) ||
        overlap(a->dequant_scale, a->rows * 4, a->q_nope, in_bytes) ||
        overlap(a->dequant_scale, a->rows * 4, a->q_out, a->rows * a->Hckv))
        return KVR_ERR_ALIAS;
    DqParams p;
    p.q = a->q_nope;
    p.out = a->q_out;
    p.scale = a->dequant_scale;
    p.rows = a->rows;
    p.H = a->Hckv;
    p.q_stride = stride;
    p.exact = a->exact != 0;
    const bool vec = a->Hckv % 8 == 0 && a->Hckv <= 1024 && stride % 8 == 0 && aligned(a->q_nope, 16) &&
                     aligned(a->q_out, 8);
    (void)cudaGetLastError();
    return cuda_status(launch_dq(p, a->in_dtype, vec, stream));
}

kvr_status kvr_device_copy(void* dst, const void* src, int64_t bytes, cudaStream_t stream) {
    if (bytes == 0) return KVR_OK;
    if (dst == nullptr || src == nullptr) return KVR_ERR_NULL;
    if (bytes < 0 || bytes % 16 != 0 || !aligned(dst, 16) || !aligned(src, 16)) return KVR_ERR_SHAPE;
    if (overlap(dst, bytes, src, bytes)) return KVR_ERR_ALIAS;
    (void)cudaGetLastError();
    return cuda_status(launch_device_copy(dst, src, bytes, stream));
}

}  // extern "C"
