// Fused KV prologue kernels: RMSNorm (left Dv) + interleaved RoPE (right Dk)
// + optional 8-bit quantisation + scatter into two caches.
//
// Operation: "aclnnKvRmsNormRopeCache" (hiascend.com), "Description",
// "Formulas (1) interleaveRope", "Formulas (2) rmsNorm", "Restrictions on
// index", "Restrictions on quantization scenarios"; the alpha_kv factor of
// "aclnnMlaPrologV3WeightNz" ("Formula", key path).
//
// Design (memory-bound stream, ~1 flop per byte, no tensor cores):
//  * one warp per token row, grid-stride over rows, 4 warps per CTA, grid
//    sized to the resident capacity of the GPU;
//  * per row every lane issues its loads at once: the int64 index, 16-byte
//    non-caching loads of the Dv part (CPL chunks of 8 elements per lane),
//    and, on the first Dk/8 lanes, one 16-byte chunk of the Dk part (4 RoPE
//    pairs) plus the four 8-byte cos/sin pieces those pairs need;
//  * sum of squares in float32 with a warp butterfly, one rsqrt;
//  * gamma (and per-channel scales) staged once per CTA in shared memory;
//  * whole cache rows written with 16-byte (8-byte for 8-bit codes) stores:
//    512 contiguous bytes per warp instruction for the Dv part, two 64-byte
//    runs for the Dk part, so every 32-byte sector is fully written;
//  * index -1 skips the row; an out-of-range index skips it and raises
//    KVR_DEVERR_INDEX. No atomics touch data.
#include <map>
#include <mutex>
#include <utility>

#include "kvr_internal.cuh"

namespace kvr {

constexpr int KV_THREADS = 128;
constexpr int KV_WARPS = KV_THREADS / 32;
constexpr int64_t ROW_SKIP = -1;
constexpr int64_t ROW_BAD = -2;

// Position in `index` of the entry that governs token t.
__device__ __forceinline__ int64_t index_pos(const KvParams& p, int64_t t) {
    if (p.mode == KVR_CACHE_PA_BLK_BSND) {
        int64_t b = t / p.Skv;
        int64_t s = t - b * p.Skv;
        return b * p.nblk + s / p.d1;
    }
    return t;
}

// Flat cache row (in units of one D*-row) for token t with index entry v.
__device__ __forceinline__ int64_t resolve_row(const KvParams& p, int64_t t, int64_t v) {
    if (v == -1) return ROW_SKIP;
    if (p.mode == KVR_CACHE_NORM) {
        if (v < 0 || v >= p.d1) return ROW_BAD;
        return (t / p.Skv) * p.d1 + v;
    }
    const int64_t nslots = p.d0 * p.d1;
    if (v < 0 || v >= nslots) return ROW_BAD;
    if (p.mode == KVR_CACHE_PA_BSND) return v;
    const int64_t off = (t % p.Skv) % p.d1;
    if ((v % p.d1) + off >= p.d1) return ROW_BAD;
    return v + off;
}

struct RowRegs {
    int64_t v;
    uint4 x[4];
    uint4 xr;
    uint2 c0, c1, s0, s1;
};

template <int CPL>
__device__ __forceinline__ void load_row(const KvParams& p, int64_t t, int lane, int nch, int nrl,
                                         int h, RowRegs& r) {
    r.v = ld_stream_s64(p.index + index_pos(p, t));
    const char* x = static_cast<const char*>(p.kv) + t * p.kv_stride * 2;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int ch = c * 32 + lane;
        if (ch < nch) r.x[c] = ld_stream_v4(x + ch * 16);
    }
    if (lane < nrl) {
        r.xr = ld_stream_v4(x + int64_t(p.Dv) * 2 + lane * 16);
        const char* cr = static_cast<const char*>(p.cos) + t * p.Dk * 2;
        const char* sr = static_cast<const char*>(p.sin) + t * p.Dk * 2;
        r.c0 = ld_stream_v2(cr + lane * 8);
        r.c1 = ld_stream_v2(cr + h * 2 + lane * 8);
        r.s0 = ld_stream_v2(sr + lane * 8);
        r.s1 = ld_stream_v2(sr + h * 2 + lane * 8);
    }
}

// Vector path: Dv % 8 == 0 and Dv <= 256*CPL, Dk % 8 == 0 and Dk <= 256,
// 16-byte aligned rows. CK = OutKind of the ckv cache.
template <class IT, int CPL, int CK>
__global__ void __launch_bounds__(KV_THREADS) kv_vec_kernel(const KvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint4* s_gamma = reinterpret_cast<uint4*>(smem);                  // Dv 16-bit values
    float* s_cscale = reinterpret_cast<float*>(smem + p.Dv * 2);      // Dv floats
    float* s_kscale = s_cscale + p.Dv;                                // Dk floats

    const int lane = threadIdx.x & 31;
    const int nch = p.Dv >> 3;
    const int nrl = p.Dk >> 3;
    const int h = p.Dk >> 1;
    const int64_t stride_rows = int64_t(gridDim.x) * KV_WARPS;
    int64_t t = int64_t(blockIdx.x) * KV_WARPS + (threadIdx.x >> 5);

    RowRegs r;
    if (t < p.T) load_row<CPL>(p, t, lane, nch, nrl, h, r);

    // Stage per-channel constants once per CTA (overlaps the first row's loads).
    for (int i = threadIdx.x; i < nch; i += KV_THREADS)
        s_gamma[i] = ld_stream_v4(static_cast<const char*>(p.gamma) + i * 16);
    const bool cq = CK != OUT16;
    const bool kq = p.k_kind != OUT16;
    if (cq && p.ckv_scale_per_ch)
        for (int i = threadIdx.x; i < p.Dv; i += KV_THREADS) s_cscale[i] = p.ckv_scale[i];
    if (kq && p.k_scale_per_ch)
        for (int i = threadIdx.x; i < p.Dk; i += KV_THREADS) s_kscale[i] = p.k_scale[i];
    const float cscale0 = (cq && !p.ckv_scale_per_ch) ? p.ckv_scale[0] : 1.f;
    const float kscale0 = (kq && !p.k_scale_per_ch) ? p.k_scale[0] : 1.f;
    __syncthreads();

    while (t < p.T) {
        const int64_t row = resolve_row(p, t, r.v);
        if (row >= 0) {
            // ---- RMSNorm of the Dv part ----
            float ss = 0.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                if (c * 32 + lane < nch) {
                    const uint32_t w[4] = {r.x[c].x, r.x[c].y, r.x[c].z, r.x[c].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float a = IT::lo(w[k]), b = IT::hi(w[k]);
                        ss = fmaf(a, a, ss);
                        ss = fmaf(b, b, ss);
                    }
                }
            }
            ss = warp_sum(ss);
            const float rr = rsqrtf(fmaf(ss, p.inv_dv, p.eps)) * p.alpha;
            char* crow = static_cast<char*>(p.ckv) + row * p.Dv * (CK == OUT16 ? 2 : 1);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = c * 32 + lane;
                if (ch < nch) {
                    const uint4 gv = s_gamma[ch];
                    const uint32_t w[4] = {r.x[c].x, r.x[c].y, r.x[c].z, r.x[c].w};
                    const uint32_t g[4] = {gv.x, gv.y, gv.z, gv.w};
                    float y[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        y[2 * k] = IT::lo(w[k]) * rr * IT::lo(g[k]);
                        y[2 * k + 1] = IT::hi(w[k]) * rr * IT::hi(g[k]);
                    }
                    if constexpr (CK == OUT16) {
                        uint4 o;
                        o.x = IT::pack(y[0], y[1]);
                        o.y = IT::pack(y[2], y[3]);
                        o.z = IT::pack(y[4], y[5]);
                        o.w = IT::pack(y[6], y[7]);
                        *reinterpret_cast<uint4*>(crow + ch * 16) = o;
                    } else {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            y[k] *= p.ckv_scale_per_ch ? s_cscale[ch * 8 + k] : cscale0;
                        uint2 o;
                        o.x = enc8x2<CK>(y[0], y[1]) | (enc8x2<CK>(y[2], y[3]) << 16);
                        o.y = enc8x2<CK>(y[4], y[5]) | (enc8x2<CK>(y[6], y[7]) << 16);
                        *reinterpret_cast<uint2*>(crow + ch * 8) = o;
                    }
                }
            }
            // ---- interleaved RoPE of the Dk part: lane owns pairs 4*lane .. 4*lane+3 ----
            if (lane < nrl) {
                const uint32_t w[4] = {r.xr.x, r.xr.y, r.xr.z, r.xr.w};
                const uint32_t cw0[2] = {r.c0.x, r.c0.y}, cw1[2] = {r.c1.x, r.c1.y};
                const uint32_t sw0[2] = {r.s0.x, r.s0.y}, sw1[2] = {r.s1.x, r.s1.y};
                float o1[4], o2[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a = IT::lo(w[k]);   // x1[i] = x[2i]
                    const float b = IT::hi(w[k]);   // x2[i] = x[2i+1]
                    const float ca = (k & 1) ? IT::hi(cw0[k >> 1]) : IT::lo(cw0[k >> 1]);
                    const float sa = (k & 1) ? IT::hi(sw0[k >> 1]) : IT::lo(sw0[k >> 1]);
                    const float cb = (k & 1) ? IT::hi(cw1[k >> 1]) : IT::lo(cw1[k >> 1]);
                    const float sb = (k & 1) ? IT::hi(sw1[k >> 1]) : IT::lo(sw1[k >> 1]);
                    o1[k] = a * ca - b * sa;        // lane i:      x1*cos + (-x2)*sin
                    o2[k] = b * cb + a * sb;        // lane i+Dk/2: x2*cos + x1*sin
                }
                if (p.k_kind == OUT16) {
                    char* krow = static_cast<char*>(p.kc) + row * p.Dk * 2;
                    uint2 q1, q2;
                    q1.x = IT::pack(o1[0], o1[1]);
                    q1.y = IT::pack(o1[2], o1[3]);
                    q2.x = IT::pack(o2[0], o2[1]);
                    q2.y = IT::pack(o2[2], o2[3]);
                    *reinterpret_cast<uint2*>(krow + lane * 8) = q1;
                    *reinterpret_cast<uint2*>(krow + h * 2 + lane * 8) = q2;
                } else {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        o1[k] *= p.k_scale_per_ch ? s_kscale[lane * 4 + k] : kscale0;
                        o2[k] *= p.k_scale_per_ch ? s_kscale[h + lane * 4 + k] : kscale0;
                    }
                    char* krow = static_cast<char*>(p.kc) + row * p.Dk;
                    const uint32_t q1 = enc8x2_rt(p.k_kind, o1[0], o1[1]) | (enc8x2_rt(p.k_kind, o1[2], o1[3]) << 16);
                    const uint32_t q2 = enc8x2_rt(p.k_kind, o2[0], o2[1]) | (enc8x2_rt(p.k_kind, o2[2], o2[3]) << 16);
                    *reinterpret_cast<uint32_t*>(krow + lane * 4) = q1;
                    *reinterpret_cast<uint32_t*>(krow + h + lane * 4) = q2;
                }
            }
        } else if (row == ROW_BAD && lane == 0 && p.status != nullptr) {
            atomicOr(p.status, KVR_DEVERR_INDEX);
        }
        t += stride_rows;
        if (t < p.T) load_row<CPL>(p, t, lane, nch, nrl, h, r);
    }
}

// Generic path: any Dv >= 1, any even Dk, element-aligned pointers, any row
// stride. One warp per row, element-wise loops (two passes over the Dv part).
template <class IT>
__global__ void __launch_bounds__(KV_THREADS) kv_generic_kernel(const KvParams p, int ck) {
    const int lane = threadIdx.x & 31;
    const int h = p.Dk >> 1;
    const uint16_t* gamma = static_cast<const uint16_t*>(p.gamma);
    const uint16_t* cosb = static_cast<const uint16_t*>(p.cos);
    const uint16_t* sinb = static_cast<const uint16_t*>(p.sin);
    for (int64_t t = int64_t(blockIdx.x) * KV_WARPS + (threadIdx.x >> 5); t < p.T;
         t += int64_t(gridDim.x) * KV_WARPS) {
        const int64_t row = resolve_row(p, t, p.index[index_pos(p, t)]);
        if (row < 0) {
            if (row == ROW_BAD && lane == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_INDEX);
            continue;
        }
        const uint16_t* x = static_cast<const uint16_t*>(p.kv) + t * p.kv_stride;
        float ss = 0.f;
        for (int c = lane; c < p.Dv; c += 32) {
            const float a = IT::one(x[c]);
            ss = fmaf(a, a, ss);
        }
        ss = warp_sum(ss);
        const float rr = rsqrtf(fmaf(ss, p.inv_dv, p.eps)) * p.alpha;
        for (int c = lane; c < p.Dv; c += 32) {
            float y = IT::one(x[c]) * rr * IT::one(gamma[c]);
            if (ck == OUT16) {
                static_cast<uint16_t*>(p.ckv)[row * p.Dv + c] = IT::one_out(y);
            } else {
                y *= p.ckv_scale[p.ckv_scale_per_ch ? c : 0];
                static_cast<uint8_t*>(p.ckv)[row * p.Dv + c] = uint8_t(enc8x2_rt(ck, y, 0.f) & 0xFFu);
            }
        }
        const uint16_t* cr = cosb + t * p.Dk;
        const uint16_t* sr = sinb + t * p.Dk;
        for (int i = lane; i < h; i += 32) {
            const float a = IT::one(x[p.Dv + 2 * i]);
            const float b = IT::one(x[p.Dv + 2 * i + 1]);
            float o1 = a * IT::one(cr[i]) - b * IT::one(sr[i]);
            float o2 = b * IT::one(cr[h + i]) + a * IT::one(sr[h + i]);
            if (p.k_kind == OUT16) {
                static_cast<uint16_t*>(p.kc)[row * p.Dk + i] = IT::one_out(o1);
                static_cast<uint16_t*>(p.kc)[row * p.Dk + h + i] = IT::one_out(o2);
            } else {
                o1 *= p.k_scale[p.k_scale_per_ch ? i : 0];
                o2 *= p.k_scale[p.k_scale_per_ch ? h + i : 0];
                static_cast<uint8_t*>(p.kc)[row * p.Dk + i] = uint8_t(enc8x2_rt(p.k_kind, o1, 0.f) & 0xFFu);
                static_cast<uint8_t*>(p.kc)[row * p.Dk + h + i] = uint8_t(enc8x2_rt(p.k_kind, o2, 0.f) & 0xFFu);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Host launch
// ---------------------------------------------------------------------------

typedef void (*VecKernel)(const KvParams);

template <class IT, int CPL>
static VecKernel pick_ck(int ck) {
    switch (ck) {
        case OUT16: return kv_vec_kernel<IT, CPL, OUT16>;
        case OUT_I8: return kv_vec_kernel<IT, CPL, OUT_I8>;
        case OUT_E4M3: return kv_vec_kernel<IT, CPL, OUT_E4M3>;
        default: return kv_vec_kernel<IT, CPL, OUT_E5M2>;
    }
}

template <class IT>
static VecKernel pick_cpl(int cpl, int ck) {
    if (cpl == 1) return pick_ck<IT, 1>(ck);
    if (cpl == 2) return pick_ck<IT, 2>(ck);
    return pick_ck<IT, 4>(ck);
}

// Resident CTAs per SM for (kernel, dynamic shared memory), computed once and
// cached: later calls (including calls under stream capture) make no query.
// All devices this library runs on are the same architecture.
static int ctas_per_sm(const void* fn, size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<const void*, size_t>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({fn, smem});
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, KV_THREADS, smem) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    cache[{fn, smem}] = n;
    return n;
}

cudaError_t launch_kv(const KvParams& p, int in_dtype, int ckv_kind, bool vec, cudaStream_t s) {
    const int64_t rows_ctas = (p.T + KV_WARPS - 1) / KV_WARPS;
    const int sms = sm_count_current_device();
    if (vec) {
        const int nch = p.Dv / 8;
        const int cpl = nch <= 32 ? 1 : (nch <= 64 ? 2 : 4);
        VecKernel fn = in_dtype == KVR_BF16 ? pick_cpl<BF16>(cpl, ckv_kind) : pick_cpl<F16>(cpl, ckv_kind);
        const size_t smem = size_t(p.Dv) * 2 + size_t(p.Dv) * 4 + size_t(p.Dk) * 4;
        const int64_t cap = int64_t(ctas_per_sm(reinterpret_cast<const void*>(fn), smem)) * sms;
        const int grid = int(rows_ctas < cap ? rows_ctas : cap);
        fn<<<grid, KV_THREADS, smem, s>>>(p);
    } else {
        auto fn = in_dtype == KVR_BF16 ? kv_generic_kernel<BF16> : kv_generic_kernel<F16>;
        const int64_t cap = int64_t(ctas_per_sm(reinterpret_cast<const void*>(fn), 0)) * sms;
        const int grid = int(rows_ctas < cap ? rows_ctas : cap);
        fn<<<grid, KV_THREADS, 0, s>>>(p, ckv_kind);
    }
    return cudaGetLastError();
}

}  // namespace kvr
