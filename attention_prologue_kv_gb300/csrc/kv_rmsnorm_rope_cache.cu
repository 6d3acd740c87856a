// Fused KV prologue kernels: RMSNorm (left Dv) + interleaved RoPE (right Dk)
// + optional 8-bit quantisation + scatter into two caches.
//
// Operation: "aclnnKvRmsNormRopeCache" (hiascend.com), "Description",
// "Formulas (1) interleaveRope", "Formulas (2) rmsNorm", "Restrictions on
// index", "Restrictions on quantization scenarios"; the alpha_kv factor of
// "aclnnMlaPrologV3WeightNz" ("Formula", key path).
//
// Design (memory-bound stream, ~1 flop per byte, no tensor cores):
//  * one warp per token row, grid-stride over rows, grid sized to the
//    resident capacity of the GPU; 2-warp CTAs with gamma in registers for
//    small batches into 16-bit caches (latency), 4-warp CTAs with gamma and
//    the scales staged once per CTA in shared memory otherwise;
//  * before the programmatic-dependent-launch wait each warp prefetches its
//    first row into L2 (one 128-byte line per lane); with params_ready the
//    constants are also read before the wait;
//  * per row every lane issues its loads at once: the int64 index, 16-byte
//    non-caching loads of the Dv part (CPL chunks of 8 elements per lane),
//    and, on the first Dk/2 lanes, one RoPE pair plus its four cos/sin
//    entries;
//  * sum of squares in float32 with a warp butterfly, one rsqrt;
//  * whole cache rows written with 16-byte (8-byte for 8-bit codes) stores:
//    512 contiguous bytes per warp instruction for the Dv part, so every
//    32-byte sector is fully written;
//  * index -1 skips the row; an out-of-range index skips it and raises
//    KVR_DEVERR_INDEX. No atomics touch data.
#include <map>
#include <mutex>
#include <utility>

#include "kv_common.cuh"

// Batches below this many rows (16-bit caches) keep gamma in registers.
#ifndef KVR_REG_GAMMA_MAX_ROWS
#define KVR_REG_GAMMA_MAX_ROWS 2048
#endif

namespace kvr {

// Registers of one row in flight: the index entry, CPL 16-byte chunks of the
// Dv part, and this lane's RoPE pair with its four table entries.
struct RowRegs {
    int64_t v;
    uint4 x[4];
    uint32_t xp;
    uint16_t c0, c1, s0, s1;
};

template <int CPL>
__device__ __forceinline__ void load_row(const KvParams& p, int64_t t, int lane, int nch, int h, int Dv, int Dk,
                                         RowRegs& r) {
    r.v = ld_stream_s64(p.index + index_pos(p, t));
    const char* x = static_cast<const char*>(p.kv) + t * p.kv_stride * 2;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        const int ch = c * 32 + lane;
        if (ch < nch) r.x[c] = ld_stream_v4(x + ch * 16);
    }
    if (lane < h) {
        r.xp = ld_stream_u32(x + int64_t(Dv) * 2 + lane * 4);
        const uint16_t* cr = static_cast<const uint16_t*>(p.cos) + t * Dk;
        const uint16_t* sr = static_cast<const uint16_t*>(p.sin) + t * Dk;
        r.c0 = ld_stream_u16(cr + lane);
        r.c1 = ld_stream_u16(cr + h + lane);
        r.s0 = ld_stream_u16(sr + lane);
        r.s1 = ld_stream_u16(sr + h + lane);
    }
}

// Register path: Dv % 8 == 0 and Dv <= 256*CPL, Dk % 8 == 0, 16-byte aligned
// rows. Every load of a row is issued before any of its results is needed,
// and the next row's loads are issued right after the current row's stores.
// CK = OutKind of ckv. Two flavours for the per-channel constants:
//  * REG_GAMMA (16-bit caches, small batches): gamma lives in registers for
//    the whole kernel; no shared memory and no CTA barrier, so the first row
//    starts as soon as its loads land (lowest latency);
//  * otherwise gamma and the scales are staged once per CTA in shared
//    memory, pre-widened to float (fewest instructions per row).
#ifndef KVR_VEC_SPECIALISE
#define KVR_VEC_SPECIALISE 1
#endif
// Threads per CTA of the shared-memory flavour (its CTAs stage the constants).
#ifndef KVR_VEC_THREADS
#define KVR_VEC_THREADS 128
#endif
#ifndef KVR_VEC_MIN_CTAS
#define KVR_VEC_MIN_CTAS (1024 / KVR_VEC_THREADS)
#endif
// Small batches (the REG_GAMMA flavour) use 2-warp CTAs: the rows spread
// over more SMs, which measured faster for a 256-row decode batch.
template <bool REG_GAMMA>
struct VecShape {
    static constexpr int threads = REG_GAMMA ? 64 : KVR_VEC_THREADS;
    static constexpr int warps = threads / 32;
};

// DV / DK: the row split when fixed at compile time (0: from the parameters).
template <class IT, int CPL, int CK, bool REG_GAMMA, bool PARAMS_READY, int DV = 0, int DK = 0>
__global__ void __launch_bounds__(VecShape<REG_GAMMA>::threads, REG_GAMMA ? 8 : KVR_VEC_MIN_CTAS)
    kv_vec_kernel(const KvParams p) {
    const int Dv = DV ? DV : p.Dv;
    const int Dk = DK ? DK : p.Dk;
    constexpr int WARPS = VecShape<REG_GAMMA>::warps;
    constexpr int THREADS = VecShape<REG_GAMMA>::threads;
    extern __shared__ __align__(16) unsigned char smem[];
    const int nch = Dv >> 3;
    float4* g_lo = reinterpret_cast<float4*>(smem);
    float4* g_hi = g_lo + nch;
    float4* c_lo = g_hi + nch;
    float4* c_hi = c_lo + nch;
    float* s_kscale = reinterpret_cast<float*>(c_hi + nch);

    const int lane = threadIdx.x & 31;
    const int h = Dk >> 1;
    const int64_t stride_rows = int64_t(gridDim.x) * WARPS;
    int64_t t = int64_t(blockIdx.x) * WARPS + (threadIdx.x >> 5);

    // While the preceding grid may still run, start this warp's first row on
    // its way from HBM into L2: one 128-byte line per lane (the kv row, which
    // may straddle one more line than its length, then its cos, sin and
    // index entries). A prefetch moves nothing into registers and L2 is the
    // coherence point, so this is safe before the dependency wait. (Per-line
    // prefetches measured 2% faster per decode call than bulk prefetches.)
    if (t < p.T) {
        const char* kvrow = static_cast<const char*>(p.kv) + t * p.kv_stride * 2;
        const int kb = (Dv + Dk) * 2;
        const int nl = min((kb + 127) / 128 + 1, 29);
        if (lane < nl) prefetch_l2(kvrow + min(lane * 128, kb - 1));
        else if (lane == 29) prefetch_l2(static_cast<const char*>(p.cos) + t * Dk * 2);
        else if (lane == 30) prefetch_l2(static_cast<const char*>(p.sin) + t * Dk * 2);
        else if (lane == 31) prefetch_l2(p.index + index_pos(p, t));
    }
    const bool cper = CK != OUT16 && p.ckv_scale_per_ch;
    const bool kq = p.k_kind != OUT16;
    float cscale0 = 1.f, kscale0 = 1.f;
    uint4 graw[CPL];
    // The launch's constants (gamma and the scales). With PARAMS_READY the
    // caller promises that the kernel launched just before this one does not
    // write them, so they are read before the dependency wait, overlapping
    // that kernel; otherwise after the first row's loads are issued (staging
    // them first would hold the row loads behind the staging stores).
    auto load_consts = [&]() {
        if (CK != OUT16 && !p.ckv_scale_per_ch) cscale0 = p.ckv_scale[0];
        if (kq && !p.k_scale_per_ch) kscale0 = p.k_scale[0];
        if constexpr (REG_GAMMA) {
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = c * 32 + lane;
                if (ch < nch) graw[c] = ld_stream_v4(static_cast<const char*>(p.gamma) + ch * 16);
            }
        } else {
            stage_gamma<IT>(g_lo, g_hi, nch, p.gamma, threadIdx.x, THREADS);
            if (cper) stage_chan_f32(c_lo, c_hi, nch, p.ckv_scale, threadIdx.x, THREADS);
            if (kq && p.k_scale_per_ch)
                for (int i = threadIdx.x; i < Dk; i += THREADS) s_kscale[i] = p.k_scale[i];
        }
    };
    if constexpr (PARAMS_READY) load_consts();
    pdl_wait();
    pdl_launch_dependents();
    if (REG_GAMMA && t >= p.T) return;
    RowRegs r;
    if (t < p.T) load_row<CPL>(p, t, lane, nch, h, Dv, Dk, r);
    if constexpr (!PARAMS_READY) load_consts();
    const float* kscale = (kq && p.k_scale_per_ch) ? (REG_GAMMA ? p.k_scale : s_kscale) : nullptr;
    if constexpr (!REG_GAMMA) __syncthreads();

    while (t < p.T) {
        const int64_t row = resolve_row(p, t, r.v);
        if (row >= 0) {
            float2 xg[CPL][4];
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = c * 32 + lane;
                if (ch < nch) {
                    if constexpr (REG_GAMMA) {
                        const uint4 g = graw[c];
                        chunk_xg<IT>(r.x[c], make_float4(IT::lo(g.x), IT::hi(g.x), IT::lo(g.y), IT::hi(g.y)),
                                     make_float4(IT::lo(g.z), IT::hi(g.z), IT::lo(g.w), IT::hi(g.w)), xg[c], acc);
                    } else {
                        chunk_xg<IT>(r.x[c], g_lo[ch], g_hi[ch], xg[c], acc);
                    }
                }
            }
            const float ss = warp_sum(acc.x + acc.y);
            const float rr = rsqrtf(fmaf(ss, p.inv_dv, p.eps)) * p.alpha;
            char* crow = static_cast<char*>(p.ckv) + row * Dv * (CK == OUT16 ? 2 : 1);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = c * 32 + lane;
                if (ch < nch)
                    chunk_store<IT, CK>(crow + ch * (CK == OUT16 ? 16 : 8), xg[c], rr, cper ? &c_lo[ch] : nullptr,
                                        cper ? &c_hi[ch] : nullptr, cscale0);
            }
            char* krow = static_cast<char*>(p.kc) + row * Dk * (kq ? 1 : 2);
            if (lane < h) rope_pair_store<IT>(krow, lane, h, r.xp, r.c0, r.s0, r.c1, r.s1, p.k_kind, kscale, kscale0);
            for (int i = lane + 32; i < h; i += 32) {
                const char* x = static_cast<const char*>(p.kv) + t * p.kv_stride * 2;
                const uint16_t* cr = static_cast<const uint16_t*>(p.cos) + t * Dk;
                const uint16_t* sr = static_cast<const uint16_t*>(p.sin) + t * Dk;
                rope_pair_store<IT>(krow, i, h, ld_stream_u32(x + int64_t(Dv) * 2 + i * 4), cr[i], sr[i], cr[h + i],
                                    sr[h + i], p.k_kind, kscale, kscale0);
            }
        } else if (row == ROW_BAD && lane == 0 && p.status != nullptr) {
            atomicOr(p.status, KVR_DEVERR_INDEX);
        }
        t += stride_rows;
        if (t < p.T) load_row<CPL>(p, t, lane, nch, h, Dv, Dk, r);
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
    pdl_wait();
    pdl_launch_dependents();
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

// The register-gamma flavour ignores params_ready (the flag permits early
// reads, it does not require them): reading gamma before the dependency wait
// made a back-to-back decode call slower (1.76 vs 1.51 us).
template <class IT, int CPL, bool PR, int DV = 0, int DK = 0>
static VecKernel pick_ck(int ck, bool reg_gamma) {
    switch (ck) {
        case OUT16:
            return reg_gamma ? kv_vec_kernel<IT, CPL, OUT16, true, false, DV, DK>
                             : kv_vec_kernel<IT, CPL, OUT16, false, PR, DV, DK>;
        case OUT_I8: return kv_vec_kernel<IT, CPL, OUT_I8, false, PR, DV, DK>;
        case OUT_E4M3: return kv_vec_kernel<IT, CPL, OUT_E4M3, false, PR, DV, DK>;
        default: return kv_vec_kernel<IT, CPL, OUT_E5M2, false, PR, DV, DK>;
    }
}

template <class IT, bool PR>
static VecKernel pick_cpl_pr(int cpl, int ck, bool reg_gamma) {
    if (cpl == 1) return pick_ck<IT, 1, PR>(ck, reg_gamma);
    if (cpl == 2) return pick_ck<IT, 2, PR>(ck, reg_gamma);
    return pick_ck<IT, 4, PR>(ck, reg_gamma);
}

// The MLA latent split (Dv = 512, Dk = 64) is compiled as constants: the
// chunk bounds tests, the second RoPE loop and the row offsets fold away.
template <class IT>
static VecKernel pick_cpl(int cpl, int ck, bool reg_gamma, bool params_ready, int Dv, int Dk) {
    if (KVR_VEC_SPECIALISE && Dv == 512 && Dk == 64)
        return params_ready ? pick_ck<IT, 2, true, 512, 64>(ck, reg_gamma) : pick_ck<IT, 2, false, 512, 64>(ck, reg_gamma);
    return params_ready ? pick_cpl_pr<IT, true>(cpl, ck, reg_gamma) : pick_cpl_pr<IT, false>(cpl, ck, reg_gamma);
}

// Resident CTAs per SM for (kernel, dynamic shared memory), computed once and
// cached: later calls (including calls under stream capture) make no query.
// All devices this library runs on are the same architecture.
static int ctas_per_sm(const void* fn, size_t smem, int threads = KV_THREADS) {
    static std::mutex mu;
    static std::map<std::pair<const void*, size_t>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({fn, smem});
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    cache[{fn, smem}] = n;
    return n;
}

cudaError_t launch_kv(const KvParams& p, int in_dtype, int ckv_kind, int path, cudaStream_t s) {
    if (path == KV_BULK) return launch_kv_bulk(p, in_dtype, ckv_kind, s);
    const int64_t rows_ctas = (p.T + KV_WARPS - 1) / KV_WARPS;
    const int sms = sm_count_current_device();
    if (path == KV_VEC) {
        const int nch = p.Dv / 8;
        const int cpl = nch <= 32 ? 1 : (nch <= 64 ? 2 : 4);
        // Register-held gamma for small batches into 16-bit caches (latency),
        // shared-memory constants otherwise (instructions per row).
        const bool reg_gamma = ckv_kind == OUT16 && p.T < KVR_REG_GAMMA_MAX_ROWS;
        VecKernel fn = in_dtype == KVR_BF16 ? pick_cpl<BF16>(cpl, ckv_kind, reg_gamma, p.params_ready != 0, p.Dv, p.Dk)
                                            : pick_cpl<F16>(cpl, ckv_kind, reg_gamma, p.params_ready != 0, p.Dv, p.Dk);
        const size_t smem = reg_gamma ? 0 : size_t(p.Dv) * 8 + size_t(p.Dk) * 4;
        const int threads = reg_gamma ? VecShape<true>::threads : VecShape<false>::threads;
        const int64_t ctas = (p.T + threads / 32 - 1) / (threads / 32);
        const int64_t cap = int64_t(ctas_per_sm(reinterpret_cast<const void*>(fn), smem, threads)) * sms;
        const int grid = int(ctas < cap ? ctas : cap);
        return launch_pdl(fn, dim3(grid), dim3(threads), smem, s, p);
    }
    auto fn = in_dtype == KVR_BF16 ? kv_generic_kernel<BF16> : kv_generic_kernel<F16>;
    const int64_t cap = int64_t(ctas_per_sm(reinterpret_cast<const void*>(fn), 0)) * sms;
    const int grid = int(rows_ctas < cap ? rows_ctas : cap);
    return launch_pdl(fn, dim3(grid), dim3(KV_THREADS), size_t(0), s, p, ckv_kind);
}

}  // namespace kvr
