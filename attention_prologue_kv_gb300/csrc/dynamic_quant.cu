// DynamicQuant of q^N: per-row symmetric int8 quantisation.
//
// Operation: "aclnnMlaPrologV3WeightNz" (hiascend.com), "Formula":
// dequantScaleQNope = RowMax(abs(q^N)) / 127, q^N = round(q^N / dequantScaleQNope),
// one scale per (token, head) row ("Shape restrictions": (T, N, 1)).
//
// Design: one warp per row, grid-stride, 4 warps per CTA. A lane loads its
// 16-byte chunks of the row; the row max of |q| is a packed 16-bit maximum
// and a warp butterfly (exact); the scale is one IEEE division (the correctly
// rounded float32 value of RowMax/127); each code is the rounded product of
// q and RN(1/scale), within one code of round(q*127/RowMax) and equal to it
// unless q*127/RowMax lies within 2^-15 of a half-integer (dq_chunk_fast).
// With `exact` set, such near-tie elements are recomputed from the exact
// rational (dq_code_exact), so every code is round-half-even(q*127/RowMax).
// Each lane stores 8 codes with one 8-byte store. The first row of each warp
// is prefetched into L2 before the programmatic-dependent-launch wait.
#include <map>
#include <mutex>

#include "kvr_internal.cuh"

namespace kvr {

constexpr int DQ_THREADS = 128;
#ifndef KVR_DQ_SPECIALISE
#define KVR_DQ_SPECIALISE 1
#endif
constexpr int DQ_WARPS = DQ_THREADS / 32;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// round-half-even(x * 127 / m), clamped to [-127, 127], for 16-bit inputs x
// and row maximum m > 0 (else 0). x*127 is exact in float32 (at most 11 + 7
// significant bits) and the IEEE division is correctly rounded: when the
// rational x*127/m is a half-integer the quotient is exactly that value, and
// when it is not, it lies at least 2^-19 (relative) from every half-integer
// (numerator and denominator are short binary numbers), far beyond the
// division's 2^-24 rounding error, so rounding the quotient decides the code
// of the rational itself. Rows with m >= 2^64 are scaled by 2^-64 first
// (exact, or the element is so small that its code is 0 either way), so
// x*127 cannot overflow.
__device__ __forceinline__ int dq_code_exact(float x, float m) {
    if (!(m > 0.f)) return 0;
    if (m >= 0x1p64f) {
        x *= 0x1p-64f;
        m *= 0x1p-64f;
    }
    const int c = __float2int_rn(__fdiv_rn(x * 127.f, m));
    return min(max(c, -127), 127);
}

// Eight codes of one 16-byte chunk at once, packed into 8 bytes, without a
// division per element. With y = RN(1/s) and s = RN(m/127), the product
// q0 = RN(x*y) differs from the rational x*127/m by at most
// (3*2^-24 + O(2^-48))|q0|, i.e. by less than 2^-15.4 for |q0| < 128, so
// rint(q0) is that rational's code, or (within 2^-15.4 of a half-integer)
// its neighbour: at most one code off. With EXACT, bit `base + j` of `near` is
// set for element j when |q0 - rint(q0)| >= 1/2 - 2^-15, and the caller
// recomputes those elements exactly (dq_fix_element).
// Valid while 1/s is a normal float (the caller checks s >= 2^-100).
// Rounding: with M = 1.5 * 2^23, t = fl(q0 + M) rounds q0 (|q0| < 2^22) to an
// integer with ties to even inside the addition, and the low byte of t's bits
// is that integer's two's-complement byte.
template <class IT, bool EXACT>
__device__ __forceinline__ uint2 dq_chunk_fast(const uint4& x, float y, uint32_t& near, int base) {
    const float T = 0.5f - 0x1p-15f;
    const float M = 12582912.0f;
    const float2 y2 = make_float2(y, y), M2 = make_float2(M, M), nM2 = make_float2(-M, -M),
                 m1 = make_float2(-1.f, -1.f);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t b[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 q0 = __fmul2_rn(make_float2(IT::lo(w[k]), IT::hi(w[k])), y2);
        const float2 t = __fadd2_rn(q0, M2);
        if (EXACT) {
            const float2 r = __fadd2_rn(t, nM2);          // rint(q0), exact
            const float2 d = __ffma2_rn(r, m1, q0);       // q0 - r, exact
            near |= (fabsf(d.x) >= T ? 1u : 0u) << (base + 2 * k);
            near |= (fabsf(d.y) >= T ? 1u : 0u) << (base + 2 * k + 1);
        }
        b[k] = __byte_perm(__float_as_uint(t.x), __float_as_uint(t.y), 0x0040);   // two code bytes
    }
    return make_uint2(__byte_perm(b[0], b[1], 0x5410), __byte_perm(b[2], b[3], 0x5410));
}

// The same eight codes, each from the exact rational (rows whose scale is too
// small for the reciprocal).
template <class IT>
__device__ __forceinline__ uint2 dq_chunk_exact(const uint4& x, float m) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t b[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        b[2 * k] = uint32_t(dq_code_exact(IT::lo(w[k]), m)) & 0xFFu;
        b[2 * k + 1] = uint32_t(dq_code_exact(IT::hi(w[k]), m)) & 0xFFu;
    }
    return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24), b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// Recompute one element's code (element e of this lane's chunks: chunk e / 8,
// 16-bit lane e % 8) from the exact rational. The element is picked from the
// registers by selects, so the array never goes to local memory. On
// bfloat16 rows near ties are common (q*127/m is often a dyadic rational):
// 0.2% of elements, but in 59% of warp-rows some lane has one, usually a
// single element.
template <class IT, int CPL>
__device__ __forceinline__ void dq_fix_element(const uint4 (&x)[CPL], int e, float m, uint2 (&o)[CPL]) {
    const int c = e >> 3, w = (e >> 1) & 3;
    uint32_t word = 0;
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) {
        const uint32_t a = w == 0 ? x[cc].x : (w == 1 ? x[cc].y : (w == 2 ? x[cc].z : x[cc].w));
        word = cc == c ? a : word;
    }
    const float v = (e & 1) ? IT::hi(word) : IT::lo(word);
    const uint32_t code = uint32_t(dq_code_exact(v, m)) & 0xFFu;
    const int sh = 8 * (e & 3);
#pragma unroll
    for (int cc = 0; cc < CPL; ++cc) {
        if (cc == c) {
            if (e & 4) o[cc].y = (o[cc].y & ~(0xFFu << sh)) | (code << sh);
            else o[cc].x = (o[cc].x & ~(0xFFu << sh)) | (code << sh);
        }
    }
}

// max(|a|, |b|) over the two 16-bit lanes of w, exact: clear the sign bits and
// take the packed bf16/f16 maximum.
template <class IT>
__device__ __forceinline__ uint32_t absmax2(uint32_t acc, uint32_t w);
template <>
__device__ __forceinline__ uint32_t absmax2<BF16>(uint32_t acc, uint32_t w) {
    w &= 0x7FFF7FFFu;
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&acc), b = *reinterpret_cast<__nv_bfloat162*>(&w);
    __nv_bfloat162 m = __hmax2(a, b);
    return *reinterpret_cast<uint32_t*>(&m);
}
template <>
__device__ __forceinline__ uint32_t absmax2<F16>(uint32_t acc, uint32_t w) {
    w &= 0x7FFF7FFFu;
    __half2 a = *reinterpret_cast<__half2*>(&acc), b = *reinterpret_cast<__half2*>(&w);
    __half2 m = __hmax2(a, b);
    return *reinterpret_cast<uint32_t*>(&m);
}

// Vector path: H % 8 == 0, H <= 256 * CPL, 16-byte aligned rows and outputs
// 8-byte aligned. Rows are double-buffered in registers: the loads of a
// warp's next row are issued before the current row is quantised, so every
// warp keeps two rows (2 KB for H = 512) in flight.
template <class IT, int CPL, int HC, bool EXACT>
__global__ void __launch_bounds__(DQ_THREADS) dq_vec_kernel(const DqParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t H = HC ? HC : p.H;   // row length, a constant when compiled for one
    const int nch = int(H >> 3);
    const int64_t stride_rows = int64_t(gridDim.x) * DQ_WARPS;
    int64_t t = int64_t(blockIdx.x) * DQ_WARPS + (threadIdx.x >> 5);
    if (t < p.rows && lane == 0)
        prefetch_l2_bulk(static_cast<const char*>(p.q) + t * p.q_stride * 2, uint32_t(H) * 2);
    pdl_wait();
    pdl_launch_dependents();
    uint4 x[CPL], nx[CPL];
    auto load = [&](int64_t row, uint4 (&dst)[CPL]) {
        const char* src = static_cast<const char*>(p.q) + row * p.q_stride * 2;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int ch = c * 32 + lane;
            if (ch < nch) dst[c] = ld_stream_v4(src + ch * 16);
        }
    };
    if (t < p.rows) load(t, x);
    for (; t < p.rows; t += stride_rows) {
        if (t + stride_rows < p.rows) load(t + stride_rows, nx);
        uint32_t am = 0;   // packed |q| maxima
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            if (c * 32 + lane < nch) {
                am = absmax2<IT>(am, x[c].x);
                am = absmax2<IT>(am, x[c].y);
                am = absmax2<IT>(am, x[c].z);
                am = absmax2<IT>(am, x[c].w);
            }
        }
        const float m = warp_max(fmaxf(IT::lo(am), IT::hi(am)));
        const float s = __fdiv_rn(m, 127.f);
        const bool fast = s >= 0x1p-100f;
        const float y = fast ? __frcp_rn(s) : 0.f;
        char* dst = reinterpret_cast<char*>(p.out) + t * H;
        uint2 o[CPL];
        uint32_t near = 0;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            if (c * 32 + lane < nch) o[c] = fast ? dq_chunk_fast<IT, EXACT>(x[c], y, near, 8 * c) : dq_chunk_exact<IT>(x[c], m);
        if (EXACT) {
            // Products within 2^-15 of a half-integer: recompute those codes exactly.
            while (near != 0) {
                const int e = __ffs(near) - 1;
                near &= near - 1;
                dq_fix_element<IT, CPL>(x, e, m, o);
            }
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const int ch = c * 32 + lane;
            if (ch < nch) *reinterpret_cast<uint2*>(dst + ch * 8) = o[c];
        }
        if (lane == 0) p.scale[t] = s;
#pragma unroll
        for (int c = 0; c < CPL; ++c) x[c] = nx[c];
    }
}

// Generic path: any H, element-aligned rows; two passes over the row.
template <class IT>
__global__ void __launch_bounds__(DQ_THREADS) dq_generic_kernel(const DqParams p) {
    const int lane = threadIdx.x & 31;
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t t = int64_t(blockIdx.x) * DQ_WARPS + (threadIdx.x >> 5); t < p.rows;
         t += int64_t(gridDim.x) * DQ_WARPS) {
        const uint16_t* src = static_cast<const uint16_t*>(p.q) + t * p.q_stride;
        float m = 0.f;
        for (int64_t c = lane; c < p.H; c += 32) m = fmaxf(m, fabsf(IT::one(src[c])));
        m = warp_max(m);
        const float s = __fdiv_rn(m, 127.f);
        int8_t* dst = p.out + t * p.H;
        for (int64_t c = lane; c < p.H; c += 32) dst[c] = int8_t(dq_code_exact(IT::one(src[c]), m));
        if (lane == 0) p.scale[t] = s;
    }
}

// Resident CTAs per SM of a kernel, queried once per kernel and cached.
static int dq_ctas_per_sm(const void* fn) {
    static std::mutex mu;
    static std::map<const void*, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(fn);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, DQ_THREADS, 0) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        n = 1;
    }
    cache[fn] = n;
    return n;
}

typedef void (*DqKernel)(const DqParams);

// The vector kernel for a row length: compiled row lengths (512 is the MLA
// query's Hckv) fold the per-chunk bounds tests and row offsets.
template <bool EXACT>
static DqKernel pick_dq_vec(bool bf, int64_t H, int cpl) {
    if (KVR_DQ_SPECIALISE && H == 512) return bf ? dq_vec_kernel<BF16, 2, 512, EXACT> : dq_vec_kernel<F16, 2, 512, EXACT>;
    if (KVR_DQ_SPECIALISE && H == 256) return bf ? dq_vec_kernel<BF16, 1, 256, EXACT> : dq_vec_kernel<F16, 1, 256, EXACT>;
    if (KVR_DQ_SPECIALISE && H == 1024) return bf ? dq_vec_kernel<BF16, 4, 1024, EXACT> : dq_vec_kernel<F16, 4, 1024, EXACT>;
    if (bf)
        return cpl == 1 ? dq_vec_kernel<BF16, 1, 0, EXACT>
                        : (cpl == 2 ? dq_vec_kernel<BF16, 2, 0, EXACT> : dq_vec_kernel<BF16, 4, 0, EXACT>);
    return cpl == 1 ? dq_vec_kernel<F16, 1, 0, EXACT>
                    : (cpl == 2 ? dq_vec_kernel<F16, 2, 0, EXACT> : dq_vec_kernel<F16, 4, 0, EXACT>);
}

cudaError_t launch_dq(const DqParams& p, int in_dtype, bool vec, cudaStream_t s) {
    const int64_t ctas = (p.rows + DQ_WARPS - 1) / DQ_WARPS;
    const int sms = sm_count_current_device();
    typedef DqKernel K;
    if (vec) {
        const int nch = int(p.H / 8);
        const int cpl = nch <= 32 ? 1 : (nch <= 64 ? 2 : 4);
        const K fn = p.exact ? pick_dq_vec<true>(in_dtype == KVR_BF16, p.H, cpl)
                             : pick_dq_vec<false>(in_dtype == KVR_BF16, p.H, cpl);
        const int64_t cap = int64_t(dq_ctas_per_sm(reinterpret_cast<const void*>(fn))) * sms;
        return launch_pdl(fn, dim3(int(ctas < cap ? ctas : cap)), dim3(DQ_THREADS), size_t(0), s, p);
    }
    auto fn = in_dtype == KVR_BF16 ? dq_generic_kernel<BF16> : dq_generic_kernel<F16>;
    const int64_t cap = int64_t(dq_ctas_per_sm(reinterpret_cast<const void*>(fn))) * sms;
    return launch_pdl(fn, dim3(int(ctas < cap ? ctas : cap)), dim3(DQ_THREADS), size_t(0), s, p);
}

}  // namespace kvr
