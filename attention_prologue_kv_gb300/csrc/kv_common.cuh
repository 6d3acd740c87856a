// Row mapping shared by the KV prologue kernels: which index entry governs
// a token, and which cache row it names ("aclnnKvRmsNormRopeCache",
// "Restrictions on index").
#pragma once

#include "kvr_internal.cuh"

namespace kvr {

#ifndef KVR_KV_THREADS
#define KVR_KV_THREADS 128
#endif
constexpr int KV_THREADS = KVR_KV_THREADS;
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

// ---------------------------------------------------------------------------
// Per-row arithmetic shared by the vectorised kernels
// ---------------------------------------------------------------------------
//
// Per-channel constants live in shared memory as float, split so that a
// warp reading chunk `ch` (8 channels) on lane ch % 32 is conflict-free:
// lo[ch] = channels 8ch..8ch+3, hi[ch] = channels 8ch+4..8ch+7.
struct ChanF32 {
    const float4* lo;
    const float4* hi;
};

//
// The constants are read with L1-allocating loads: every CTA of a launch
// reads the same few lines, so CTAs sharing an SM then hit in L1 instead of
// all queueing on the same L2 slices (with a thousand CTAs that hot spot cost
// ~1.2 us per launch). `src` is 16-byte aligned (8 floats per chunk).
__device__ __forceinline__ void stage_chan_f32(float4* lo, float4* hi, int nch, const float* src, int tid, int nthr) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
    for (int i = tid; i < nch; i += nthr) {
        lo[i] = __ldg(s4 + 2 * i);
        hi[i] = __ldg(s4 + 2 * i + 1);
    }
}

template <class IT>
__device__ __forceinline__ void stage_gamma(float4* lo, float4* hi, int nch, const void* gamma, int tid, int nthr) {
    for (int i = tid; i < nch; i += nthr) {
        const uint4 g = __ldg(static_cast<const uint4*>(gamma) + i);
        lo[i] = make_float4(IT::lo(g.x), IT::hi(g.x), IT::lo(g.y), IT::hi(g.y));
        hi[i] = make_float4(IT::lo(g.z), IT::hi(g.z), IT::lo(g.w), IT::hi(g.w));
    }
}

// One chunk of 8 inputs: xg = x * gamma (exact in float32 for 16-bit x and
// gamma), and the sum of squares accumulated into acc (two partial sums).
template <class IT>
__device__ __forceinline__ void chunk_xg(const uint4& x, const float4& g0, const float4& g1, float2 (&xg)[4],
                                         float2& acc) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    const float2 g[4] = {make_float2(g0.x, g0.y), make_float2(g0.z, g0.w), make_float2(g1.x, g1.y),
                         make_float2(g1.z, g1.w)};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 xf = make_float2(IT::lo(w[k]), IT::hi(w[k]));
        acc = __ffma2_rn(xf, xf, acc);
        xg[k] = __fmul2_rn(xf, g[k]);
    }
}

// y = xg * rr (* scale) for one chunk, encoded and stored at dst (16 bytes
// for 16-bit caches, 8 bytes for 8-bit codes).
template <class IT, int CK>
__device__ __forceinline__ void chunk_store(char* dst, const float2 (&xg)[4], float rr, const float4* s0,
                                            const float4* s1, float sc) {
    const float2 r2 = make_float2(rr, rr);
    float2 y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = __fmul2_rn(xg[k], r2);
    if constexpr (CK == OUT16) {
        uint4 o;
        o.x = IT::pack(y[0].x, y[0].y);
        o.y = IT::pack(y[1].x, y[1].y);
        o.z = IT::pack(y[2].x, y[2].y);
        o.w = IT::pack(y[3].x, y[3].y);
        *reinterpret_cast<uint4*>(dst) = o;
    } else {
        if (s0 != nullptr) {
            const float4 a = *s0, b = *s1;
            y[0] = __fmul2_rn(y[0], make_float2(a.x, a.y));
            y[1] = __fmul2_rn(y[1], make_float2(a.z, a.w));
            y[2] = __fmul2_rn(y[2], make_float2(b.x, b.y));
            y[3] = __fmul2_rn(y[3], make_float2(b.z, b.w));
        } else {
            const float2 s2 = make_float2(sc, sc);
#pragma unroll
            for (int k = 0; k < 4; ++k) y[k] = __fmul2_rn(y[k], s2);
        }
        uint2 o;
        o.x = enc8x2<CK>(y[0].x, y[0].y) | (enc8x2<CK>(y[1].x, y[1].y) << 16);
        o.y = enc8x2<CK>(y[2].x, y[2].y) | (enc8x2<CK>(y[3].x, y[3].y) << 16);
        *reinterpret_cast<uint2*>(dst) = o;
    }
}

// Interleaved RoPE of pair i (x1 = x[2i], x2 = x[2i+1], packed in xpair):
// out[i] = x1*cos[i] - x2*sin[i], out[i+h] = x2*cos[i+h] + x1*sin[i+h];
// stored (and, for an 8-bit k cache, scaled and encoded) into krow.
template <class IT>
__device__ __forceinline__ void rope_pair_store(void* krow, int i, int h, uint32_t xpair, uint16_t c_lo, uint16_t s_lo,
                                                uint16_t c_hi, uint16_t s_hi, int k_kind, const float* kscale,
                                                float ksc0) {
    const float a = IT::lo(xpair);
    const float b = IT::hi(xpair);
    float o1 = a * IT::one(c_lo) - b * IT::one(s_lo);
    float o2 = b * IT::one(c_hi) + a * IT::one(s_hi);
    if (k_kind == OUT16) {
        static_cast<uint16_t*>(krow)[i] = IT::one_out(o1);
        static_cast<uint16_t*>(krow)[h + i] = IT::one_out(o2);
    } else {
        o1 *= kscale != nullptr ? kscale[i] : ksc0;
        o2 *= kscale != nullptr ? kscale[h + i] : ksc0;
        static_cast<uint8_t*>(krow)[i] = uint8_t(enc8x2_rt(k_kind, o1, 0.f) & 0xFFu);
        static_cast<uint8_t*>(krow)[h + i] = uint8_t(enc8x2_rt(k_kind, o2, 0.f) & 0xFFu);
    }
}

}  // namespace kvr
