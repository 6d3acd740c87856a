// QSA block-key prepare: one key per key block completed by the new tokens.
//
// Operation: "openvino.opset17.qsa_prepare" (docs.openvino.ai), summary and
// Parameters: block key = mean of the block's key_block_size raw index keys,
// RMS-normalised with k_norm_weight, rotated with the RoPE of the block's
// first token; past tokens of the incomplete block come from the carried
// past_incomplete_raw_keys / past_incomplete_rope. The normalisation and the
// rotation are the rmsNorm / interleaveRope formulas of
// "aclnnKvRmsNormRopeCache" ("Formulas (1)", "Formulas (2)"), the rotation by
// default on the last Dr channels with interleaved pairs (the first Dr
// channels and rotate-half pairs on request). In the concat-output form the
// past block keys are copied from past_block_index_keys first.
//
// Design: one warp or CTA per (sequence, candidate block); it reads
// key_length on the device, derives the past length P = K - L, and exits at
// once if its block is not completed by this call (no host sync). Three
// variants:
//  * qsa_warp_kernel (Di in {64, 128, 256}, kbs in {32, 64, 128}, 16-byte
//    aligned; described at its definition): one warp per candidate;
//  * qsa_bulk_kernel (other 16-byte-aligned shapes up to 96 KB of rows): 128
//    threads; before the dependency wait the CTA prefetches its slice of
//    new keys into L2; after it, thread 0 reads key_length, derives the
//    block's scalars once and pulls the block's rows, its first token's
//    cos/sin and k_norm_weight into shared memory with bulk copies on one
//    mbarrier; the CTA then sums the rows from shared memory;
//  * qsa_kernel (any shape): 256 threads, each keeping kbs/G independent
//    loads of a (row group g, channel chunk c) slice in flight.
// The CTA variants reduce the G partial rows in shared memory (the warp
// variant by shuffles), then take the mean, the sum of squares, the rotation
// and one rounding to the output type; the 2*Di-byte key row is written
// once. One extra CTA (warp) per sequence writes the optional carry outputs,
// and in the concat-output form `ncopy` more copy its past block-key rows.
#include <mutex>
#include <set>

#include "kvr_internal.cuh"

namespace kvr {

constexpr int QSA_THREADS = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    if (threadIdx.x < 32) {
        float x = threadIdx.x < QSA_THREADS / 32 ? red[threadIdx.x] : 0.f;
        x = warp_sum(x);
        if (threadIdx.x == 0) red[QSA_THREADS / 32] = x;
    }
    __syncthreads();
    return red[QSA_THREADS / 32];
}

// Lanes (within the rotated channels) of pair member a and b for output lane
// i in [0, Dr): pair q = i mod Dr/2 is (2q, 2q+1) interleaved or (q, q+Dr/2)
// rotate-half; lane i < Dr/2 takes a*cos - b*sin, the rest b*cos + a*sin.
__device__ __forceinline__ void rope_pair_lanes(int i, int h, int half, int& la, int& lb) {
    const int q = i < h ? i : i - h;
    la = half ? q : 2 * q;
    lb = half ? q + h : 2 * q + 1;
}

// Concat-output form: copy CTA `c` of sequence n copies past block-key rows
// [c*copy_rows, (c+1)*copy_rows) below min(Bp, floor(P/kbs), Bcap).
__device__ __forceinline__ void copy_past_block_keys(const QsaParams& p, int64_t n, int64_t c, int64_t j0,
                                                     int tid, int nthreads) {
    const int64_t lim = min(min(p.Bp, j0), p.Bcap);
    const int64_t r0 = c * p.copy_rows;
    const int64_t r1 = min(r0 + int64_t(p.copy_rows), lim);
    if (r1 <= r0) return;
    const int64_t row_b = int64_t(p.Di) * 2;
    const char* src = static_cast<const char*>(p.past_bk) + (n * p.Bp + r0) * row_b;
    char* dst = static_cast<char*>(p.block_keys) + (n * p.Bcap + r0) * row_b;
    const int64_t bytes = (r1 - r0) * row_b;
    if (p.copy_vec) {
#pragma unroll 8
        for (int64_t e = tid; e < (bytes >> 4); e += nthreads)
            reinterpret_cast<uint4*>(dst)[e] = ld_stream_v4(src + 16 * e);
    } else {
        for (int64_t e = tid; e < (bytes >> 1); e += nthreads)
            reinterpret_cast<uint16_t*>(dst)[e] = reinterpret_cast<const uint16_t*>(src)[e];
    }
}

// Status bits of the concat-output form for sequence n (one thread).
__device__ __forceinline__ void past_block_status(const QsaParams& p, int64_t j0) {
    if (p.past_bk == nullptr || p.status == nullptr) return;
    if (p.Bp < j0) atomicOr(p.status, KVR_DEVERR_PAST_BLOCKS);
    if (min(p.Bp, j0) > p.Bcap) atomicOr(p.status, KVR_DEVERR_BLOCK_CAP);
}

template <class IT, int VW>
__device__ __forceinline__ void accumulate(const uint16_t* src, float* acc) {
    if constexpr (VW == 8) {
        const uint4 v = ld_stream_v4(src);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc[2 * k] += IT::lo(w[k]);
            acc[2 * k + 1] += IT::hi(w[k]);
        }
    } else {
        acc[0] += IT::one(*src);
    }
}

template <class IT, int VW>
__global__ void __launch_bounds__(QSA_THREADS) qsa_kernel(const QsaParams p) {
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const int64_t per_seq = p.nbmax + 1 + p.ncopy;
    const int64_t n = int64_t(blockIdx.x) / per_seq;
    const int64_t jl = int64_t(blockIdx.x) - n * per_seq;

    pdl_wait();
    pdl_launch_dependents();
    const int64_t K = p.key_length[p.key_length_per_seq ? n : 0];
    const int64_t P = K - p.L;
    if (P < 0) {
        if (jl == 0 && tid == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_KEY_LENGTH);
        return;
    }
    const int64_t kbs = p.kbs;
    const int64_t F = P - P % kbs;            // first token of the incomplete block
    const int64_t j0 = P / kbs;
    const int64_t nb = K / kbs - j0;          // blocks completed by this call
    const int Di = p.Di;
    const uint16_t* raw = static_cast<const uint16_t*>(p.raw) + n * p.L * Di;
    const uint16_t* past = static_cast<const uint16_t*>(p.past_raw) + n * (kbs - 1) * Di;

    if (jl > p.nbmax) {
        copy_past_block_keys(p, n, jl - p.nbmax - 1, j0, tid, QSA_THREADS);
        return;
    }
    if (jl == p.nbmax) {
        if (tid == 0) past_block_status(p, j0);
        // ---- carry outputs: tokens after the last completed block ----
        const int64_t Fn = (K / kbs) * kbs;
        const int64_t rem = K - Fn;
        if (p.next_raw != nullptr) {
            uint16_t* dst = static_cast<uint16_t*>(p.next_raw) + n * (kbs - 1) * Di;
            for (int64_t e = tid; e < rem * Di; e += QSA_THREADS) {
                const int64_t r = e / Di, ch = e - r * Di;
                const int64_t tok = Fn + r;
                dst[e] = tok < P ? past[(tok - F) * Di + ch] : raw[(tok - P) * Di + ch];
            }
        }
        if (p.next_rope != nullptr && p.Dr > 0 && rem > 0) {
            uint16_t* dst = static_cast<uint16_t*>(p.next_rope) + n * 2 * p.Dr;
            for (int e = tid; e < 2 * p.Dr; e += QSA_THREADS) {
                uint16_t v;
                if (Fn >= P) {
                    const int64_t row = (n * p.L + (Fn - P)) * p.Dr;
                    v = e < p.Dr ? static_cast<const uint16_t*>(p.cos)[row + e]
                                 : static_cast<const uint16_t*>(p.sin)[row + e - p.Dr];
                } else {
                    v = static_cast<const uint16_t*>(p.past_rope)[n * 2 * p.Dr + e];
                }
                dst[e] = v;
            }
        }
        return;
    }
    if (jl >= nb) return;
    const int64_t j = j0 + jl;
    if (j >= p.Bcap) {
        if (tid == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_BLOCK_CAP);
        return;
    }
    const int64_t tok0 = j * kbs;

    // ---- block sum: thread (g, c) sums rows g, g+G, ... of chunk c ----
    const int C = Di / VW;
    const int G = C >= QSA_THREADS ? 1 : QSA_THREADS / C;
    float* part = sm;                 // [G][Di]
    float* u = sm + G * Di;           // [Di]
    float* red = u + Di;              // [QSA_THREADS/32 + 1]
    for (int cbase = 0; cbase < (C > QSA_THREADS ? C : 1); cbase += QSA_THREADS) {
        const int c = C >= QSA_THREADS ? cbase + tid : tid % C;
        const int g = C >= QSA_THREADS ? 0 : tid / C;
        if (c < C && g < G) {
            float acc[VW];
#pragma unroll
            for (int k = 0; k < VW; ++k) acc[k] = 0.f;
#pragma unroll 4
            for (int64_t r = g; r < kbs; r += G) {
                const int64_t tok = tok0 + r;
                const uint16_t* src = tok < P ? past + (tok - F) * Di : raw + (tok - P) * Di;
                accumulate<IT, VW>(src + c * VW, acc);
            }
#pragma unroll
            for (int k = 0; k < VW; ++k) part[g * Di + c * VW + k] = acc[k];
        }
    }
    __syncthreads();

    // ---- mean, optional RMS normalisation ----
    float ss = 0.f;
    for (int ch = tid; ch < Di; ch += QSA_THREADS) {
        float s = 0.f;
        for (int g = 0; g < G; ++g) s += part[g * Di + ch];
        const float m = s / float(kbs);
        u[ch] = m;
        ss = fmaf(m, m, ss);
    }
    if (p.w != nullptr) {
        const float tot = block_sum(ss, red);
        const float rr = rsqrtf(fmaf(tot, p.inv_di, p.eps));
        const uint16_t* w = static_cast<const uint16_t*>(p.w);
        for (int ch = tid; ch < Di; ch += QSA_THREADS) u[ch] = u[ch] * rr * IT::one(w[ch]);
    }
    __syncthreads();

    // ---- rotation with the first token's RoPE, write ----
    const uint16_t* cr = nullptr;
    const uint16_t* sr = nullptr;
    if (p.Dr > 0) {
        if (tok0 >= P) {
            cr = static_cast<const uint16_t*>(p.cos) + (n * p.L + (tok0 - P)) * p.Dr;
            sr = static_cast<const uint16_t*>(p.sin) + (n * p.L + (tok0 - P)) * p.Dr;
        } else {
            cr = static_cast<const uint16_t*>(p.past_rope) + n * 2 * p.Dr;
            sr = cr + p.Dr;
        }
    }
    const int base = p.rope_first ? 0 : Di - p.Dr;
    const int h = p.Dr >> 1;
    uint16_t* out = static_cast<uint16_t*>(p.block_keys) + (n * p.Bcap + j) * Di;
    for (int ch = tid; ch < Di; ch += QSA_THREADS) {
        float v;
        const int i = ch - base;                  // table lane in [0, Dr) when rotated
        if (unsigned(i) >= unsigned(p.Dr)) {
            v = u[ch];
        } else {
            int la, lb;
            rope_pair_lanes(i, h, p.rope_half, la, lb);
            const float a = u[base + la];
            const float b = u[base + lb];
            const float c = IT::one(cr[i]);
            const float s = IT::one(sr[i]);
            v = i < h ? a * c - b * s : b * c + a * s;
        }
        out[ch] = IT::one_out(v);
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy variant: the block's kbs rows (carried rows, then new rows: each
// run contiguous) and its first token's cos/sin arrive in shared memory by
// a few bulk copies (with k_norm_weight), so every block's bytes are
// requested at once and the whole problem is one wave of loads. Needs
// Di % 8 == 0, Dr % 8 == 0, 16-byte aligned bases and about kbs*Di*2 bytes
// of shared memory.
// ---------------------------------------------------------------------------

#ifndef KVR_QSA_RAW_PREFETCH
#define KVR_QSA_RAW_PREFETCH 1
#endif
#ifndef KVR_QSA_KL_PREFETCH
#define KVR_QSA_KL_PREFETCH 1
#endif
// Suspend-time hint (ns) of thread 0's polls of the copy barrier.
#ifndef KVR_QSA_WAIT_SLEEP_NS
#define KVR_QSA_WAIT_SLEEP_NS 128
#endif
#ifndef KVR_QSA_BULK_THREADS
#define KVR_QSA_BULK_THREADS 128
#endif
constexpr int QSA_BULK_THREADS = KVR_QSA_BULK_THREADS;

// DI / KBS: the key width and block size when fixed at compile time (0: read
// from the parameters). Only the runtime-shape form is instantiated: the
// compiled shapes take the warp kernel below.
template <class IT, int DI, int KBS>
__global__ void __launch_bounds__(QSA_BULK_THREADS) qsa_bulk_kernel(const QsaParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    const int Di = DI ? DI : p.Di;
    const int64_t kbs = KBS ? KBS : p.kbs;
    unsigned char* rows_s = smem + 128;                                      // kbs x Di 16-bit
    uint16_t* w_s = reinterpret_cast<uint16_t*>(rows_s + kbs * Di * 2);      // k_norm_weight [Di]
    uint16_t* rope_s = w_s + Di;                                             // [cos | sin] of the first token
    const int C = Di / 8;
    const int G = C >= QSA_BULK_THREADS ? 1 : QSA_BULK_THREADS / C;
    float* part = reinterpret_cast<float*>(rope_s + 2 * p.Dr + 8);          // [G][Di]
    float* u = part + G * Di;                                                // [Di]
    float* red = u + Di;                                                     // [QSA_BULK_THREADS/32 + 1]
    const int tid = threadIdx.x;

    // This CTA's candidate (sequence n, local block jl); 32-bit: the grid has
    // fewer than 2^31 CTAs.
    const uint32_t per_seq = uint32_t(p.nbmax + 1 + p.ncopy);
    const uint32_t n32 = blockIdx.x / per_seq;
    const int64_t n = n32;
    const int64_t jl = int64_t(blockIdx.x - n32 * per_seq);
    // The block's scalars, derived once by thread 0 (a 64-bit division is a
    // long instruction sequence) and shared.
    __shared__ int64_t sc[5];   // K, P, first block j0, completed blocks nb, status
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
#if KVR_QSA_RAW_PREFETCH
        // New-key rows [jl*kbs, (jl+1)*kbs) on their way into L2 while
        // key_length is read: the block this CTA computes starts P mod kbs
        // rows earlier, but the union over the sequence's CTAs covers every
        // row a completed block reads. (A prefetch is only a hint; L2 is the
        // coherence point, so it is safe before the dependency wait.)
        if (jl < p.nbmax) {
            const int64_t r0 = jl * kbs;
            const int64_t nr = min(kbs, p.L - r0);
            prefetch_l2_bulk(static_cast<const uint16_t*>(p.raw) + (n * p.L + r0) * Di, uint32_t(nr * Di * 2));
        }
#endif
#if KVR_QSA_KL_PREFETCH
        // The sequence's key_length entry, by its first CTA only (every CTA
        // of the sequence reads it; one prefetch per sequence avoids a hot
        // spot on its L2 line).
        if (jl == 0) prefetch_l2(p.key_length + (p.key_length_per_seq ? n : 0));
#endif
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) {
        const int64_t Kv = p.key_length[p.key_length_per_seq ? n : 0];
        const int64_t Pv = Kv - p.L;
        sc[0] = Kv;
        sc[1] = Pv;
        if (Pv >= 0) {
            const int64_t j0v = Pv / kbs;
            sc[2] = j0v;
            sc[3] = Kv / kbs - j0v;
        }
    }
    __syncthreads();
    const int64_t K = sc[0];
    const int64_t P = sc[1];
    if (P < 0) {
        if (jl == 0 && tid == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_KEY_LENGTH);
        return;
    }
    const int64_t j0 = sc[2];
    const int64_t nb = sc[3];
    const int64_t F = j0 * kbs;                  // first token of the incomplete block
    const uint16_t* raw = static_cast<const uint16_t*>(p.raw) + n * p.L * Di;
    const uint16_t* past = static_cast<const uint16_t*>(p.past_raw) + n * (kbs - 1) * Di;

    if (jl > p.nbmax) {
        copy_past_block_keys(p, n, jl - p.nbmax - 1, j0, tid, QSA_BULK_THREADS);
        return;
    }
    if (jl == p.nbmax) {
        if (tid == 0) past_block_status(p, j0);
        // carry outputs (small; plain loads and stores)
        const int64_t Fn = (j0 + nb) * kbs;
        const int rem = int(K - Fn);
        if (p.next_raw != nullptr) {
            uint16_t* dst = static_cast<uint16_t*>(p.next_raw) + n * (kbs - 1) * Di;
            for (int r = 0; r < rem; ++r) {
                const int64_t tok = Fn + r;
                const uint16_t* src = tok < P ? past + (tok - F) * Di : raw + (tok - P) * Di;
                for (int ch = tid; ch < Di; ch += QSA_BULK_THREADS) dst[int64_t(r) * Di + ch] = src[ch];
            }
        }
        if (p.next_rope != nullptr && p.Dr > 0 && rem > 0) {
            uint16_t* dst = static_cast<uint16_t*>(p.next_rope) + n * 2 * p.Dr;
            for (int e = tid; e < 2 * p.Dr; e += QSA_BULK_THREADS) {
                uint16_t v;
                if (Fn >= P) {
                    const int64_t row = (n * p.L + (Fn - P)) * p.Dr;
                    v = e < p.Dr ? static_cast<const uint16_t*>(p.cos)[row + e]
                                 : static_cast<const uint16_t*>(p.sin)[row + e - p.Dr];
                } else {
                    v = static_cast<const uint16_t*>(p.past_rope)[n * 2 * p.Dr + e];
                }
                dst[e] = v;
            }
        }
        return;
    }
    if (jl >= nb) return;
    const int64_t j = j0 + jl;
    if (j >= p.Bcap) {
        if (tid == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_BLOCK_CAP);
        return;
    }
    const int64_t tok0 = j * kbs;
    const int64_t n_past = tok0 < P ? P - tok0 : 0;   // only the first block can hold carried rows
    const int64_t n_new = kbs - n_past;
    const uint32_t row_b = uint32_t(Di) * 2;

    if (tid == 0) {
        const uint32_t rope_b = uint32_t(p.Dr) * 2;
        const uint32_t w_b = p.w != nullptr ? row_b : 0;
        mbar_arrive_expect_tx(bar, uint32_t(kbs) * row_b + 2 * rope_b + w_b);
        if (w_b) bulk_g2s(w_s, p.w, w_b, bar);
        if (n_past > 0) bulk_g2s(rows_s, past + (tok0 - F) * Di, uint32_t(n_past) * row_b, bar);
        bulk_g2s(rows_s + n_past * row_b, raw + (tok0 + n_past - P) * Di, uint32_t(n_new) * row_b, bar);
        if (p.Dr > 0) {
            if (tok0 >= P) {
                const int64_t row = (n * p.L + (tok0 - P)) * p.Dr;
                bulk_g2s(rope_s, static_cast<const uint16_t*>(p.cos) + row, rope_b, bar);
                bulk_g2s(rope_s + p.Dr, static_cast<const uint16_t*>(p.sin) + row, rope_b, bar);
            } else {
                bulk_g2s(rope_s, static_cast<const uint16_t*>(p.past_rope) + n * 2 * p.Dr, 2 * rope_b, bar);
            }
        }
    }
    // Thread 0 waits for the copies; the rest of the CTA sleeps in the barrier
    // (which also orders thread 0's observation before every thread's reads).
    __shared__ int timed_out;
    if (tid == 0) {
        timed_out = 0;
        if (!mbar_wait(bar, 0, nullptr, KVR_QSA_WAIT_SLEEP_NS)) {
            timed_out = 1;
            if (p.status != nullptr) atomicOr(p.status, KVR_DEVERR_TIMEOUT);
            mbar_wait(bar, 0, nullptr);   // the copies must land before the CTA exits
        }
    }
    __syncthreads();
    if (timed_out) return;

    // ---- block sum from shared memory: thread (g, c) sums rows g, g+G, ... of chunk c ----
    for (int cbase = 0; cbase < (C > QSA_BULK_THREADS ? C : 1); cbase += QSA_BULK_THREADS) {
        const int c = C >= QSA_BULK_THREADS ? cbase + tid : tid % C;
        const int g = C >= QSA_BULK_THREADS ? 0 : tid / C;
        if (c < C && g < G) {
            float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                             make_float2(0.f, 0.f)};
            const unsigned char* src = rows_s + c * 16;
            const int nrow = int(kbs);
#pragma unroll 4
            for (int r = g; r < nrow; r += G) {
                const uint4 v = *reinterpret_cast<const uint4*>(src + r * row_b);
                acc[0] = __fadd2_rn(acc[0], make_float2(IT::lo(v.x), IT::hi(v.x)));
                acc[1] = __fadd2_rn(acc[1], make_float2(IT::lo(v.y), IT::hi(v.y)));
                acc[2] = __fadd2_rn(acc[2], make_float2(IT::lo(v.z), IT::hi(v.z)));
                acc[3] = __fadd2_rn(acc[3], make_float2(IT::lo(v.w), IT::hi(v.w)));
            }
            float4* dst = reinterpret_cast<float4*>(part + g * Di + c * 8);
            dst[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
            dst[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
        }
    }
    __syncthreads();

    // ---- mean, optional RMS normalisation ----
    float ss = 0.f;
    for (int ch = tid; ch < Di; ch += QSA_BULK_THREADS) {
        float s = 0.f;
        for (int g = 0; g < G; ++g) s += part[g * Di + ch];
        const float m = s * p.inv_kbs;
        u[ch] = m;
        ss = fmaf(m, m, ss);
    }
    if (p.w != nullptr) {
        float v = warp_sum(ss);
        if ((tid & 31) == 0) red[tid >> 5] = v;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < QSA_BULK_THREADS / 32; ++w) tot += red[w];
        const float rr = rsqrtf(fmaf(tot, p.inv_di, p.eps));
        for (int ch = tid; ch < Di; ch += QSA_BULK_THREADS) u[ch] = u[ch] * rr * IT::one(w_s[ch]);
    }
    __syncthreads();

    // ---- rotation of the layout's Dr channels, one rounding, write the key row ----
    const int base = p.rope_first ? 0 : Di - p.Dr;
    const int h = p.Dr >> 1;
    uint16_t* out = static_cast<uint16_t*>(p.block_keys) + (n * p.Bcap + j) * Di;
    for (int ch = tid; ch < Di; ch += QSA_BULK_THREADS) {
        float v;
        const int i = ch - base;
        if (unsigned(i) >= unsigned(p.Dr)) {
            v = u[ch];
        } else {
            int la, lb;
            rope_pair_lanes(i, h, p.rope_half, la, lb);
            const float a = u[base + la];
            const float b = u[base + lb];
            const float c = IT::one(rope_s[i]);
            const float s = IT::one(rope_s[p.Dr + i]);
            v = i < h ? a * c - b * s : b * c + a * s;
        }
        out[ch] = IT::one_out(v);
    }
}

// ---------------------------------------------------------------------------
// Warp variant for the compile-time shapes (DI, KBS): one warp per
// candidate, QSA_WARP_TASKS independent warps per CTA, no shared-memory
// staging and no CTA barrier. A call's warps hold few registers and almost
// no shared memory, so the next call's warps become resident (and issue
// their L2 prefetches) while this call still runs. Lane (g, c) sums rows
// g, g+G, ... of 16-byte chunk c straight from global memory; the loads are
// issued in batches of 16 rows, so a lane keeps up to 16 loads in flight.
// The G partial rows meet by warp shuffles; the key row is written by the
// lanes of group 0 as 16-byte stores. Needs Di % 8 == 0, Dr % 8 == 0 and
// 16-byte aligned bases (as the bulk variant).
//
// Default form: before the dependency wait each block warp reads key_length
// with a relaxed load as a hint (the preceding grid may still be writing
// it), derives the block the hint gives it and prefetches exactly that
// block's rows, carried rows, first-token cos/sin and, once per sequence,
// k_norm_weight into L2. Issuing the row prefetch only once the hint has
// arrived, rather than at the warp's start, leaves the DRAM queues to the
// running call's own loads a little longer: on the 32 x 2048-token workload
// a call went from 4.6 to 3.4 us. After the wait the warp loads the real
// key_length together with the hinted block's data, sums the rows, and
// compares the two key lengths before anything is written; if they differ
// it starts over from the real one. Every address taken from the hint is
// bounds-checked, so a stale or torn hint costs time, never correctness.
//
// PR (params_ready): the caller promises that the kernel launched just
// before does not write key_length, the RoPE tables, past_incomplete_rope
// or k_norm_weight. The warp then reads key_length, derives its block,
// loads the block's cos/sin and weight chunk and prefetches exactly the
// block's rows into L2 before the dependency wait; after the wait only the
// row loads remain on its path. Outputs and status bits are written after
// the wait in both forms.
// ---------------------------------------------------------------------------

#ifndef KVR_QSA_WARP
#define KVR_QSA_WARP 1
#endif
// Warps (candidates) per CTA: 4 measured faster than 1, 2 or 8.
constexpr int QSA_WARP_TASKS = 4;

// Scalars of sequence n: K = key_length, past length P = K - L (-1 when
// K < L), first block j0 = floor(P / KBS) and the number nb of blocks
// completed by the call.
struct QsaSeq {
    int64_t K, P, j0, nb;
};
template <int KBS>
__device__ __forceinline__ QsaSeq qsa_seq_of(const QsaParams& p, int64_t K) {
    QsaSeq q;
    q.K = K;
    q.P = K >= p.L ? K - p.L : -1;
    q.j0 = q.P >= 0 ? q.P / KBS : 0;
    q.nb = q.P >= 0 ? q.K / KBS - q.j0 : 0;
    return q;
}
template <int KBS>
__device__ __forceinline__ QsaSeq qsa_seq(const QsaParams& p, int64_t n) {
    return qsa_seq_of<KBS>(p, p.key_length[p.key_length_per_seq ? n : 0]);
}

// A relaxed (morally strong) read, for the key_length hint taken before the
// dependency wait.
__device__ __forceinline__ int64_t ld_relaxed_s64(const int64_t* ptr) {
    int64_t v;
    asm volatile("ld.relaxed.gpu.global.s64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
    return v;
}

// The first token's cos/sin for chunk c (when it lies in the rotated
// channels) and the chunk's k_norm_weight.
template <int DI>
__device__ __forceinline__ void qsa_chunk_consts(const QsaParams& p, int64_t n, int64_t tok0, int64_t P, int c,
                                                 uint4& cv, uint4& sv, uint4& wv) {
    const int base = p.rope_first ? 0 : DI - p.Dr;
    const int i0 = c * 8 - base;
    if (p.Dr > 0 && unsigned(i0) < unsigned(p.Dr)) {
        const uint16_t* cr;
        const uint16_t* sr;
        if (tok0 >= P) {
            cr = static_cast<const uint16_t*>(p.cos) + (n * p.L + (tok0 - P)) * p.Dr;
            sr = static_cast<const uint16_t*>(p.sin) + (n * p.L + (tok0 - P)) * p.Dr;
        } else {
            cr = static_cast<const uint16_t*>(p.past_rope) + n * 2 * p.Dr;
            sr = cr + p.Dr;
        }
        cv = ld_stream_v4(cr + i0);
        sv = ld_stream_v4(sr + i0);
    }
    if (p.w != nullptr) wv = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.w) + c * 8);
}

// L2 prefetch of block jl of sequence n for the scalars q (lane 0 only): its
// new and carried rows and, with ROPE, its first token's cos/sin (or the
// carried RoPE row). The caller has checked q.P >= 0, jl < q.nb and
// q.j0 + jl < Bcap, which keeps every address inside the inputs.
template <int DI, int KBS, bool ROPE>
__device__ __forceinline__ void qsa_prefetch_block(const QsaParams& p, const QsaSeq& q, int64_t n, int64_t jl,
                                                   const uint16_t* raw, const uint16_t* past) {
    const int64_t tok0 = (q.j0 + jl) * KBS;
    const int n_past = tok0 < q.P ? int(q.P - tok0) : 0;
    prefetch_l2_bulk(raw + (tok0 + n_past - q.P) * DI, uint32_t(KBS - n_past) * DI * 2);
    if (n_past > 0) prefetch_l2_bulk(past, uint32_t(n_past) * DI * 2);
    if (ROPE && p.Dr > 0) {
        if (tok0 >= q.P) {
            prefetch_l2(static_cast<const uint16_t*>(p.cos) + (n * p.L + (tok0 - q.P)) * p.Dr);
            prefetch_l2(static_cast<const uint16_t*>(p.sin) + (n * p.L + (tok0 - q.P)) * p.Dr);
        } else {
            prefetch_l2_bulk(static_cast<const uint16_t*>(p.past_rope) + n * 2 * p.Dr, uint32_t(p.Dr) * 4);
        }
    }
}

// Block jl of sequence n from its scalars q: the row sum (RB loads in flight
// per lane), mean, normalisation, rotation and the 16-byte stores of the key
// row by the lanes of group 0. LOADC: load the cos/sin and weight chunk here
// (otherwise cv, sv, wv hold them). With `verify`, q came from a key_length
// hint: once the rows are summed, q.K is compared with the real key_length
// Kt, and on a mismatch nothing is written and false is returned.
template <class IT, int DI, int KBS, int RB, bool LOADC>
__device__ __forceinline__ bool qsa_warp_block(const QsaParams& p, const QsaSeq& q, int64_t n, int64_t jl,
                                               const uint16_t* raw, const uint16_t* past, int c, int g, float* u,
                                               uint4 cv, uint4 sv, uint4 wv, bool verify, int64_t Kt) {
    constexpr int C = DI / 8;
    constexpr int G = 32 / C;
    constexpr int NR = KBS / G;
    static_assert(NR % RB == 0, "row batches must tile the block");
    const int64_t P = q.P;
    const int64_t j = q.j0 + jl;
    const int64_t tok0 = j * KBS;
    // Rows r < n_past are carried (past row r: only the first block can hold
    // them); row r >= n_past is new row (tok0 - P) + r.
    const int n_past = tok0 < P ? int(P - tok0) : 0;
    const int64_t off = (tok0 - P) * DI;
    if (LOADC) qsa_chunk_consts<DI>(p, n, tok0, P, c, cv, sv, wv);

    // ---- block sum ----
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int b = 0; b < NR; b += RB) {
        uint4 v[RB];
#pragma unroll
        for (int k = 0; k < RB; ++k) {
            const int r = g + G * (b + k);
            const uint16_t* src = r < n_past ? past + r * DI : raw + (off + int64_t(r) * DI);
            v[k] = ld_stream_v4(src + c * 8);
        }
#pragma unroll
        for (int k = 0; k < RB; ++k) {
            acc[0] = __fadd2_rn(acc[0], make_float2(IT::lo(v[k].x), IT::hi(v[k].x)));
            acc[1] = __fadd2_rn(acc[1], make_float2(IT::lo(v[k].y), IT::hi(v[k].y)));
            acc[2] = __fadd2_rn(acc[2], make_float2(IT::lo(v[k].z), IT::hi(v[k].z)));
            acc[3] = __fadd2_rn(acc[3], make_float2(IT::lo(v[k].w), IT::hi(v[k].w)));
        }
    }
    if (verify && Kt != q.K) return false;   // the same value in every lane
    float m[8] = {acc[0].x, acc[0].y, acc[1].x, acc[1].y, acc[2].x, acc[2].y, acc[3].x, acc[3].y};
#pragma unroll
    for (int o = C; o < 32; o <<= 1)
#pragma unroll
        for (int k = 0; k < 8; ++k) m[k] += __shfl_xor_sync(0xFFFFFFFFu, m[k], o);

    // ---- mean, optional RMS normalisation (every group holds the whole row) ----
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m[k] *= p.inv_kbs;
        ss = fmaf(m[k], m[k], ss);
    }
    if (p.w != nullptr) {
#pragma unroll
        for (int o = 1; o < C; o <<= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
        const float rr = rsqrtf(fmaf(ss, p.inv_di, p.eps));
        const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m[2 * k] = m[2 * k] * rr * IT::lo(ww[k]);
            m[2 * k + 1] = m[2 * k + 1] * rr * IT::hi(ww[k]);
        }
    }

    // ---- rotation of the layout's Dr channels, one rounding, write ----
    const int base = p.rope_first ? 0 : DI - p.Dr;
    const int i0 = c * 8 - base;               // table lane of the chunk's first channel
    if (g == 0 && p.Dr > 0) {
        reinterpret_cast<float4*>(u + c * 8)[0] = make_float4(m[0], m[1], m[2], m[3]);
        reinterpret_cast<float4*>(u + c * 8)[1] = make_float4(m[4], m[5], m[6], m[7]);
    }
    __syncwarp();
    if (g != 0) return true;
    if (p.Dr > 0 && unsigned(i0) < unsigned(p.Dr)) {
        const int h = p.Dr >> 1;
        const uint32_t cw[4] = {cv.x, cv.y, cv.z, cv.w};
        const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + k;
            int la, lb;
            rope_pair_lanes(i, h, p.rope_half, la, lb);
            const float a = u[base + la];
            const float bb = u[base + lb];
            const float cs = (k & 1) ? IT::hi(cw[k >> 1]) : IT::lo(cw[k >> 1]);
            const float sn = (k & 1) ? IT::hi(sw[k >> 1]) : IT::lo(sw[k >> 1]);
            m[k] = i < h ? a * cs - bb * sn : bb * cs + a * sn;
        }
    }
    uint16_t* out = static_cast<uint16_t*>(p.block_keys) + (n * p.Bcap + j) * DI;
    reinterpret_cast<uint4*>(out)[c] =
        make_uint4(IT::pack(m[0], m[1]), IT::pack(m[2], m[3]), IT::pack(m[4], m[5]), IT::pack(m[6], m[7]));
    return true;
}

template <class IT, int DI, int KBS, bool PR>
__global__ void __launch_bounds__(32 * QSA_WARP_TASKS, 16 / QSA_WARP_TASKS) qsa_warp_kernel(const QsaParams p) {
    static_assert(DI % 8 == 0 && DI / 8 <= 32 && 32 % (DI / 8) == 0, "one row must span a power-of-two number of lanes");
    constexpr int C = DI / 8;              // 16-byte chunks per row
    constexpr int G = 32 / C;              // row groups per warp
    static_assert(KBS % G == 0, "block rows must split evenly over the row groups");
    constexpr int NR = KBS / G;            // rows summed per lane
    // Loads in flight per lane: the whole block when it is at most 32 rows
    // per lane and the constants were read before the wait (PR): 3.51 -> 3.34 us
    // per call on the 32 x 2048-token workload; otherwise batches of 16 (the
    // default form measured slower with 32: 4.63 -> 4.73 us with the window
    // prefetch, 3.58 -> 4.59 us with the hinted block).
    constexpr int RB = (PR && NR <= 32) ? NR : (NR < 16 ? NR : 16);
    __shared__ __align__(16) float u_s[QSA_WARP_TASKS][DI];

    const int lane = threadIdx.x & 31;
    const int wid = threadIdx.x >> 5;
    const int c = lane % C;
    const int g = lane / C;
    const uint32_t per_seq = uint32_t(p.nbmax + 1 + p.ncopy);
    const uint32_t task = blockIdx.x * QSA_WARP_TASKS + wid;
    const uint32_t n32 = task / per_seq;
    const bool live = n32 < uint32_t(p.N);   // the last CTA may hold spare warps
    const int64_t n = n32;
    const int64_t jl = int64_t(task - n32 * per_seq);
    const uint16_t* raw = static_cast<const uint16_t*>(p.raw) + n * p.L * DI;
    const uint16_t* past = static_cast<const uint16_t*>(p.past_raw) + n * (KBS - 1) * DI;
    const int64_t* kl = p.key_length + (p.key_length_per_seq ? n : 0);

    QsaSeq q = {0, 0, 0, 0};
    QsaSeq qh = {0, -1, 0, 0};   // default form: scalars from the key_length hint (P < 0: none usable)
    uint4 cv = make_uint4(0, 0, 0, 0), sv = make_uint4(0, 0, 0, 0), wv = make_uint4(0, 0, 0, 0);
    if (live) {
        if (PR) q = qsa_seq<KBS>(p, n);
        // Prefetches are only hints, and L2 is the coherence point: they are
        // safe before the wait even for inputs the preceding grid writes.
        if (jl > p.nbmax) {
            // concat-output copy task: its past block-key rows (all rows below
            // min(Bp, Bcap) that it may copy; with PR exactly those below j0)
            if (lane == 0 && p.copy_vec) {
                int64_t lim = min(p.Bp, p.Bcap);
                if (PR) lim = q.P >= 0 ? min(lim, q.j0) : 0;
                const int64_t r0 = (jl - p.nbmax - 1) * p.copy_rows;
                const int64_t r1 = min(r0 + int64_t(p.copy_rows), lim);
                if (r1 > r0)
                    prefetch_l2_bulk(static_cast<const uint16_t*>(p.past_bk) + (n * p.Bp + r0) * DI,
                                     uint32_t(r1 - r0) * DI * 2);
            }
        } else if (PR) {
            if (q.P >= 0 && jl < q.nb && q.j0 + jl < p.Bcap) {
                // exactly the block's rows, and its constants
                if (lane == 0) qsa_prefetch_block<DI, KBS, false>(p, q, n, jl, raw, past);
                qsa_chunk_consts<DI>(p, n, (q.j0 + jl) * KBS, q.P, c, cv, sv, wv);
            }
        } else if (jl < p.nbmax) {
            if (lane == 0 && jl == 0 && p.w != nullptr) prefetch_l2_bulk(p.w, DI * 2);
            const QsaSeq h = p.key_length_late ? QsaSeq{0, -1, 0, 0} : qsa_seq_of<KBS>(p, ld_relaxed_s64(kl));
            if (h.P >= 0 && jl < h.nb && h.j0 + jl < p.Bcap) {
                if (lane == 0) qsa_prefetch_block<DI, KBS, true>(p, h, n, jl, raw, past);
                qh = h;
            } else if (lane == 0) {
#if KVR_QSA_RAW_PREFETCH
                // no block from the hint: new-key rows [jl*KBS, (jl+1)*KBS)
                const int64_t r0 = jl * KBS;
                prefetch_l2_bulk(raw + r0 * DI, uint32_t(min(int64_t(KBS), p.L - r0) * DI * 2));
#endif
            }
        } else if (p.next_raw != nullptr && !p.key_length_late) {
            // carry task: the rows after the last completed block, as the hint
            // places them
            const QsaSeq h = qsa_seq_of<KBS>(p, ld_relaxed_s64(kl));
            if (lane == 0 && h.P >= 0 && h.nb <= p.nbmax) {
                const int64_t Fn = (h.j0 + h.nb) * KBS;
                const int64_t rem = h.K - Fn;
                if (Fn >= h.P && rem > 0 && rem < KBS)
                    prefetch_l2_bulk(raw + (Fn - h.P) * DI, uint32_t(rem) * DI * 2);
            }
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (!live) return;
    if (!PR) {
        if (qh.P >= 0) {
            // the hinted block's loads go out together with the real key_length
            const int64_t Kt = *kl;
            if (qsa_warp_block<IT, DI, KBS, RB, true>(p, qh, n, jl, raw, past, c, g, u_s[wid], cv, sv, wv, true, Kt))
                return;
            q = qsa_seq_of<KBS>(p, Kt);   // a stale hint: start over from the real key_length
        } else {
            q = qsa_seq<KBS>(p, n);
        }
    }

    const int64_t P = q.P;
    if (P < 0) {
        if (jl == 0 && lane == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_KEY_LENGTH);
        return;
    }
    const int64_t F = q.j0 * KBS;              // first token of the incomplete block

    if (jl > p.nbmax) {
        copy_past_block_keys(p, n, jl - p.nbmax - 1, q.j0, lane, 32);
        return;
    }
    if (jl == p.nbmax) {
        if (lane == 0) past_block_status(p, q.j0);
        // carry outputs: the tokens after the last completed block
        const int64_t Fn = (q.j0 + q.nb) * KBS;
        const int rem = int(q.K - Fn);
        if (p.next_raw != nullptr) {
            uint16_t* dst = static_cast<uint16_t*>(p.next_raw) + n * (KBS - 1) * DI;
            const bool v16 = (reinterpret_cast<uintptr_t>(dst) & 15) == 0;
            const int per_row = v16 ? C : DI;
            for (int e = lane; e < rem * per_row; e += 32) {
                const int r = e / per_row, k = e - r * per_row;
                const int64_t tok = Fn + r;
                const uint16_t* src = tok < P ? past + (tok - F) * DI : raw + (tok - P) * DI;
                if (v16)
                    reinterpret_cast<uint4*>(dst + int64_t(r) * DI)[k] = reinterpret_cast<const uint4*>(src)[k];
                else
                    dst[int64_t(r) * DI + k] = src[k];
            }
        }
        if (p.next_rope != nullptr && p.Dr > 0 && rem > 0) {
            uint16_t* dst = static_cast<uint16_t*>(p.next_rope) + n * 2 * p.Dr;
            for (int e = lane; e < 2 * p.Dr; e += 32) {
                uint16_t v;
                if (Fn >= P) {
                    const int64_t row = (n * p.L + (Fn - P)) * p.Dr;
                    v = e < p.Dr ? static_cast<const uint16_t*>(p.cos)[row + e]
                                 : static_cast<const uint16_t*>(p.sin)[row + e - p.Dr];
                } else {
                    v = static_cast<const uint16_t*>(p.past_rope)[n * 2 * p.Dr + e];
                }
                dst[e] = v;
            }
        }
        return;
    }
    if (jl >= q.nb) return;
    if (q.j0 + jl >= p.Bcap) {
        if (lane == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_BLOCK_CAP);
        return;
    }
    qsa_warp_block<IT, DI, KBS, RB, !PR>(p, q, n, jl, raw, past, c, g, u_s[wid], cv, sv, wv, false, 0);
}

typedef void (*QsaKernel)(const QsaParams);

// Compile-time shapes for common key widths and block sizes take the warp
// kernel (with the sizes as constants, a small call's per-block instruction
// chain is shorter); any other aligned shape takes the bulk kernel.
template <class IT, int DI, bool PR>
static QsaKernel pick_qsa_warp_kbs(int64_t kbs) {
    switch (kbs) {
        case 32: return qsa_warp_kernel<IT, DI, 32, PR>;
        case 64: return qsa_warp_kernel<IT, DI, 64, PR>;
        case 128: return qsa_warp_kernel<IT, DI, 128, PR>;
        default: return nullptr;
    }
}

template <class IT, bool PR>
static QsaKernel pick_qsa_warp(int Di, int64_t kbs) {
    if (Di == 64) return pick_qsa_warp_kbs<IT, 64, PR>(kbs);
    if (Di == 128) return pick_qsa_warp_kbs<IT, 128, PR>(kbs);
    if (Di == 256) return pick_qsa_warp_kbs<IT, 256, PR>(kbs);
    return nullptr;
}

bool qsa_warp_shape(int64_t Di, int64_t kbs) {
#if KVR_QSA_WARP
    return (Di == 64 || Di == 128 || Di == 256) && (kbs == 32 || kbs == 64 || kbs == 128);
#else
    (void)Di;
    (void)kbs;
    return false;
#endif
}


// Shared memory the bulk variant needs (0 if it does not fit).
static size_t qsa_bulk_smem(const QsaParams& p) {
    const int C = p.Di / 8;
    const int G = C >= QSA_BULK_THREADS ? 1 : QSA_BULK_THREADS / C;
    const size_t bytes = 128 + size_t(p.kbs) * p.Di * 2 + size_t(p.Di) * 2 + (2 * size_t(p.Dr) + 8) * 2 +
                         (size_t(G) * p.Di + p.Di + QSA_BULK_THREADS / 32 + 1) * 4;
    return bytes <= 96 * 1024 ? bytes : 0;
}

cudaError_t launch_qsa(const QsaParams& p, int in_dtype, bool vec, bool bulk, bool warp, cudaStream_t s) {
    const int64_t grid = p.N * (p.nbmax + 1 + p.ncopy);
    if (warp) {
        const bool bf = in_dtype == KVR_BF16;
        QsaKernel fn = p.params_ready ? (bf ? pick_qsa_warp<BF16, true>(p.Di, p.kbs) : pick_qsa_warp<F16, true>(p.Di, p.kbs))
                                      : (bf ? pick_qsa_warp<BF16, false>(p.Di, p.kbs) : pick_qsa_warp<F16, false>(p.Di, p.kbs));
        if (fn == nullptr) return cudaErrorInvalidValue;
        return launch_pdl(fn, dim3(unsigned((grid + QSA_WARP_TASKS - 1) / QSA_WARP_TASKS)),
                          dim3(32 * QSA_WARP_TASKS), 0, s, p);
    }
    const size_t bsmem = bulk ? qsa_bulk_smem(p) : 0;
    if (bsmem > 0) {
        QsaKernel fn = in_dtype == KVR_BF16 ? qsa_bulk_kernel<BF16, 0, 0> : qsa_bulk_kernel<F16, 0, 0>;
        if (bsmem > 48 * 1024) {
            static std::mutex mu;
            static std::set<const void*> done;
            std::lock_guard<std::mutex> lock(mu);
            if (!done.count(reinterpret_cast<const void*>(fn))) {
                cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
                if (e != cudaSuccess) return e;
                done.insert(reinterpret_cast<const void*>(fn));
            }
        }
        return launch_pdl(fn, dim3(unsigned(grid)), dim3(QSA_BULK_THREADS), bsmem, s, p);
    }
    const int C = vec ? p.Di / 8 : p.Di;
    const int G = C >= QSA_THREADS ? 1 : QSA_THREADS / C;
    const size_t smem = (size_t(G) * p.Di + p.Di + QSA_THREADS / 32 + 1) * sizeof(float);
    if (vec) {
        auto fn = in_dtype == KVR_BF16 ? qsa_kernel<BF16, 8> : qsa_kernel<F16, 8>;
        return launch_pdl(fn, dim3(unsigned(grid)), dim3(QSA_THREADS), smem, s, p);
    }
    auto fn = in_dtype == KVR_BF16 ? qsa_kernel<BF16, 1> : qsa_kernel<F16, 1>;
    return launch_pdl(fn, dim3(unsigned(grid)), dim3(QSA_THREADS), smem, s, p);
}

}  // namespace kvr
