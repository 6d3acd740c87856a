// Pipelined KV prologue kernel: bulk async copies (TMA engine) of whole row
// tiles into a shared-memory ring, consumed by compute warps.
//
// Operation: "aclnnKvRmsNormRopeCache" (hiascend.com), "Description",
// "Formulas (1) interleaveRope", "Formulas (2) rmsNorm", "Restrictions on
// index", "Restrictions on quantization scenarios"; alpha_kv of
// "aclnnMlaPrologV3WeightNz" ("Formula", key path).
//
// Why this shape on GB300: the op moves ~2.6 KB per token at ~1 flop/byte,
// so HBM must see enough bytes in flight (Little's law: ~44 KB per SM at
// ~7 TB/s and ~1 us latency). Register-staged loads cap that by occupancy;
// here the in-flight data lives in shared memory instead:
//  * one persistent CTA per SM; warp 0 is the producer, BULK_CONSUMERS warps
//    compute;
//  * CTA b owns one contiguous range of about T / gridDim rows (starting on
//    an even row), cut into tiles of up to R rows: every SM moves the same
//    bytes (dealing whole tiles round-robin left 7 tiles on some SMs and 6
//    on others for a 32768-row prefill);
//  * a tile is R consecutive token rows; per tile the producer issues one
//    bulk copy for the kv rows (one per row when rows are strided), one for
//    the cos rows, one for the sin rows and one for the index entries, all
//    completing on the stage's `full` mbarrier (expect_tx byte count);
//  * S stages in flight per SM (S*R rows, up to 200 KB: 4 stages of 32 rows
//    for the 512 + 64 split), recycled through an
//    `empty` mbarrier that each consumer warp arrives on;
//  * a consumer warp owns one row at a time: 16-byte shared loads of the Dv
//    part (conflict-free), fp32 sum of squares with a warp butterfly, gamma
//    from shared memory, 16-byte global stores of the whole cache row; the
//    RoPE runs one pair per lane (all 32 lanes busy for Dk = 64);
//  * every wait is bounded (KVR_DEVERR_TIMEOUT), and a CTA never exits with
//    its copies in flight;
//  * programmatic dependent launch: the CTA initialises its barriers, then
//    waits for the previous grid before its first global access.
#include <mutex>
#include <set>

#include "kv_common.cuh"

namespace kvr {

#ifndef KVR_BULK_CONSUMERS
#define KVR_BULK_CONSUMERS 16
#endif
constexpr int BULK_CONSUMERS = KVR_BULK_CONSUMERS;
constexpr int BULK_THREADS = 32 * (1 + BULK_CONSUMERS);
// Resident CTAs per SM (each with its own ring of KVR_BULK_RING_KB).
#ifndef KVR_BULK_CTAS_PER_SM
#define KVR_BULK_CTAS_PER_SM 1
#endif
// Before the dependency wait, prefetch this CTA's first S - 1 tiles (all but
// one stage of its ring) into L2; a hint only, L2 is the coherence point.
// The next call's CTAs start as this call's CTAs finish, and their prefetch
// burst shares DRAM with this call's tail: on the 32768-token prefill (S = 4
// stages of 32 rows) a call took 15.4 us with no prefetch, 14.75 / 14.1 /
// 14.05 us with 1 / 2 / 3 tiles and 14.55 us with the whole ring.
#ifndef KVR_BULK_PREFETCH
#define KVR_BULK_PREFETCH 1
#endif

// DV / DK: the row split when fixed at compile time (0: from the parameters).
template <class IT, int CPL, int CK, int DV = 0, int DK = 0>
__global__ void __launch_bounds__(BULK_THREADS, KVR_BULK_CTAS_PER_SM) kv_bulk_kernel(const KvParams p) {
    const int Dv = DV ? DV : p.Dv;
    const int Dk = DK ? DK : p.Dk;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + p.S;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + p.S);
    const int nch = Dv >> 3;
    float4* g_lo = reinterpret_cast<float4*>(smem + p.off_consts);
    float4* g_hi = g_lo + nch;
    float4* c_lo = g_hi + nch;
    float4* c_hi = c_lo + nch;
    float* s_kscale = reinterpret_cast<float*>(c_hi + nch);
    unsigned char* stages = smem + p.off_stages;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // This CTA's rows [lo, hi): even starts keep the index tiles 16-byte aligned.
    const int64_t lo = (p.T * int64_t(blockIdx.x) / gridDim.x) & ~int64_t(1);
    const int64_t hi = blockIdx.x + 1 == gridDim.x ? p.T : ((p.T * int64_t(blockIdx.x + 1) / gridDim.x) & ~int64_t(1));
    const uint32_t kv_row = uint32_t(Dv + Dk) * 2;
    const uint32_t cs_row = uint32_t(Dk) * 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], BULK_CONSUMERS);
        }
        *abort_flag = 0;
        fence_mbar_init();
#if KVR_BULK_PREFETCH
        int64_t it = 0;
        const int64_t npf = p.S > 1 ? p.S - 1 : 1;
        for (int64_t r0 = lo; r0 < hi && it < npf; r0 += p.R, ++it) {
            const int rows = int(hi - r0 < p.R ? hi - r0 : p.R);
            if (p.kv_contig) prefetch_l2_bulk(static_cast<const char*>(p.kv) + r0 * kv_row, rows * kv_row);
            prefetch_l2_bulk(static_cast<const char*>(p.cos) + r0 * cs_row, rows * cs_row);
            prefetch_l2_bulk(static_cast<const char*>(p.sin) + r0 * cs_row, rows * cs_row);
            if (p.idx_bulk && rows >= 2) prefetch_l2_bulk(p.index + r0, uint32_t(rows & ~1) * 8);
        }
#endif
    }
    __syncthreads();
    pdl_wait();
    pdl_launch_dependents();

    if (warp == 0) {
        // ---------------- producer ----------------
        const uint64_t policy = l2_policy_evict_first();
        int64_t it = 0;
        bool ok = true;
        for (int64_t r0 = lo; r0 < hi; r0 += p.R, ++it) {
            const int s = int(it % p.S);
            if (it >= p.S && !mbar_wait_warp(&empty[s], uint32_t(((it / p.S) - 1) & 1), abort_flag)) {
                ok = false;
                break;
            }
            const int rows = int(hi - r0 < p.R ? hi - r0 : p.R);
            const int idx_rows = p.idx_bulk ? (rows & ~1) : 0;
            unsigned char* st = stages + size_t(s) * p.stage_bytes;
            if (lane == 0) mbar_arrive_expect_tx(&full[s], rows * kv_row + 2 * rows * cs_row + idx_rows * 8);
            __syncwarp();
            const char* kvb = static_cast<const char*>(p.kv);
            if (p.kv_contig) {
                if (lane == 0) bulk_g2s_hint(st, kvb + r0 * kv_row, rows * kv_row, &full[s], policy);
            } else {
                for (int r = lane; r < rows; r += 32)
                    bulk_g2s_hint(st + r * kv_row, kvb + (r0 + r) * p.kv_stride * 2, kv_row, &full[s], policy);
            }
            if (lane == 1)
                bulk_g2s_hint(st + p.off_cos, static_cast<const char*>(p.cos) + r0 * cs_row, rows * cs_row, &full[s], policy);
            if (lane == 2)
                bulk_g2s_hint(st + p.off_sin, static_cast<const char*>(p.sin) + r0 * cs_row, rows * cs_row, &full[s], policy);
            if (lane == 3 && idx_rows > 0) bulk_g2s_hint(st + p.off_idx, p.index + r0, idx_rows * 8, &full[s], policy);
        }
        if (!ok && lane == 0) {
            *abort_flag = 1;
            if (p.status != nullptr) atomicOr(p.status, KVR_DEVERR_TIMEOUT);
        }
        // The CTA's shared memory must outlive every copy this warp issued.
        for (int64_t j = (it > p.S ? it - p.S : 0); j < it; ++j)
            mbar_wait_warp(&full[j % p.S], uint32_t((j / p.S) & 1), nullptr);
        return;
    }

    // ---------------- consumers ----------------
    const int ct = threadIdx.x - 32;
    const int h = Dk >> 1;
    stage_gamma<IT>(g_lo, g_hi, nch, p.gamma, ct, 32 * BULK_CONSUMERS);
    const bool cper = CK != OUT16 && p.ckv_scale_per_ch;
    const bool kq = p.k_kind != OUT16;
    if (cper) stage_chan_f32(c_lo, c_hi, nch, p.ckv_scale, ct, 32 * BULK_CONSUMERS);
    if (kq && p.k_scale_per_ch)
        for (int i = ct; i < Dk; i += 32 * BULK_CONSUMERS) s_kscale[i] = p.k_scale[i];
    const float cscale0 = (CK != OUT16 && !p.ckv_scale_per_ch) ? p.ckv_scale[0] : 1.f;
    const float kscale0 = (kq && !p.k_scale_per_ch) ? p.k_scale[0] : 1.f;
    const float* kscale = (kq && p.k_scale_per_ch) ? s_kscale : nullptr;
    asm volatile("bar.sync 1, %0;" ::"r"(32 * BULK_CONSUMERS) : "memory");

    const int cw = warp - 1;
    int64_t it = 0;
    for (int64_t r0 = lo; r0 < hi; r0 += p.R, ++it) {
        const int s = int(it % p.S);
        if (!mbar_wait_warp(&full[s], uint32_t((it / p.S) & 1), abort_flag)) {
            if (lane == 0) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, KVR_DEVERR_TIMEOUT);
            }
            break;
        }
        const int rows = int(hi - r0 < p.R ? hi - r0 : p.R);
        const int idx_rows = p.idx_bulk ? (rows & ~1) : 0;
        const unsigned char* st = stages + size_t(s) * p.stage_bytes;
        // Rows are dealt round-robin over the consumer warps across stages:
        // this CTA's q-th row goes to warp q % BULK_CONSUMERS (every tile
        // but the range's last has R rows, so q = it * R + r).
        const int first = int((cw - (it * p.R) % BULK_CONSUMERS + BULK_CONSUMERS) % BULK_CONSUMERS);
        for (int r = first; r < rows; r += BULK_CONSUMERS) {
            const int64_t t = r0 + r;
            const int64_t v = r < idx_rows ? reinterpret_cast<const int64_t*>(st + p.off_idx)[r]
                                           : p.index[index_pos(p, t)];
            const int64_t row = resolve_row(p, t, v);
            if (row < 0) {
                if (row == ROW_BAD && lane == 0 && p.status != nullptr) atomicOr(p.status, KVR_DEVERR_INDEX);
                continue;
            }
            const unsigned char* xr = st + size_t(r) * kv_row;
            float2 xg[CPL][4];
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const int ch = c * 32 + lane;
                if (ch < nch)
                    chunk_xg<IT>(*reinterpret_cast<const uint4*>(xr + ch * 16), g_lo[ch], g_hi[ch], xg[c], acc);
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
            const uint32_t* xp = reinterpret_cast<const uint32_t*>(xr + Dv * 2);
            const uint16_t* cr = reinterpret_cast<const uint16_t*>(st + p.off_cos) + size_t(r) * Dk;
            const uint16_t* sr = reinterpret_cast<const uint16_t*>(st + p.off_sin) + size_t(r) * Dk;
            char* krow = static_cast<char*>(p.kc) + row * Dk * (kq ? 1 : 2);
            for (int i = lane; i < h; i += 32)
                rope_pair_store<IT>(krow, i, h, xp[i], cr[i], sr[i], cr[h + i], sr[h + i], p.k_kind, kscale, kscale0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
}

typedef void (*BulkKernel)(const KvParams);

template <class IT, int CPL, int DV = 0, int DK = 0>
static BulkKernel pick_ck(int ck) {
    switch (ck) {
        case OUT16: return kv_bulk_kernel<IT, CPL, OUT16, DV, DK>;
        case OUT_I8: return kv_bulk_kernel<IT, CPL, OUT_I8, DV, DK>;
        case OUT_E4M3: return kv_bulk_kernel<IT, CPL, OUT_E4M3, DV, DK>;
        default: return kv_bulk_kernel<IT, CPL, OUT_E5M2, DV, DK>;
    }
}

// The MLA latent split (Dv = 512, Dk = 64) is compiled as constants.
#ifndef KVR_BULK_SPECIALISE
#define KVR_BULK_SPECIALISE 1
#endif
template <class IT>
static BulkKernel pick_cpl(int cpl, int ck, int Dv, int Dk) {
    if (KVR_BULK_SPECIALISE && Dv == 512 && Dk == 64) return pick_ck<IT, 2, 512, 64>(ck);
    if (cpl == 1) return pick_ck<IT, 1>(ck);
    if (cpl == 2) return pick_ck<IT, 2>(ck);
    return pick_ck<IT, 4>(ck);
}

static uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Shared memory the ring may use per CTA (one CTA per SM), and the largest
// tile (rows per stage).
#ifndef KVR_BULK_RING_KB
#define KVR_BULK_RING_KB 200
#endif
#ifndef KVR_BULK_MAX_ROWS
#define KVR_BULK_MAX_ROWS 32
#endif
constexpr uint32_t BULK_RING_BYTES = KVR_BULK_RING_KB * 1024;

// Allow the kernel its dynamic shared memory once (not a stream operation,
// so later calls under stream capture make no attribute call).
static cudaError_t ensure_smem(BulkKernel fn) {
    static std::mutex mu;
    static std::set<BulkKernel> done;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count(fn)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess) done.insert(fn);
    return e;
}

cudaError_t launch_kv_bulk(const KvParams& p0, int in_dtype, int ckv_kind, cudaStream_t s) {
    KvParams p = p0;
    const int sms = sm_count_current_device();
    // Rows per tile: up to KVR_BULK_MAX_ROWS, halved while that leaves fewer
    // than four tiles per SM (load balance across the SMs).
    int R = KVR_BULK_MAX_ROWS;
    while (R > 2 && (p.T + R - 1) / R < int64_t(4) * sms) R >>= 1;
    const uint32_t kv_row = uint32_t(p.Dv + p.Dk) * 2;
    const uint32_t cs_row = uint32_t(p.Dk) * 2;
    p.R = R;
    p.off_cos = R * kv_row;
    p.off_sin = p.off_cos + R * cs_row;
    p.off_idx = p.off_sin + R * cs_row;
    p.stage_bytes = align_up(p.off_idx + R * 8, 128);
    const int S = int(BULK_RING_BYTES / p.stage_bytes);
    p.S = S < 2 ? 2 : (S > 16 ? 16 : S);
    const uint32_t header = align_up(16 * p.S + 16, 128);
    p.off_consts = header;
    const uint32_t consts = align_up(uint32_t(p.Dv) * 8 + uint32_t(p.Dk) * 4, 128);
    p.off_stages = header + consts;
    const size_t smem = size_t(p.off_stages) + size_t(p.S) * p.stage_bytes;
    if (smem > 227 * 1024) return cudaErrorInvalidValue;

    const int nch = p.Dv / 8;
    const int cpl = nch <= 32 ? 1 : (nch <= 64 ? 2 : 4);
    BulkKernel fn = in_dtype == KVR_BF16 ? pick_cpl<BF16>(cpl, ckv_kind, p.Dv, p.Dk)
                                         : pick_cpl<F16>(cpl, ckv_kind, p.Dv, p.Dk);
    cudaError_t e = ensure_smem(fn);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (p.T + R - 1) / R;
    const int64_t slots = int64_t(sms) * KVR_BULK_CTAS_PER_SM;
    const int grid = int(ntiles < slots ? ntiles : slots);
    return launch_pdl(fn, dim3(grid), dim3(BULK_THREADS), smem, s, p);
}

}  // namespace kvr
