/*
 * kvr.h - C ABI of libkvr.so, the GB300 (sm_103a) attention-prologue key path.
 *
 * Three operations:
 *
 *   kv_rmsnorm_rope_cache()  the fused KV prologue of the page
 *       "aclnnKvRmsNormRopeCache" (hiascend.com, CANN ops-transformer):
 *       each token row of width D = Dv + Dk is split on its tail axis
 *       ("Description"); the left Dv part is RMS-normalised
 *       ("Formulas (2) rmsNorm": y = x / sqrt(mean(x^2) + eps) * gamma),
 *       the right Dk part gets the interleaved RoPE ("Formulas (1)
 *       interleaveRope": y = cat(x[::2], x[1::2]) * cos + cat(-x[1::2], x[::2]) * sin),
 *       and both results are scattered by slot index into two caches
 *       ("Restrictions on index"), optionally quantised to 8-bit codes
 *       ("Restrictions on quantization scenarios"). The kcScale factor
 *       alpha_kv of "aclnnMlaPrologV3WeightNz" ("Formula", key path) may
 *       scale the normalised part.
 *
 *   qsa_prepare()  the block-key prepare of "openvino.opset17.qsa_prepare"
 *       (docs.openvino.ai): one key per key block completed by the new
 *       tokens = mean of the block's raw index keys, RMS-normalised with
 *       k_norm_weight, rotated with the RoPE of the block's first token;
 *       incomplete blocks are carried across calls.
 *
 *   dynamic_quant()  DynamicQuant of q^N, the query-side step beside this
 *       path on "aclnnMlaPrologV3WeightNz": per-row int8 codes and scales.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller (the
 *     host-staged entry points also take pinned host buffers); the library
 *     allocates no device memory and keeps no per-call state, with one
 *     exception: kv_rmsnorm_rope_cache_staged_static stages its inputs in a
 *     static device array of the library, shared by all its calls on a
 *     device. Rows are dense and row-major unless a stride argument says
 *     otherwise.
 *   - Calls are asynchronous on `stream`: they validate on the host, launch,
 *     and return. Nothing is read back to the host (except the status word
 *     the host-staged entry point copies back, asynchronously, and the index
 *     that the opt-in debug validation, kvr_set_debug_validate, checks).
 *   - Host-side errors (a NULL that is required, a bad shape, dtype or
 *     mode) are returned before any launch; nothing is written. Sizes whose
 *     element offsets or byte counts would reach 2^62 are KVR_ERR_SHAPE.
 *   - Data-dependent errors are found on the device: the offending row or
 *     block is skipped (never written out of bounds) and, if `dev_status`
 *     is non-NULL, the matching KVR_DEVERR_* bit is OR-ed into *dev_status.
 *     No kernel traps or asserts. Waits inside a kernel (its copy pipeline)
 *     are bounded: past one second a kernel raises KVR_DEVERR_TIMEOUT, lets
 *     its copies in flight land, and returns.
 *   - Each launch uses programmatic dependent launch: it may start while the
 *     previous kernel on the stream finishes, and waits for that kernel's
 *     results before it uses any input (the one exception is opt-in:
 *     the params_ready flags let constants be read earlier). Before the wait
 *     a kernel issues L2 prefetches of its inputs; qsa_prepare's
 *     compiled-shape kernel also reads key_length there, as a hint for those
 *     prefetches only (a relaxed read; kvr_qsa_args.key_length_late turns
 *     it off), and takes its value after the wait.
 *   - An empty problem (T = Bkv*Skv = 0, or N = 0) returns KVR_OK with no
 *     launch, mirroring the empty-tensor rule of "aclnnMlaPrologV3WeightNz"
 *     ("Shape restrictions": caches are not updated). A qsa_prepare call
 *     with L = 0 launches only when it has carry outputs or a separate past
 *     buffer to write.
 *   - Results are deterministic: no atomics touch data.
 *   - Thread safe: entry points may be called concurrently from any host
 *     thread on any stream; overlapping writes to the same cache rows from
 *     concurrent calls are the caller's race. The exception is
 *     kv_rmsnorm_rope_cache_staged_static: its calls that can run at the
 *     same time on the GPU share its staging area and race on it.
 */
#ifndef KVR_H
#define KVR_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVR_ABI_VERSION 10

typedef enum kvr_status {
    KVR_OK = 0,
    KVR_ERR_NULL = 1,         /* a required pointer is NULL, or optional pairs disagree */
    KVR_ERR_SHAPE = 2,        /* a size is out of its documented range */
    KVR_ERR_DTYPE = 3,        /* an element type is not supported for that argument */
    KVR_ERR_MODE = 4,         /* unknown cache mode */
    KVR_ERR_ALIAS = 5,        /* an output overlaps an input it must not overlap */
    KVR_ERR_CUDA = 6,         /* the launch failed (see cudaGetLastError) */
    KVR_ERR_INDEX = 7         /* debug validation only (kvr_set_debug_validate): an index
                                 entry is out of range or names a cache row that another
                                 entry of the call names */
} kvr_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define KVR_DEVERR_INDEX 0x1       /* kv: an index entry outside {-1} U [0, range) */
#define KVR_DEVERR_KEY_LENGTH 0x2  /* qsa: key_length[n] < L (the past length would be negative) */
#define KVR_DEVERR_BLOCK_CAP 0x4   /* qsa: a completed block's number is >= Bcap */
#define KVR_DEVERR_TIMEOUT 0x8     /* a pipeline wait inside a kernel exceeded its limit
                                      (one second); that CTA stopped early, output incomplete */
#define KVR_DEVERR_PAST_BLOCKS 0x10 /* qsa, concat-output form: past_block_index_keys holds
                                      fewer than floor(P/kbs) rows for a sequence */

typedef enum kvr_dtype {
    KVR_BF16 = 0,
    KVR_F16 = 1,
    KVR_INT8 = 2,             /* caches only: round half to even, clamp to [-128, 127] */
    KVR_FP8_E4M3FN = 3,       /* caches only: round to nearest even, saturate to +-448 */
    KVR_FP8_E5M2 = 4          /* caches only: round to nearest even, saturate to +-57344 */
} kvr_dtype;

/* Cache layouts of "aclnnKvRmsNormRopeCache" ("Restrictions on index"); the
 * head axis N is 1, so BNSD and BSND are the same bytes. */
typedef enum kvr_cache_mode {
    /* cache [Bcache=d0, Scache=d1, 1, D*]; index [Bkv, Skv] in [-1, Scache);
     * token (b, s) goes to cache row (b, index[b, s]); requires Bcache >= Bkv. */
    KVR_CACHE_NORM = 0,
    /* cache [BlockNum=d0, BlockSize=d1, 1, D*]; index [Bkv*Skv] in
     * [-1, BlockNum*BlockSize); token t goes to slot index[t]. */
    KVR_CACHE_PA_BSND = 1,
    /* cache as PA_BSND; index [Bkv * ceil(Skv/BlockSize)], one entry per
     * BlockSize tokens of a sequence; token s goes to slot
     * index[b, s / BlockSize] + s % BlockSize, which must stay inside the
     * block the entry names (else KVR_DEVERR_INDEX). */
    KVR_CACHE_PA_BLK_BSND = 2
} kvr_cache_mode;

/*
 * Arguments of kv_rmsnorm_rope_cache(). T = Bkv * Skv token rows.
 *
 *   kv         [Bkv, 1, Skv, >= Dv+Dk] input rows, element type `in_dtype`
 *              (bf16 or f16). Row t starts kv_row_stride elements after row
 *              t-1 (0 means Dv+Dk, i.e. dense); a larger stride reads kv as
 *              a column slice of a wider row (e.g. a fused projection output).
 *   gamma      [Dv] RMSNorm weight, `in_dtype`.
 *   cos, sin   [Bkv, 1, Skv, Dk] full-width RoPE tables, `in_dtype`; output
 *              lane i < Dk/2 uses entry i, lane i + Dk/2 uses entry i + Dk/2.
 *   index      int64, layout per `mode` (see kvr_cache_mode); -1 = skip.
 *              Repeated targets within one call (forbidden by the page) leave
 *              an unspecified winner.
 *   cache_d0, cache_d1   the two leading cache dims (Bcache, Scache) or
 *              (BlockNum, BlockSize).
 *   ckv_cache  [d0, d1, 1, Dv] of `ckv_dtype`; k_cache [d0, d1, 1, Dk] of `k_dtype`.
 *              A cache dtype is `in_dtype` (bf16/f16) or an 8-bit code type.
 *   ckv_scale  float32 [ckv_scale_len], len Dv (per channel) or 1 (per
 *              tensor); required iff ckv_dtype is an 8-bit type, else NULL.
 *              The code written is encode(alpha_kv * y[c] * ckv_scale[c]).
 *   k_scale    same for the k cache (len Dk or 1), applied to the RoPE output lane c.
 *   eps        added to the mean square (>= 0).
 *   kc_scale   alpha_kv, multiplies the normalised part; pass 1.0f for none.
 *   dev_status optional int32 device word; KVR_DEVERR_INDEX is OR-ed in when
 *              an index entry is out of range (that token is skipped).
 *   params_ready  0 (default): every input is read after the kernel waits for
 *              the preceding kernel on the stream (programmatic dependent
 *              launch). Nonzero: the caller promises that the kernel launched
 *              immediately before this call on `stream` does not write gamma,
 *              ckv_scale or k_scale (true of model weights and calibrated
 *              scales); they may then be read before that wait, overlapping
 *              the preceding kernel (the small-batch kernel for 16-bit caches
 *              does not, as that measured slower). Breaking the promise gives
 *              stale values.
 *
 * Limits: Dv >= 1, Dk >= 2 and even, Bkv, Skv >= 0, d0, d1 >= 1.
 * All arithmetic is float32 with one rounding to the cache type.
 */
typedef struct kvr_kv_args {
    const void* kv;
    kvr_dtype in_dtype;
    int64_t Bkv, Skv, Dv, Dk;
    int64_t kv_row_stride;
    const void* gamma;
    const void* cos;
    const void* sin;
    const int64_t* index;
    kvr_cache_mode mode;
    int64_t cache_d0, cache_d1;
    void* ckv_cache;
    kvr_dtype ckv_dtype;
    const float* ckv_scale;
    int64_t ckv_scale_len;
    void* k_cache;
    kvr_dtype k_dtype;
    const float* k_scale;
    int64_t k_scale_len;
    float eps;
    float kc_scale;
    int32_t* dev_status;
    int32_t params_ready;
} kvr_kv_args;

kvr_status kv_rmsnorm_rope_cache(const kvr_kv_args* args, cudaStream_t stream);

/*
 * Host-staged form of kv_rmsnorm_rope_cache (no counterpart on the pages: a
 * convenience for callers whose inputs are in host memory). On `stream`, in
 * order: copy `bytes` bytes from host memory `host_src` to device memory
 * `dev_dst` (the caller lays the step's inputs out there, so that the device
 * pointers in *args point into it), run kv_rmsnorm_rope_cache(args), and,
 * when `host_status` is given, copy *args->dev_status into *host_status.
 * All asynchronous: the host values are read and written when the stream
 * reaches the copies, so `host_src` and `host_status` should be pinned
 * (page-locked) and stay valid until the stream passes them; the caller
 * synchronises before reading *host_status. Arguments are validated first
 * and nothing is enqueued on an error (as kv_rmsnorm_rope_cache; plus
 * KVR_ERR_SHAPE for bytes < 0, KVR_ERR_NULL for a missing copy pointer or a
 * host_status without args->dev_status). A failed enqueue returns
 * KVR_ERR_CUDA (copies enqueued before it stay enqueued). Pinned buffers
 * (reported as host memory with a device address) in whole 16-byte units
 * are copied by kernels chained with the call (no copy-engine latency);
 * other memory goes through cudaMemcpyAsync.
 */
kvr_status kv_rmsnorm_rope_cache_staged(const kvr_kv_args* args, const void* host_src, void* dev_dst, int64_t bytes,
                                        int32_t* host_status, cudaStream_t stream);

/* Largest packed input, in bytes, that kv_rmsnorm_rope_cache_staged_static
 * stages: 8 MiB (a 256-token decode batch of the 512 + 64 split packs into
 * 354 KiB, a 4096-token batch into 5.5 MiB). */
#define KVR_STATIC_STAGE_BYTES (8 * 1024 * 1024)

/*
 * kv_rmsnorm_rope_cache_staged for callers that cannot allocate device memory
 * (no counterpart on the pages). The host-staged call needs a device buffer
 * to copy the step's inputs into, and some callers have none to give: code
 * running where cudaMalloc is not allowed (inside an allocator's own
 * callbacks, or under a framework that owns all device memory and offers its
 * plugins no way to ask for more) or a process whose memory budget is spent.
 * This entry point allocates nothing: it stages into one area of
 * KVR_STATIC_STAGE_BYTES that the library holds as a static device array on
 * every device that loads it, from load until the process exits.
 *
 *   args        as for kv_rmsnorm_rope_cache, except that args->kv, cos, sin
 *               and index are ignored: those four inputs are read from the
 *               staging area at the byte offsets below.
 *   host_src    `bytes` bytes of packed inputs in host memory (pinned for the
 *               copy to run as a kernel, as for kv_rmsnorm_rope_cache_staged);
 *               kv at kv_offset, cos at cos_offset, sin at sin_offset (each a
 *               multiple of 2) and index at index_offset (a multiple of 8),
 *               laid out as kv_rmsnorm_rope_cache expects them.
 *   bytes       at most KVR_STATIC_STAGE_BYTES; every input must lie inside
 *               [0, bytes), so each byte the call reads was written by its own
 *               copy and nothing in the area has to start at zero.
 *   host_status as for kv_rmsnorm_rope_cache_staged.
 *
 * Errors: bytes < 0 or > KVR_STATIC_STAGE_BYTES: KVR_ERR_SHAPE; an input
 * that does not fit inside [0, bytes) at its offset (the T kv rows at their
 * row stride, the cos and sin tables, the index entries of the mode; so in
 * particular a row width or row stride larger than `bytes`) or is misaligned:
 * KVR_ERR_SHAPE; nothing is enqueued on these errors. Everything else as
 * kv_rmsnorm_rope_cache_staged (KVR_ERR_CUDA if the area's address cannot be
 * found). Every call with T > 0 looks up the area's device address in the
 * current context (cudaGetSymbolAddress, which allocates nothing); the first
 * such call on a device may load the library's device code there, so make
 * it before any stream capture on the device. The address is never kept
 * between calls, so a device reset or another context stays safe. All calls
 * on a device share the one area, which keeps the last call's contents:
 * calls on the same stream are ordered, but calls that can run at the same
 * time on the GPU (other streams, other host threads) overwrite each other's
 * inputs.
 */
kvr_status kv_rmsnorm_rope_cache_staged_static(const kvr_kv_args* args, const void* host_src, int64_t bytes,
                                               int64_t kv_offset, int64_t cos_offset, int64_t sin_offset,
                                               int64_t index_offset, int32_t* host_status, cudaStream_t stream);

/* Which Dr channels the QSA rotation acts on and how it pairs them (the
 * qsa_prepare page names neither). Every layout writes pair i's results to
 * lanes i and i + Dr/2 of the rotated channels with cos/sin lanes i and
 * i + Dr/2, as the interleaved RoPE of "aclnnKvRmsNormRopeCache" does. */
typedef enum kvr_qsa_rope {
    KVR_QSA_ROPE_INTERLEAVE_LAST = 0,   /* pairs (x[2i], x[2i+1]) of channels [Di-Dr, Di) */
    KVR_QSA_ROPE_INTERLEAVE_FIRST = 1,  /* the same pairs of channels [0, Dr) */
    KVR_QSA_ROPE_HALF_LAST = 2,         /* rotate-half pairs (x[i], x[i+Dr/2]) of [Di-Dr, Di) */
    KVR_QSA_ROPE_HALF_FIRST = 3         /* rotate-half pairs of [0, Dr) */
} kvr_qsa_rope;

/*
 * Arguments of qsa_prepare(). Inputs follow the parameter list of
 * "openvino.opset17.qsa_prepare".
 *
 *   raw_index_keys  [N, L, Di] raw index key of every new token, `in_dtype`.
 *   block_keys      [N, Bcap, Di] in/out, `in_dtype`: the block keys of
 *                   earlier calls (past_block_index_keys) followed by room for
 *                   new ones. Block j (tokens [j*kbs, (j+1)*kbs) of the
 *                   sequence) is written at row j; no other row is touched.
 *                   In the concat-output form (below) rows j < floor(P/kbs)
 *                   are first copied from past_block_index_keys.
 *   key_length      int64 [N] or [1] (key_length_len = N or 1): valid key
 *                   tokens of each sequence AFTER this call, so the past
 *                   length is P = key_length - L (< 0: KVR_DEVERR_KEY_LENGTH,
 *                   the sequence is skipped). A [1] value applies to all N.
 *   rope_cos, rope_sin  [N, L, Dr] RoPE of every new token, or both NULL to
 *                   disable the rotation. By default the rotation is the
 *                   interleaved RoPE of "aclnnKvRmsNormRopeCache" on channels
 *                   [Di-Dr, Di); rope_layout selects another (kvr_qsa_rope).
 *   k_norm_weight   [Di] or NULL (NULL disables the RMS normalisation).
 *   past_incomplete_raw_keys  [N, kbs-1, Di]: raw keys of the past tokens of
 *                   the incomplete block (rows >= P mod kbs are never read).
 *   past_incomplete_rope      [N, 2*Dr] = [cos | sin] of the incomplete
 *                   block's first token; NULL iff rope_cos is NULL. Read only
 *                   when P mod kbs > 0.
 *   key_block_size  kbs > 1.   eps >= 0.
 *   next_incomplete_raw_keys  optional out [N, kbs-1, Di]: raw keys of the
 *                   tokens after the last completed block (K mod kbs rows;
 *                   the other rows are left untouched).
 *   next_incomplete_rope      optional out [N, 2*Dr]: [cos | sin] of the
 *                   first of those tokens (untouched when K mod kbs = 0).
 *                   The next_* outputs must not overlap any input
 *                   (KVR_ERR_ALIAS), so two carry buffers alternate between calls.
 *   dev_status      optional int32 device word (KVR_DEVERR_KEY_LENGTH,
 *                   KVR_DEVERR_BLOCK_CAP, KVR_DEVERR_PAST_BLOCKS).
 *   rope_layout     kvr_qsa_rope (0, the default, keeps the reading above).
 *   past_block_index_keys, Bp  concat-output form: [N, Bp, Di] `in_dtype`,
 *                   the page's past_block_index_keys as a separate input.
 *                   NULL (or equal to block_keys) = in place: block_keys
 *                   already holds them. Otherwise rows j < min(Bp,
 *                   floor(P/kbs)) are copied to block_keys (past rows at or
 *                   beyond Bcap: KVR_DEVERR_BLOCK_CAP; Bp < floor(P/kbs):
 *                   KVR_DEVERR_PAST_BLOCKS, the missing rows stay untouched),
 *                   so block_keys ends as the past keys followed by the new
 *                   ones. It must not overlap block_keys or the next_* outputs.
 *   params_ready    0 (default): every input is used as read after the kernel
 *                   waits for the preceding kernel on the stream (programmatic
 *                   dependent launch); the compiled-shape kernel reads
 *                   key_length once before that wait as a prefetch hint and
 *                   compares it with the value read after it (a stale hint,
 *                   e.g. key_length written by that preceding kernel, costs
 *                   time, never correctness: the warp sums its block a second
 *                   time, about 2 us on the 32 x 2048-token workload). Nonzero:
 *                   the caller promises that the
 *                   kernel launched immediately before this call on `stream`
 *                   writes none of key_length, rope_cos, rope_sin,
 *                   past_incomplete_rope and k_norm_weight (true when
 *                   sequence lengths come from the scheduler, the tables are
 *                   precomputed and the weight is a model weight); the kernel
 *                   for the compiled shapes (Di in {64, 128, 256}, kbs in
 *                   {32, 64, 128}, 16-byte aligned) then reads them before
 *                   that wait, so that only the key rows are read after it.
 *                   Other shapes ignore the flag. Breaking the promise gives
 *                   stale values.
 *   key_length_late 0 (default): as above. Nonzero (with params_ready 0): the
 *                   caller says that the kernel launched immediately before
 *                   this call writes key_length, so an early read would be
 *                   stale; the compiled-shape kernel then takes no key_length
 *                   hint and prefetches each warp's window of new keys
 *                   instead, which skips the second pass a stale hint costs.
 *                   Results are the same either way.
 *
 * Limits: N, L >= 0; Di >= 1; 0 <= Dr <= Di, Dr even; Bcap >= 1; Bp >= 0.
 * Mean, normalisation and rotation in float32, one rounding to `in_dtype`.
 */
typedef struct kvr_qsa_args {
    const void* raw_index_keys;
    kvr_dtype in_dtype;
    int64_t N, L, Di;
    void* block_keys;
    int64_t Bcap;
    const int64_t* key_length;
    int64_t key_length_len;
    const void* rope_cos;
    const void* rope_sin;
    int64_t Dr;
    const void* k_norm_weight;
    const void* past_incomplete_raw_keys;
    const void* past_incomplete_rope;
    int64_t key_block_size;
    float eps;
    void* next_incomplete_raw_keys;
    void* next_incomplete_rope;
    int32_t* dev_status;
    kvr_qsa_rope rope_layout;
    const void* past_block_index_keys;
    int64_t Bp;
    int32_t params_ready;
    int32_t key_length_late;
} kvr_qsa_args;

kvr_status qsa_prepare(const kvr_qsa_args* args, cudaStream_t stream);

/*
 * Arguments of dynamic_quant(): DynamicQuant of q^N from "aclnnMlaPrologV3WeightNz"
 * ("Formula": dequantScaleQNope = RowMax(abs(q^N)) / 127,
 * q^N = round(q^N / dequantScaleQNope); "Shape restrictions": one scale per
 * (token, head), shape (T, N, 1)).
 *
 *   q_nope          [rows, Hckv] input, `in_dtype` (bf16 or f16); rows = T*N
 *                   (tokens x heads). Row r starts q_row_stride elements after
 *                   row r-1 (0 means Hckv).
 *   q_out           [rows, Hckv] int8 codes, dense.
 *   dequant_scale   [rows] float32 scales.
 *
 *   exact           0 (default) or 1, see below.
 *
 * Per row: dequant_scale = RowMax(|q|) / 127, rounded once to float32 (the
 * IEEE division), and code = round-half-even(q / (RowMax/127)) =
 * round-half-even(q * 127 / RowMax), clamped to [-127, 127]; an all-zero row
 * gets scale 0 and codes 0. With exact = 0 each code is computed from a
 * float32 reciprocal product and is within one code of that value (equal to
 * it unless q * 127 / RowMax lies within 2^-15 of a half-integer). With
 * exact = 1 those near-tie codes are recomputed from the exact rational, so
 * every code equals it; this costs about a third more time on bf16 rows,
 * where such quotients are common. Inputs are finite. Limits: rows >= 0,
 * Hckv >= 1; the outputs must not overlap the input (KVR_ERR_ALIAS).
 */
typedef struct kvr_dq_args {
    const void* q_nope;
    kvr_dtype in_dtype;
    int64_t rows, Hckv;
    int64_t q_row_stride;
    int8_t* q_out;
    float* dequant_scale;
    int32_t exact;
} kvr_dq_args;

kvr_status dynamic_quant(const kvr_dq_args* args, cudaStream_t stream);

/* Measurement helper (no counterpart on the pages): a 16-byte vectorised
 * device-to-device copy of `bytes` bytes (a multiple of 16, both pointers
 * 16-byte aligned), used to measure the achievable HBM bandwidth in the same
 * process as the kernels above. */
kvr_status kvr_device_copy(void* dst, const void* src, int64_t bytes, cudaStream_t stream);

/* Failure-detection check (no counterpart on the pages): one small kernel
 * waits, the way the pipeline kernels wait on their copies, for an mbarrier
 * phase that never completes (it expects bytes that no copy delivers). It
 * gives up after `limit_ns` nanoseconds (1e3 .. 1e9), or after
 * `abort_after_ns` (0 = never; at most limit_ns) when a second warp raises
 * the abort flag the pipelines use, then ORs KVR_DEVERR_TIMEOUT into the
 * device word *dev_status and returns: nothing traps and the context stays
 * usable. Asynchronous on `stream`. */
kvr_status kvr_check_bounded_wait(int32_t* dev_status, int64_t limit_ns, int64_t abort_after_ns, cudaStream_t stream);

/* Test helper (no counterpart on the pages): a late producer of device
 * words. One small kernel, launched with programmatic dependent launch like
 * the calls above, waits for its own predecessor on `stream`, lets the next
 * launch on `stream` start at once, spins for `delay_ns` nanoseconds
 * (0 .. 1e8) and only then copies `count` (0 .. 2^20) int64 words from the
 * device array `src` to the device array `dst` (both 8-byte aligned, not
 * overlapping; the caller keeps both alive until the stream has passed the
 * kernel). A call launched right after it therefore starts while `dst` still
 * holds its old values, and must see the new ones after its dependency wait:
 * the check that qsa_prepare's default form takes key_length only after the
 * wait (its earlier read is a prefetch hint). Returns KVR_ERR_SHAPE for a
 * count or delay out of range or a misaligned pointer, KVR_ERR_NULL for a
 * null pointer (count > 0), KVR_ERR_ALIAS for overlapping arrays; count 0
 * launches nothing. Asynchronous on `stream`. */
kvr_status kvr_store_after_delay(int64_t* dst, const int64_t* src, int64_t count, int64_t delay_ns,
                                 cudaStream_t stream);

/* Debug validation of kv_rmsnorm_rope_cache's index (off by default; the
 * environment variable KVR_DEBUG_VALIDATE=1 turns it on at the first call,
 * this call sets it either way, for every thread). When on, each
 * kv_rmsnorm_rope_cache / kv_rmsnorm_rope_cache_staged call copies its index
 * to the host, synchronising `stream`, and returns KVR_ERR_INDEX without
 * launching when an entry is out of range or two tokens name the same cache
 * row ("aclnnKvRmsNormRopeCache", "Restrictions on index": distinct within a
 * batch in Norm mode, anywhere in the paged modes; in PA_BLK_BSND every
 * token's row is checked and must stay inside its entry's block). Without
 * it, repeated rows leave an unspecified winner and out-of-range entries are
 * skipped and reported through dev_status. A call made while its stream is
 * being captured into a CUDA graph is not checked. For debugging only: the
 * copy and the synchronisation cost far more than the call. */
void kvr_set_debug_validate(int on);

/* Static description of a status code (never NULL). */
const char* kvr_status_string(kvr_status status);

/* KVR_ABI_VERSION of the loaded library. */
int kvr_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVR_H */
