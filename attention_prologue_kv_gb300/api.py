"""Python entry points: marshal torch CUDA tensors into the C ABI of
libkvr.so and call it on the current (or given) stream. Argument checking
beyond marshalling (shapes, ranges, aliasing) is done by the library, whose
status is raised as KvrError. Calls are asynchronous; nothing synchronises."""
import ctypes

import torch

from . import _native as N

_IN_DTYPES = {torch.bfloat16: N.KVR_BF16, torch.float16: N.KVR_F16}
_CACHE_DTYPES = {
    torch.bfloat16: N.KVR_BF16,
    torch.float16: N.KVR_F16,
    torch.int8: N.KVR_INT8,
    torch.float8_e4m3fn: N.KVR_FP8_E4M3FN,
    torch.float8_e5m2: N.KVR_FP8_E5M2,
}


class KvrError(RuntimeError):
    def __init__(self, code, where):
        self.code = int(code)
        super().__init__("%s: %s (status %d)" % (where, N.status_string(code), self.code))


def _cuda(t, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor: the kernels run on the GPU only" % name)
    return t


def _ptr(t, name, contiguous=True):
    if t is None:
        return None
    _cuda(t, name)
    if contiguous and not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else int(stream)


def _kv_rows(kv):
    """(Bkv, Skv, row stride in elements) of a [Bkv,1,Skv,D] / [Bkv,Skv,D] / [T,D]
    tensor whose rows are uniformly strided and whose last dim is dense."""
    if kv.stride(-1) != 1:
        raise ValueError("kv must be dense along its last dimension")
    if kv.dim() == 4:
        if kv.shape[1] != 1:
            raise ValueError("kv must be [Bkv, 1, Skv, D]: the head axis N is 1")
        B, S = kv.shape[0], kv.shape[2]
        sb, ss = kv.stride(0), kv.stride(2)
    elif kv.dim() == 3:
        B, S = kv.shape[0], kv.shape[1]
        sb, ss = kv.stride(0), kv.stride(1)
    elif kv.dim() == 2:
        B, S = kv.shape[0], 1
        sb, ss = kv.stride(0), kv.stride(0)
    else:
        raise ValueError("kv must be 2-D, 3-D or 4-D")
    stride = ss if S > 1 else sb
    if B > 1 and S > 0 and sb != S * stride:
        raise ValueError("kv rows must be uniformly strided")
    return B, S, stride


def _cache_dims(c, name):
    _cuda(c, name)
    if not c.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if c.dim() == 4 and c.shape[2] != 1:
        raise ValueError("%s must be [d0, d1, 1, D*]" % name)
    if c.dim() not in (3, 4):
        raise ValueError("%s must be [d0, d1, 1, D*] or [d0, d1, D*]" % name)
    if c.dtype not in _CACHE_DTYPES:
        raise ValueError("%s has unsupported dtype %s" % (name, c.dtype))
    return c.shape[0], c.shape[1], c.shape[-1]


def _kv_args(kv, gamma, cos, sin, index, ckv_cache, k_cache, cache_mode, eps, ckv_scale, k_scale,
             kc_scale, dev_status, params_ready=False):
    _cuda(kv, "kv")
    Bkv, Skv, stride = _kv_rows(kv)
    if kv.dtype not in _IN_DTYPES:
        raise ValueError("kv must be bfloat16 or float16")
    Dv = gamma.numel()
    Dk = kv.shape[-1] - Dv
    d0, d1, _ = _cache_dims(ckv_cache, "ckv_cache")
    k0, k1, _ = _cache_dims(k_cache, "k_cache")
    if (k0, k1) != (d0, d1):
        raise ValueError("ckv_cache and k_cache must share their leading dims")
    if cache_mode not in N.CACHE_MODES:
        raise ValueError("cache_mode must be one of %s" % list(N.CACHE_MODES))
    for t, name in ((gamma, "gamma"), (cos, "cos"), (sin, "sin")):
        if t.dtype != kv.dtype:
            raise ValueError("%s must have kv's dtype" % name)
    if index.dtype != torch.int64:
        raise ValueError("index must be int64")
    # The kernels read exactly this many index entries (one per token, or one
    # per BlockSize tokens of a sequence in PA_BLK_BSND); the C ABI cannot
    # check a buffer's length, so the binding does.
    n_index = Bkv * (-(-Skv // d1) if cache_mode == "PA_BLK_BSND" else Skv)
    if index.numel() != n_index:
        raise ValueError("index must have %d entries for %s (Bkv=%d, Skv=%d), got %d"
                         % (n_index, cache_mode, Bkv, Skv, index.numel()))
    for t, name in ((ckv_scale, "ckv_scale"), (k_scale, "k_scale")):
        if t is not None and t.dtype != torch.float32:
            raise ValueError("%s must be float32" % name)
    for t, name in ((cos, "cos"), (sin, "sin")):
        if t.numel() != Bkv * Skv * Dk:
            raise ValueError("%s must have Bkv*Skv*Dk = %d elements, got %d" % (name, Bkv * Skv * Dk, t.numel()))
    if dev_status is not None and dev_status.numel() < 1:
        raise ValueError("dev_status must have one element")
    if dev_status is not None and dev_status.dtype != torch.int32:
        raise ValueError("dev_status must be int32")
    return N.KvArgs(
        kv=kv.data_ptr(), in_dtype=_IN_DTYPES[kv.dtype], Bkv=Bkv, Skv=Skv, Dv=Dv, Dk=Dk,
        kv_row_stride=stride, gamma=_ptr(gamma, "gamma"), cos=_ptr(cos, "cos"),
        sin=_ptr(sin, "sin"), index=_ptr(index, "index"), mode=N.CACHE_MODES[cache_mode],
        cache_d0=d0, cache_d1=d1,
        ckv_cache=ckv_cache.data_ptr(), ckv_dtype=_CACHE_DTYPES[ckv_cache.dtype],
        ckv_scale=_ptr(ckv_scale, "ckv_scale"),
        ckv_scale_len=0 if ckv_scale is None else ckv_scale.numel(),
        k_cache=k_cache.data_ptr(), k_dtype=_CACHE_DTYPES[k_cache.dtype],
        k_scale=_ptr(k_scale, "k_scale"), k_scale_len=0 if k_scale is None else k_scale.numel(),
        eps=float(eps), kc_scale=float(kc_scale), dev_status=_ptr(dev_status, "dev_status"),
        params_ready=1 if params_ready else 0)


def kv_rmsnorm_rope_cache(kv, gamma, cos, sin, index, ckv_cache, k_cache, *,
                          cache_mode="PA_BSND", eps=1e-6, ckv_scale=None, k_scale=None,
                          kc_scale=1.0, dev_status=None, params_ready=False, stream=None):
    """Fused RMSNorm(kv[..., :Dv]) -> ckv_cache and interleaved RoPE(kv[..., Dv:]) ->
    k_cache, scattered by `index` (-1 skips). Dv = gamma.numel().

    kv [Bkv, 1, Skv, D] (bf16/f16; rows may be strided, e.g. a column slice),
    cos/sin [Bkv, 1, Skv, Dk], index int64 (layout per cache_mode),
    caches [d0, d1, 1, Dv] and [d0, d1, 1, Dk] (bf16/f16 like kv, or int8 /
    float8_e4m3fn / float8_e5m2 with a float32 scale of length D* or 1).
    `dev_status` (int32, 1 element) collects device-side error bits.
    params_ready=True promises that the kernel launched just before this call
    on the stream does not write gamma or the scales (model weights and
    calibrated scales): they are then read while that kernel still runs."""
    a = _kv_args(kv, gamma, cos, sin, index, ckv_cache, k_cache, cache_mode, eps, ckv_scale,
                 k_scale, kc_scale, dev_status, params_ready)
    st = N.lib().kv_rmsnorm_rope_cache(ctypes.byref(a), _stream(stream))
    if st != N.KVR_OK:
        raise KvrError(st, "kv_rmsnorm_rope_cache")


class PreparedCall:
    """An entry point with its arguments marshalled once. Calling it launches
    on `stream` (default: the current stream at call time) with the same
    tensors, whose contents may change between calls; the caller keeps the
    tensors alive and unmoved for the object's lifetime. For serving loops
    that reuse fixed buffers every step: a call costs the C entry point only."""

    def __init__(self, fn, args, name, keep, staged_fn=None):
        self._fn = fn
        self._args = args
        self._ref = ctypes.byref(args)
        self._name = name
        self._keep = keep
        self._staged_fn = staged_fn

    def __call__(self, stream=None):
        st = self._fn(self._ref, _stream(stream))
        if st != N.KVR_OK:
            raise KvrError(st, self._name)

    def staged(self, host_src, dev_dst, nbytes, host_status=None, stream=None):
        """The call with host staging, enqueued in one C call: copy `nbytes`
        from pinned host memory `host_src` to device memory `dev_dst` (where
        the bound input tensors live), run the call, then copy the device
        status word to pinned host memory `host_status` (optional; needs
        dev_status bound). Each of host_src, dev_dst, host_status is a tensor
        or a raw address; raw addresses skip the checks. Asynchronous: the
        host buffers must stay valid until the stream has passed them."""
        if self._staged_fn is None:
            raise TypeError("%s has no host-staged form" % self._name)
        src = _host_addr(host_src, "host_src")
        dst = dev_dst if isinstance(dev_dst, int) else _ptr(dev_dst, "dev_dst")
        hst = None if host_status is None else _host_addr(host_status, "host_status")
        st = self._staged_fn(self._ref, src, dst, int(nbytes), hst, _stream(stream))
        if st != N.KVR_OK:
            raise KvrError(st, self._name + "_staged")


_EMPTY_PAST = {}


def _past_ptr(past, device):
    """Address of past_block_index_keys for the C call. An empty buffer
    (Bp = 0) still selects the concat-output form, but PyTorch gives it no
    address and NULL means in place; a small per-device placeholder, never
    read (Bp = 0), stands in for it."""
    if past is None:
        return None
    if past.numel() > 0:
        return _ptr(past, "past_block_index_keys")
    _cuda(past, "past_block_index_keys")
    key = str(device)
    if key not in _EMPTY_PAST:
        _EMPTY_PAST[key] = torch.zeros(8, dtype=torch.int16, device=device)
    return _EMPTY_PAST[key].data_ptr()


def _host_addr(t, name):
    if isinstance(t, int):
        return t
    if t.is_cuda or not t.is_pinned():
        raise ValueError("%s must be pinned host memory" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def prepare_kv_rmsnorm_rope_cache(kv, gamma, cos, sin, index, ckv_cache, k_cache, *,
                                  cache_mode="PA_BSND", eps=1e-6, ckv_scale=None, k_scale=None,
                                  kc_scale=1.0, dev_status=None, params_ready=False):
    """kv_rmsnorm_rope_cache with its arguments bound once (see PreparedCall)."""
    a = _kv_args(kv, gamma, cos, sin, index, ckv_cache, k_cache, cache_mode, eps, ckv_scale,
                 k_scale, kc_scale, dev_status, params_ready)
    keep = (kv, gamma, cos, sin, index, ckv_cache, k_cache, ckv_scale, k_scale, dev_status)
    return PreparedCall(N.lib().kv_rmsnorm_rope_cache, a, "kv_rmsnorm_rope_cache", keep,
                        staged_fn=N.lib().kv_rmsnorm_rope_cache_staged)


def qsa_prepare(raw_index_keys, block_keys, key_length, rope_cos, rope_sin, k_norm_weight,
                past_incomplete_raw_keys, past_incomplete_rope, key_block_size, epsilon=1e-6, *,
                next_incomplete_raw_keys=None, next_incomplete_rope=None, dev_status=None,
                rope_layout="interleave_last", past_block_index_keys=None, params_ready=False,
                key_length_late=False, stream=None):
    """QSA block-key prepare. Positional arguments follow the qsa_prepare
    parameter list; `block_keys` [N, Bcap, Di] holds the past block keys and
    receives the new ones in place (block j at row j). rope_cos/rope_sin
    [N, L, Dr] (or both None), k_norm_weight [Di] or None,
    past_incomplete_raw_keys [N, kbs-1, Di], past_incomplete_rope [N, 2*Dr] or
    None, key_length int64 [N] or [1] = valid tokens after this call.
    Optional carry outputs next_incomplete_raw_keys / next_incomplete_rope.
    rope_layout: "interleave_last" (default), "interleave_first", "half_last"
    or "half_first" (which Dr channels rotate; interleaved or rotate-half
    pairs). past_block_index_keys [N, Bp, Di]: concat-output form, its rows
    j < floor(P/kbs) are copied into block_keys first. params_ready=True
    promises that the kernel launched just before this call writes none of
    key_length, rope_cos/rope_sin, past_incomplete_rope and k_norm_weight,
    so the compiled-shape kernel may read them before its dependency wait.
    Without it, that kernel reads key_length before the wait only as a
    prefetch hint; key_length_late=True says the kernel launched just before
    writes key_length, and skips the hint (same results, no second pass when
    the hint would be stale)."""
    raw = _cuda(raw_index_keys, "raw_index_keys")
    if raw.dim() != 3:
        raise ValueError("raw_index_keys must be [N, L, Di]")
    if raw.dtype not in _IN_DTYPES:
        raise ValueError("raw_index_keys must be bfloat16 or float16")
    Nn, L, Di = raw.shape
    if block_keys.dim() != 3 or block_keys.dtype != raw.dtype:
        raise ValueError("block_keys must be [N, Bcap, Di] with raw_index_keys' dtype")
    if key_length.dtype != torch.int64:
        raise ValueError("key_length must be int64")
    for t, name in ((rope_cos, "rope_cos"), (rope_sin, "rope_sin"), (k_norm_weight, "k_norm_weight"),
                    (past_incomplete_raw_keys, "past_incomplete_raw_keys"),
                    (past_incomplete_rope, "past_incomplete_rope"),
                    (next_incomplete_raw_keys, "next_incomplete_raw_keys"),
                    (next_incomplete_rope, "next_incomplete_rope"),
                    (past_block_index_keys, "past_block_index_keys")):
        if t is not None and t.dtype != raw.dtype:
            raise ValueError("%s must have raw_index_keys' dtype" % name)
    if rope_layout not in N.QSA_ROPE_LAYOUTS:
        raise ValueError("rope_layout must be one of %s" % sorted(N.QSA_ROPE_LAYOUTS))
    Bp = 0
    if past_block_index_keys is not None:
        if past_block_index_keys.dim() != 3 or past_block_index_keys.shape[0] != Nn or \
                past_block_index_keys.shape[2] != Di:
            raise ValueError("past_block_index_keys must be [N, Bp, Di]")
        Bp = past_block_index_keys.shape[1]
    if dev_status is not None and dev_status.dtype != torch.int32:
        raise ValueError("dev_status must be int32")
    Dr = rope_cos.shape[-1] if rope_cos is not None else 0
    # The C ABI cannot check a buffer's length: every tensor the kernels read
    # or write must have exactly the size its role implies.
    kbs = int(key_block_size)
    sizes = ((rope_cos, "rope_cos", Nn * L * Dr), (rope_sin, "rope_sin", Nn * L * Dr),
             (k_norm_weight, "k_norm_weight", Di),
             (past_incomplete_raw_keys, "past_incomplete_raw_keys", Nn * (kbs - 1) * Di),
             (past_incomplete_rope, "past_incomplete_rope", Nn * 2 * Dr),
             (next_incomplete_raw_keys, "next_incomplete_raw_keys", Nn * (kbs - 1) * Di),
             (next_incomplete_rope, "next_incomplete_rope", Nn * 2 * Dr))
    for t, name, n in sizes:
        if t is not None and kbs > 1 and t.numel() != n:
            raise ValueError("%s must have %d elements, got %d" % (name, n, t.numel()))
    if key_length.numel() not in (1, Nn):
        raise ValueError("key_length must have 1 or N elements")
    if dev_status is not None and dev_status.numel() < 1:
        raise ValueError("dev_status must have one element")
    a = N.QsaArgs(
        raw_index_keys=_ptr(raw, "raw_index_keys"), in_dtype=_IN_DTYPES[raw.dtype], N=Nn, L=L, Di=Di,
        block_keys=_ptr(block_keys, "block_keys"), Bcap=block_keys.shape[1],
        key_length=_ptr(key_length, "key_length"), key_length_len=key_length.numel(),
        rope_cos=_ptr(rope_cos, "rope_cos"), rope_sin=_ptr(rope_sin, "rope_sin"), Dr=Dr,
        k_norm_weight=_ptr(k_norm_weight, "k_norm_weight"),
        past_incomplete_raw_keys=_ptr(past_incomplete_raw_keys, "past_incomplete_raw_keys"),
        past_incomplete_rope=_ptr(past_incomplete_rope, "past_incomplete_rope"),
        key_block_size=int(key_block_size), eps=float(epsilon),
        next_incomplete_raw_keys=_ptr(next_incomplete_raw_keys, "next_incomplete_raw_keys"),
        next_incomplete_rope=_ptr(next_incomplete_rope, "next_incomplete_rope"),
        dev_status=_ptr(dev_status, "dev_status"), rope_layout=N.QSA_ROPE_LAYOUTS[rope_layout],
        past_block_index_keys=_past_ptr(past_block_index_keys, raw.device), Bp=Bp,
        params_ready=1 if params_ready else 0, key_length_late=1 if key_length_late else 0)
    if block_keys.shape[0] != Nn or block_keys.shape[2] != Di:
        raise ValueError("block_keys must be [N, Bcap, Di]")
    st = N.lib().qsa_prepare(ctypes.byref(a), _stream(stream))
    if st != N.KVR_OK:
        raise KvrError(st, "qsa_prepare")


def set_debug_validate(on):
    """Debug validation of kv_rmsnorm_rope_cache's index (off by default, or
    on from the start with KVR_DEBUG_VALIDATE=1): each call then copies its
    index to the host, synchronising its stream, and raises KvrError
    (KVR_ERR_INDEX) without launching when an entry is out of range or two
    tokens name the same cache row. Calls under CUDA-graph capture are not
    checked. Slow: for debugging only."""
    N.lib().kvr_set_debug_validate(1 if on else 0)


def check_bounded_wait(dev_status, limit_us, abort_after_us=0, stream=None):
    """Failure-detection check: a kernel waits for an mbarrier phase that
    never completes and gives up after `limit_us` microseconds (or when a
    second warp raises the abort flag after `abort_after_us`), OR-ing
    KVR_DEVERR_TIMEOUT into `dev_status` (int32, device). Asynchronous."""
    if dev_status.dtype != torch.int32 or dev_status.numel() < 1:
        raise ValueError("dev_status must be an int32 tensor with one element")
    st = N.lib().kvr_check_bounded_wait(_ptr(dev_status, "dev_status"), int(limit_us * 1000),
                                        int(abort_after_us * 1000), _stream(stream))
    if st != N.KVR_OK:
        raise KvrError(st, "kvr_check_bounded_wait")


def store_after_delay(dst, src, delay_us, stream=None):
    """Test helper: a kernel (programmatic dependent launch) that lets the
    next launch on `stream` start at once, waits `delay_us` microseconds and
    then copies `src` into `dst` (contiguous int64 CUDA tensors of the same
    size): a late producer of an input such as key_length. Asynchronous; keep
    both tensors alive until the stream has passed it."""
    for t, name in ((dst, "dst"), (src, "src")):
        if t.dtype != torch.int64 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("%s must be a contiguous CUDA int64 tensor" % name)
    if dst.numel() != src.numel():
        raise ValueError("dst and src must have the same number of elements")
    st = N.lib().kvr_store_after_delay(dst.data_ptr(), src.data_ptr(), dst.numel(), int(delay_us * 1000),
                                       _stream(stream))
    if st != N.KVR_OK:
        raise KvrError(st, "kvr_store_after_delay")


def dynamic_quant(q_nope, q_out, dequant_scale, *, exact=False, stream=None):
    """DynamicQuant of q^N: per row (last axis, e.g. q^N [T, N, Hckv] gives
    T*N rows) dequant_scale = RowMax(|q|)/127 and q_out = round(q/scale) as
    int8. q_nope bf16/f16 with a dense last axis and uniformly strided rows;
    q_out int8 of q_nope's shape (dense); dequant_scale float32 with one
    element per row (e.g. [T, N, 1]). Codes are within one code of
    round(q*127/RowMax); exact=True makes every code equal to it."""
    _cuda(q_nope, "q_nope")
    if q_nope.dtype not in _IN_DTYPES:
        raise ValueError("q_nope must be bfloat16 or float16")
    if q_nope.stride(-1) != 1:
        raise ValueError("q_nope must be dense along its last dimension")
    H = q_nope.shape[-1]
    rows = q_nope.numel() // H if H else 0
    try:
        q2 = q_nope.view(-1, H)   # never a silent copy: the kernel runs asynchronously
    except RuntimeError:
        raise ValueError("q_nope rows must be uniformly strided")
    stride = q2.stride(0) if rows > 1 else H
    if q_out.dtype != torch.int8 or q_out.numel() != q_nope.numel():
        raise ValueError("q_out must be int8 with q_nope's number of elements")
    if dequant_scale.dtype != torch.float32 or dequant_scale.numel() != rows:
        raise ValueError("dequant_scale must be float32 with one element per row")
    a = N.DqArgs(q_nope=q2.data_ptr(), in_dtype=_IN_DTYPES[q_nope.dtype], rows=rows, Hckv=H,
                 q_row_stride=stride, q_out=_ptr(q_out, "q_out"),
                 dequant_scale=_ptr(dequant_scale, "dequant_scale"), exact=1 if exact else 0)
    st = N.lib().dynamic_quant(ctypes.byref(a), _stream(stream))
    if st != N.KVR_OK:
        raise KvrError(st, "dynamic_quant")


def device_copy(dst, src, stream=None):
    """16-byte vectorised device copy of src into dst (same byte size); the
    in-process HBM bandwidth reference."""
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("dst and src must have the same byte size")
    st = N.lib().kvr_device_copy(_ptr(dst, "dst"), _ptr(src, "src"), nbytes, _stream(stream))
    if st != N.KVR_OK:
        raise KvrError(st, "kvr_device_copy")
