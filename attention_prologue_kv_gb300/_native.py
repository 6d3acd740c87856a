"""ctypes view of libkvr.so (include/kvr.h): structure layouts, enums and the
loaded library. Loading fails loudly when the library has not been built;
there is no fallback path."""
import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkvr.so")
ABI_VERSION = 10   # KVR_ABI_VERSION of include/kvr.h these structures mirror

# kvr_status
KVR_OK, KVR_ERR_NULL, KVR_ERR_SHAPE, KVR_ERR_DTYPE, KVR_ERR_MODE, KVR_ERR_ALIAS, KVR_ERR_CUDA, KVR_ERR_INDEX = range(8)
# device status bits
KVR_DEVERR_INDEX = 0x1
KVR_DEVERR_KEY_LENGTH = 0x2
KVR_DEVERR_BLOCK_CAP = 0x4
KVR_DEVERR_TIMEOUT = 0x8
KVR_DEVERR_PAST_BLOCKS = 0x10
# kvr_qsa_rope
QSA_ROPE_LAYOUTS = {"interleave_last": 0, "interleave_first": 1, "half_last": 2, "half_first": 3}
# kvr_dtype
KVR_BF16, KVR_F16, KVR_INT8, KVR_FP8_E4M3FN, KVR_FP8_E5M2 = range(5)
# kvr_cache_mode
CACHE_MODES = {"Norm": 0, "PA_BSND": 1, "PA_BLK_BSND": 2}

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_f32 = ctypes.c_float


class KvArgs(ctypes.Structure):
    _fields_ = [
        ("kv", _vp), ("in_dtype", _int),
        ("Bkv", _i64), ("Skv", _i64), ("Dv", _i64), ("Dk", _i64),
        ("kv_row_stride", _i64),
        ("gamma", _vp), ("cos", _vp), ("sin", _vp), ("index", _vp),
        ("mode", _int), ("cache_d0", _i64), ("cache_d1", _i64),
        ("ckv_cache", _vp), ("ckv_dtype", _int), ("ckv_scale", _vp), ("ckv_scale_len", _i64),
        ("k_cache", _vp), ("k_dtype", _int), ("k_scale", _vp), ("k_scale_len", _i64),
        ("eps", _f32), ("kc_scale", _f32),
        ("dev_status", _vp), ("params_ready", ctypes.c_int32),
    ]


class QsaArgs(ctypes.Structure):
    _fields_ = [
        ("raw_index_keys", _vp), ("in_dtype", _int),
        ("N", _i64), ("L", _i64), ("Di", _i64),
        ("block_keys", _vp), ("Bcap", _i64),
        ("key_length", _vp), ("key_length_len", _i64),
        ("rope_cos", _vp), ("rope_sin", _vp), ("Dr", _i64),
        ("k_norm_weight", _vp),
        ("past_incomplete_raw_keys", _vp), ("past_incomplete_rope", _vp),
        ("key_block_size", _i64), ("eps", _f32),
        ("next_incomplete_raw_keys", _vp), ("next_incomplete_rope", _vp),
        ("dev_status", _vp),
        ("rope_layout", _int), ("past_block_index_keys", _vp), ("Bp", _i64),
        ("params_ready", ctypes.c_int32), ("key_length_late", ctypes.c_int32),
    ]


class DqArgs(ctypes.Structure):
    _fields_ = [
        ("q_nope", _vp), ("in_dtype", _int),
        ("rows", _i64), ("Hckv", _i64), ("q_row_stride", _i64),
        ("q_out", _vp), ("dequant_scale", _vp), ("exact", ctypes.c_int32),
    ]


EXPORTS = ("kv_rmsnorm_rope_cache", "kv_rmsnorm_rope_cache_staged", "kv_rmsnorm_rope_cache_staged_static",
           "qsa_prepare", "dynamic_quant", "kvr_device_copy",
           "kvr_check_bounded_wait", "kvr_store_after_delay", "kvr_set_debug_validate",
           "kvr_status_string", "kvr_abi_version")

_lib = None


def lib():
    """The loaded libkvr.so (loaded once)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "libkvr.so is not built (expected at %s). Build it with "
            "`python -m attention_prologue_kv_gb300.build`; there is no CPU fallback." % LIB_PATH)
    # PyTorch loads libcudart.so.13 first so that libkvr.so binds to the same runtime.
    import torch  # noqa: F401
    L = ctypes.CDLL(LIB_PATH)
    L.kv_rmsnorm_rope_cache.argtypes = [ctypes.POINTER(KvArgs), _vp]
    L.kv_rmsnorm_rope_cache.restype = _int
    L.kv_rmsnorm_rope_cache_staged.argtypes = [ctypes.POINTER(KvArgs), _vp, _vp, _i64, _vp, _vp]
    L.kv_rmsnorm_rope_cache_staged.restype = _int
    L.kv_rmsnorm_rope_cache_staged_static.argtypes = [ctypes.POINTER(KvArgs), _vp, _i64, _i64, _i64, _i64, _i64,
                                                      _vp, _vp]
    L.kv_rmsnorm_rope_cache_staged_static.restype = _int
    L.qsa_prepare.argtypes = [ctypes.POINTER(QsaArgs), _vp]
    L.qsa_prepare.restype = _int
    L.dynamic_quant.argtypes = [ctypes.POINTER(DqArgs), _vp]
    L.dynamic_quant.restype = _int
    L.kvr_check_bounded_wait.argtypes = [_vp, _i64, _i64, _vp]
    L.kvr_check_bounded_wait.restype = _int
    L.kvr_store_after_delay.argtypes = [_vp, _vp, _i64, _i64, _vp]
    L.kvr_store_after_delay.restype = _int
    L.kvr_set_debug_validate.argtypes = [_int]
    L.kvr_set_debug_validate.restype = None
    L.kvr_device_copy.argtypes = [_vp, _vp, _i64, _vp]
    L.kvr_device_copy.restype = _int
    L.kvr_status_string.argtypes = [_int]
    L.kvr_status_string.restype = ctypes.c_char_p
    L.kvr_abi_version.argtypes = []
    L.kvr_abi_version.restype = _int
    if L.kvr_abi_version() != ABI_VERSION:
        raise RuntimeError("libkvr.so has ABI version %d, the binding expects %d: rebuild it with "
                           "`python -m attention_prologue_kv_gb300.build`" % (L.kvr_abi_version(), ABI_VERSION))
    _lib = L
    return L


def status_string(code):
    return lib().kvr_status_string(int(code)).decode()
