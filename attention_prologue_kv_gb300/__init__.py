"""GB300-native attention-prologue key path: fused KV RMSNorm + interleaved
RoPE + quantise + cache scatter, and the QSA block-key prepare.

The compute runs in hand-written sm_103a CUDA kernels behind the C ABI of
libkvr.so (include/kvr.h); this package holds the thin ctypes binding, the
build step and the seeded synthetic workloads. There is no CPU fallback:
calling an entry point without the built library raises.
"""
from .api import (KvrError, PreparedCall, check_bounded_wait, device_copy,  # noqa: E402,F401
                  dynamic_quant, kv_rmsnorm_rope_cache, prepare_kv_rmsnorm_rope_cache, qsa_prepare,
                  set_debug_validate, store_after_delay)
