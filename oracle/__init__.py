"""Oracle: a plain, slow, obviously correct CPU (float64 NumPy) statement of
what the attention-prologue key path computes.

TEST INFRASTRUCTURE, NOT PRODUCT. Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it. It shares no code with the CUDA
path (no kernels, headers, helpers, tables or constants) and imports
nothing from it; the only thing both sides use is the seeded input
generator, which holds none of the method's arithmetic.

Modules:
  encoders               float64 -> cache codes (bf16, f16, int8, FP8 E4M3FN, FP8 E5M2)
  kv_rmsnorm_rope_cache  RMSNorm + interleaved RoPE + quantise + scatter
  qsa_prepare            QSA block-key prepare with carry across calls
  dynamic_quant          DynamicQuant of q^N: per-row RowMax/127 scale, int8 codes

Every function is pinned by `-m "not gpu"` tests to closed forms, invariants,
hand-worked toys (tests/golden) or library routines; no part is
"parity unpinned".
"""
from . import encoders
from .kv_rmsnorm_rope_cache import (NORM, PA_BLK_BSND, PA_BSND, STATUS_INDEX,
                                    cache_slot, interleave_rope, kv_values, quantise,
                                    ref_kv_rmsnorm_rope_cache,
                                    ref_kv_rmsnorm_rope_cache_loop, rms_norm)
from .qsa_prepare import (ROPE_LAYOUTS, STATUS_BLOCK_CAP, STATUS_KEY_LENGTH,
                          STATUS_PAST_BLOCKS, ref_qsa_prepare, rotate_half_rope)
from .dynamic_quant import ref_dynamic_quant

__all__ = [
    "encoders", "NORM", "PA_BSND", "PA_BLK_BSND", "STATUS_INDEX", "STATUS_KEY_LENGTH",
    "STATUS_BLOCK_CAP", "STATUS_PAST_BLOCKS", "ROPE_LAYOUTS", "rotate_half_rope", "cache_slot", "interleave_rope", "kv_values", "quantise", "rms_norm",
    "ref_kv_rmsnorm_rope_cache", "ref_kv_rmsnorm_rope_cache_loop", "ref_qsa_prepare",
    "ref_dynamic_quant",
]
