"""Oracle for the QSA block-key prepare.

Test infrastructure only (see oracle/__init__.py). Plain float64 NumPy,
written from the page "openvino.opset17.qsa_prepare" (docs.openvino.ai):

* summary: one index key per key block completed by the new tokens; a block
  key is the mean of the raw index keys of the block's key_block_size
  consecutive tokens, RMS-normalised with k_norm_weight, then rotated with
  the RoPE of the block's first token; an empty input disables a feature.
* parameters: raw_index_keys [N, L, Di]; past_block_index_keys [N, Bp, Di];
  key_length [N] or [1] (valid key tokens per sequence); rope_cos/rope_sin
  [N, L, Dr]; k_norm_weight [Di]; past_incomplete_raw_keys [N, kbs-1, Di];
  past_incomplete_rope [N, 2*Dr] (cos and sin of the first token of the
  incomplete block); key_block_size > 1; epsilon added to the mean square.

Readings where the page is silent (each also listed with the design notes):
* key_length counts the tokens after this call, so the past length is
  P = key_length - L; a [1] key_length applies to every sequence.
* Block keys live in a buffer indexed by absolute block number; block j
  covers tokens [j*kbs, (j+1)*kbs); blocks before floor(P/kbs) and rows not
  completed stay untouched.
* The RMS normalisation is the one of the aclnnKvRmsNormRopeCache page
  ("Formulas (2) rmsNorm"); an absent k_norm_weight disables the whole
  normalisation.
* The rotation is that page's interleaved RoPE ("Formulas (1)") on the last
  Dr channels, with cos/sin of the block's first token: the new tables when
  that token is new, else past_incomplete_rope laid out as [cos | sin].
* Mean, normalisation and rotation are taken in float64 with one rounding to
  bfloat16 at the end.
* Carry-out (for chaining calls): the raw keys of the tokens after the last
  completed block, and the cos/sin of the first of them.

Variants the page leaves open, each selectable (the defaults are the readings
above):
* rope_layout: which Dr channels rotate (the last or the first) and how the
  pairs are formed: "interleave" takes (x[2i], x[2i+1]) as in the
  aclnnKvRmsNormRopeCache formula; "half" takes (x[i], x[i + Dr/2]), the
  rotate-half form. Both write the pair's results to lanes i and i + Dr/2
  with the same cos/sin lanes.
* past_block_keys (concat-output form): the output is a fresh buffer; the
  rows j < floor(P/kbs) come from past_block_index_keys [N, Bp, Di], so the
  result is the past block keys followed by the new ones. Rows the past
  buffer does not hold (Bp < floor(P/kbs)) are left untouched and raise
  STATUS_PAST_BLOCKS; past rows that fall at or beyond Bcap raise
  STATUS_BLOCK_CAP.
"""
import numpy as np

from . import encoders as enc
from .kv_rmsnorm_rope_cache import interleave_rope, rms_norm

STATUS_KEY_LENGTH = 0x2   # key_length[n] < L
STATUS_BLOCK_CAP = 0x4    # a completed block's index is beyond the block-key buffer
STATUS_PAST_BLOCKS = 0x10  # past_block_index_keys holds fewer rows than floor(P/kbs)

ROPE_LAYOUTS = ("interleave_last", "interleave_first", "half_last", "half_first")


def rotate_half_rope(x, cos, sin):
    """RoPE in the rotate-half form over the last axis: x1 = first half,
    x2 = second half, y = cat(x1,x2)*cos + cat(-x2,x1)*sin."""
    h = x.shape[-1] // 2
    x1 = x[..., :h]
    x2 = x[..., h:]
    return np.concatenate((x1, x2), axis=-1) * cos + np.concatenate((-x2, x1), axis=-1) * sin


def rotate_channels(u, c, s, layout):
    """Apply the RoPE of `layout` (one of ROPE_LAYOUTS) to the Dr channels it
    names (Dr = len(c)); the other channels pass through."""
    Dr = len(c)
    style, where = layout.split("_")
    rope = interleave_rope if style == "interleave" else rotate_half_rope
    if where == "last":
        return np.concatenate((u[:len(u) - Dr], rope(u[len(u) - Dr:], c, s)))
    return np.concatenate((rope(u[:Dr], c, s), u[Dr:]))


def ref_qsa_prepare(raw, block_keys, key_length, rope_cos, rope_sin, k_norm_weight,
                    past_raw, past_rope, key_block_size, eps=1e-6,
                    next_raw=None, next_rope=None, out_dtype="bf16",
                    rope_layout="interleave_last", past_block_keys=None, values_out=None):
    """raw [N, L, Di] f64; block_keys codes [N, Bcap, Di] (written in place);
    key_length int [N] or [1]; rope_cos/rope_sin [N, L, Dr] f64 or None;
    k_norm_weight [Di] f64 or None; past_raw [N, kbs-1, Di] f64;
    past_rope [N, 2*Dr] f64 or None; next_raw [N, kbs-1, Di] f64 / next_rope
    [N, 2*Dr] f64 optional carry outputs (written in place); rope_layout
    one of ROPE_LAYOUTS; past_block_keys codes [N, Bp, Di] or None (None:
    block_keys already holds the past keys). values_out: optional dict that
    receives, for every block key written, (n, j) -> (u, b): the float64 key
    before its rounding, and per element a bound on the magnitudes of the
    terms summed into it (the same steps applied to the mean of |key|, with
    the normalisation factor of the true mean and the magnitudes of both
    rotation terms), for judging how far a finite-precision evaluation may
    stray.
    Returns the device-status bits the call would raise."""
    if rope_layout not in ROPE_LAYOUTS:
        raise ValueError(rope_layout)
    N, L, Di = raw.shape
    kbs = int(key_block_size)
    Bcap = block_keys.shape[1]
    eps = float(eps)
    Dr = 0 if rope_cos is None else rope_cos.shape[-1]
    status = 0
    for n in range(N):
        K = int(key_length[n if len(key_length) == N else 0])
        P = K - L
        if P < 0:
            status |= STATUS_KEY_LENGTH
            continue
        f = P % kbs
        F = P - f
        if past_block_keys is not None:
            Bp = past_block_keys.shape[1]
            if Bp < P // kbs:
                status |= STATUS_PAST_BLOCKS
            for j in range(min(Bp, P // kbs)):
                if j >= Bcap:
                    status |= STATUS_BLOCK_CAP
                    break
                block_keys[n, j] = past_block_keys[n, j]

        def key(p):
            return past_raw[n, p - F] if p < P else raw[n, p - P]

        def rope_at(p):
            if p >= P:
                return rope_cos[n, p - P], rope_sin[n, p - P]
            return past_rope[n, :Dr], past_rope[n, Dr:]

        for j in range(P // kbs, K // kbs):
            rows = np.stack([key(p) for p in range(j * kbs, (j + 1) * kbs)])
            m = np.mean(rows, axis=0)
            u = m if k_norm_weight is None else rms_norm(m, k_norm_weight, eps)
            bound = np.mean(np.abs(rows), axis=0)
            if k_norm_weight is not None:   # the same normalisation factor, on magnitudes
                bound = bound * np.abs(k_norm_weight) / np.sqrt(np.mean(m * m) + eps)
            if rope_cos is not None:
                c, s = rope_at(j * kbs)
                u = rotate_channels(u, c, s, rope_layout)
                zero = np.zeros_like(c)
                bound = rotate_channels(bound, np.abs(c), zero, rope_layout) + np.abs(
                    rotate_channels(bound, zero, np.abs(s), rope_layout))
            if j >= Bcap:
                status |= STATUS_BLOCK_CAP
                continue
            block_keys[n, j] = enc.encode(u, out_dtype)
            if values_out is not None:
                values_out[(n, j)] = (u, bound)

        Fn = (K // kbs) * kbs
        if next_raw is not None:
            for p in range(Fn, K):
                next_raw[n, p - Fn] = key(p)
        if next_rope is not None and rope_cos is not None and Fn < K:
            c, s = rope_at(Fn)
            next_rope[n, :Dr] = c
            next_rope[n, Dr:] = s
    return status
