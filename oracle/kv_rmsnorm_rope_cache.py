"""Oracle for the fused KV prologue: RMSNorm (left Dv) + interleaved RoPE
(right Dk) + optional quantisation + scatter into two caches.

Test infrastructure only (see oracle/__init__.py). Plain float64 NumPy,
written from the page "aclnnKvRmsNormRopeCache" (hiascend.com, CANN
ops-transformer):

* "Description": the tail axis of kv (width D) splits into a left part of
  width Dv that is RMS-normalised and a right part of width Dk that gets RoPE;
  the two results are scattered into two caches.
* "Formulas (1) interleaveRope" and "Formulas (2) rmsNorm": the arithmetic,
  restated in `interleave_rope` and `rms_norm` below step by step.
* "Restrictions on index": the placement rules per cache mode, restated in
  `cache_slot`.
* "Restrictions on quantization scenarios": which cache may hold 8-bit codes.
  The pages give no quantisation formula; the reading used is
  q = encode(y * scale) with a per-channel (length Dv or Dk) or per-tensor
  (length 1) float32 scale and no offset.
* The kcScale factor alpha_kv of the page "aclnnMlaPrologV3WeightNz"
  ("Formula", key path: c^KV = alpha_kv * RmsNorm(...)) multiplies the
  normalised part before it is encoded.

Readings where the pages are silent: everything is float64 with no
intermediate rounding, and each output takes one rounding to its cache type
at the end: 16-bit outputs round y (or r) once, 8-bit codes are decided
from the float64 product y * scale and rounded once. eps and alpha_kv are
taken as the values the caller passes (the C call receives them as float32;
the tests hand the oracle those same values).
"""
import math

import numpy as np

from . import encoders as enc

# Cache modes (names follow the pages' cacheModeOptional values).
NORM = "Norm"
PA_BSND = "PA_BSND"
PA_BLK_BSND = "PA_BLK_BSND"

# Device-status bit raised for an index outside {-1} U [0, range).
STATUS_INDEX = 0x1


def rms_norm(x, gamma, eps):
    """rmsNorm over the last axis, as "Formulas (2)" writes it:
    square, mean, sqrt(mean + epsilon), divide, times gamma."""
    square_x = x * x
    mean_square_x = square_x.mean(axis=-1, keepdims=True)
    rms = np.sqrt(mean_square_x + eps)
    return (x / rms) * gamma


def interleave_rope(x, cos, sin):
    """interleaveRope over the last axis, as "Formulas (1)" writes it:
    x1 = even lanes, x2 = odd lanes, y = cat(x1,x2)*cos + cat(-x2,x1)*sin."""
    x1 = x[..., 0::2]
    x2 = x[..., 1::2]
    x_part1 = np.concatenate((x1, x2), axis=-1)
    x_part2 = np.concatenate((-x2, x1), axis=-1)
    return x_part1 * cos + x_part2 * sin


def quantise(y, dtype, scale):
    """Encode one result vector for a cache of element type `dtype`.

    16-bit caches take one RNE rounding from float64 and no scale. 8-bit
    caches take encode(y * scale): the float64 product, rounded once to the
    code."""
    if dtype in enc.DTYPES_16:
        if scale is not None:
            raise ValueError("a 16-bit cache takes no quantisation scale")
        return enc.encode(y, dtype)
    if scale is None:
        raise ValueError("an 8-bit cache needs a quantisation scale")
    return enc.encode(y * np.asarray(scale, dtype=np.float64), dtype)


def kv_values(kv, gamma, cos, sin, *, Dv, eps, ckv_scale=None, k_scale=None, kc_scale=1.0):
    """The float64 value each cache element encodes before its one rounding,
    per token: (vy [.., Dv], vr [.., Dk], mr [.., Dk]). vy = alpha * rmsNorm
    (times the ckv scale for an 8-bit cache), vr = interleaveRope (times the
    k scale), and mr = the sum of the magnitudes of the two RoPE terms behind
    each vr element (times |k scale|): a bound for the size of the terms a
    finite-precision evaluation of vr rounds, which can exceed |vr| by far
    when the terms cancel."""
    y = float(kc_scale) * rms_norm(kv[..., :Dv], gamma, float(eps))
    z = kv[..., Dv:]
    r = interleave_rope(z, cos, sin)
    zeros = np.zeros_like(cos)
    m = interleave_rope(np.abs(z), np.abs(cos), zeros) + np.abs(interleave_rope(np.abs(z), zeros, np.abs(sin)))
    if ckv_scale is not None:
        y = y * np.asarray(ckv_scale, dtype=np.float64)
    if k_scale is not None:
        ks = np.asarray(k_scale, dtype=np.float64)
        r = r * ks
        m = m * np.abs(ks)
    return y, r, m


def cache_slot(mode, b, s, index, Skv, d0, d1):
    """Where token (b, s) goes: returns None (skip), "bad" (index out of
    range: skipped, status raised) or the (row0, row1) cache coordinates.

    Norm      cache [Bcache=d0, Scache=d1, 1, D*], index [Bkv, Skv] in
              [-1, Scache); batch b writes cache batch b.
    PA_BSND   cache [BlockNum=d0, BlockSize=d1, 1, D*], index [Bkv*Skv] in
              [-1, BlockNum*BlockSize); slot -> (slot // BlockSize, slot % BlockSize).
    PA_BLK_BSND  index [Bkv * ceil(Skv/BlockSize)], one entry per BlockSize
              tokens, in [-1, BlockNum*BlockSize); token s of a chunk goes to
              slot index + s % BlockSize, which must stay inside the block
              that index names (the page forbids repeating index/BlockSize,
              so each entry owns one block)."""
    if mode == NORM:
        v = int(index[b, s])
        if v == -1:
            return None
        if not (0 <= v < d1):
            return "bad"
        return (b, v)
    if mode == PA_BSND:
        v = int(index[b * Skv + s])
        if v == -1:
            return None
        if not (0 <= v < d0 * d1):
            return "bad"
        return (v // d1, v % d1)
    if mode == PA_BLK_BSND:
        nblk = -(-Skv // d1)
        v = int(index[b * nblk + s // d1])
        if v == -1:
            return None
        if not (0 <= v < d0 * d1) or (v % d1) + (s % d1) >= d1:
            return "bad"
        slot = v + s % d1
        return (slot // d1, slot % d1)
    raise ValueError(mode)


def ref_kv_rmsnorm_rope_cache(kv, gamma, cos, sin, index, ckv_cache, k_cache, *,
                              Dv, mode, eps, ckv_dtype="bf16", k_dtype="bf16",
                              ckv_scale=None, k_scale=None, kc_scale=1.0):
    """Token-vectorised oracle. Writes the caches in place; returns the
    device-status bits the call would raise.

    kv      float64 [Bkv, Skv, D]        (the N = 1 head axis dropped)
    gamma   float64 [Dv]
    cos/sin float64 [Bkv, Skv, Dk]
    index   int64, Norm [Bkv, Skv]; PA_BSND [Bkv*Skv]; PA_BLK_BSND [Bkv*ceil(Skv/BlockSize)]
    ckv_cache / k_cache: code arrays (uint16 or uint8) [d0, d1, Dv] / [d0, d1, Dk]
    """
    Bkv, Skv, D = kv.shape
    eps = float(eps)
    alpha = float(kc_scale)
    d0, d1 = ckv_cache.shape[0], ckv_cache.shape[1]
    y = alpha * rms_norm(kv[..., :Dv], gamma, eps)           # [Bkv, Skv, Dv]
    r = interleave_rope(kv[..., Dv:], cos, sin)              # [Bkv, Skv, Dk]
    yq = quantise(y, ckv_dtype, ckv_scale)
    rq = quantise(r, k_dtype, k_scale)
    status = 0
    for b in range(Bkv):
        for s in range(Skv):
            slot = cache_slot(mode, b, s, index, Skv, d0, d1)
            if slot is None:
                continue
            if slot == "bad":
                status |= STATUS_INDEX
                continue
            ckv_cache[slot] = yq[b, s]
            k_cache[slot] = rq[b, s]
    return status


def ref_kv_rmsnorm_rope_cache_loop(kv, gamma, cos, sin, index, ckv_cache, k_cache, *,
                                   Dv, mode, eps, ckv_dtype="bf16", k_dtype="bf16",
                                   ckv_scale=None, k_scale=None, kc_scale=1.0):
    """The same operation as one scalar Python loop per token and element,
    for tiny inputs (a brute-force cross-check of the vectorised oracle).
    The mean square uses math.fsum, a correctly rounded sum."""
    Bkv, Skv, D = kv.shape
    Dk = D - Dv
    h = Dk // 2
    eps = float(eps)
    alpha = float(kc_scale)
    d0, d1 = ckv_cache.shape[0], ckv_cache.shape[1]
    status = 0
    for b in range(Bkv):
        for s in range(Skv):
            slot = cache_slot(mode, b, s, index, Skv, d0, d1)
            if slot is None:
                continue
            if slot == "bad":
                status |= STATUS_INDEX
                continue
            x = [float(kv[b, s, c]) for c in range(Dv)]
            ms = math.fsum(v * v for v in x) / Dv
            rms = math.sqrt(ms + eps)
            y = [alpha * ((x[c] / rms) * float(gamma[c])) for c in range(Dv)]
            z = [float(kv[b, s, Dv + c]) for c in range(Dk)]
            r = [0.0] * Dk
            for i in range(h):
                # output lane i pairs x1[i] = z[2i] with -x2[i]; lane i+h pairs x2[i] with x1[i]
                r[i] = z[2 * i] * float(cos[b, s, i]) + (-z[2 * i + 1]) * float(sin[b, s, i])
                r[i + h] = z[2 * i + 1] * float(cos[b, s, i + h]) + z[2 * i] * float(sin[b, s, i + h])
            for c in range(Dv):
                sc = None if ckv_scale is None else np.asarray(ckv_scale)[c if np.size(ckv_scale) > 1 else 0]
                ckv_cache[slot + (c,)] = quantise(np.float64(y[c]), ckv_dtype, sc)
            for c in range(Dk):
                sc = None if k_scale is None else np.asarray(k_scale)[c if np.size(k_scale) > 1 else 0]
                k_cache[slot + (c,)] = quantise(np.float64(r[c]), k_dtype, sc)
    return status
