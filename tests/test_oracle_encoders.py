"""Pins for the oracle's encoders: library routines (torch CPU casts, numpy)
on exhaustive/edge grids, and hand-worked code points."""
import numpy as np
import pytest
import torch

from oracle import encoders as enc


def _f32_grid(rng, n=200000):
    """float32 values across every exponent, plus exact halfway points of
    the bf16 grid (ties) and their float32 neighbours."""
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    v = bits.view(np.float32)
    v = v[np.isfinite(v)]
    # bf16 ties: a bf16 value plus half a bf16 ulp, i.e. low 16 bits = 0x8000
    tb = (rng.integers(0, 2**16, size=20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    t = tb.view(np.float32)
    t = t[np.isfinite(t)]
    nb = np.concatenate([np.nextafter(t, np.float32(np.inf)), np.nextafter(t, np.float32(-np.inf))])
    sub = (rng.integers(1, 2**23, size=5000, dtype=np.uint64).astype(np.uint32)).view(np.float32)
    edge = np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38, 3.4028235e38, 1.1754944e-38,
                     9.183549e-41, 1e-45], dtype=np.float32)
    return np.concatenate([v, t, nb, sub, -sub, edge]).astype(np.float32)


def test_bf16_matches_torch_cast_on_float32_inputs():
    rng = np.random.default_rng(7)
    v = _f32_grid(rng)
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = enc.bf16_encode(v.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (v[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_bf16_single_rounding_from_float64():
    # 1 + 2**-8 + 2**-30 lies just above the bf16 tie between 1 and 1 + 2**-7:
    # one rounding from float64 goes up; rounding via float32 first would tie to even (down).
    v = 1.0 + 2.0**-8 + 2.0**-30
    assert enc.bf16_encode(v) == 0x3F81
    assert enc.bf16_encode(1.0 + 2.0**-8) == 0x3F80          # exact tie -> even
    assert enc.bf16_encode(1.0 + 3 * 2.0**-8) == 0x3F82      # exact tie -> even (up)
    assert enc.bf16_encode(-2.0) == 0xC000
    assert enc.bf16_encode(2.0**-133) == 0x0001               # smallest subnormal
    assert enc.bf16_encode(2.0**-134) == 0x0000               # tie with 0 -> even (0)
    assert enc.bf16_encode(3 * 2.0**-134) == 0x0002           # tie 1.5 -> 2
    assert enc.bf16_encode(2.0**128) == 0x7F80                # overflow -> inf


def test_bf16_decode_roundtrip():
    codes = np.arange(2**16, dtype=np.uint32).astype(np.uint16)
    vals = enc.bf16_decode(codes)
    fin = np.isfinite(vals)
    back = enc.bf16_encode(vals[fin])
    # +0/-0 keep their sign bit; every finite code maps back to itself
    assert np.array_equal(back, codes[fin])


def test_f16_matches_torch_cast():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(100000) * np.exp2(rng.integers(-26, 17, 100000))).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(enc.f16_encode(v.astype(np.float64)), want)


def _fp8_midpoint_grid(decode, maxfinite):
    codes = np.arange(256, dtype=np.uint8)
    vals = decode(codes)
    vals = np.unique(vals[np.isfinite(vals)])
    mids = (vals[:-1] + vals[1:]) / 2
    eps32 = np.abs(mids) * 2.0**-20 + 2.0**-40
    pts = np.concatenate([vals, mids, mids + eps32, mids - eps32,
                          [maxfinite * 1.01, -maxfinite * 1.5, 1e6, -1e6]])
    return pts.astype(np.float32)


@pytest.mark.parametrize("name,tdt,maxfinite", [
    ("fp8_e4m3fn", torch.float8_e4m3fn, 448.0),
    ("fp8_e5m2", torch.float8_e5m2, 57344.0),
])
def test_fp8_matches_torch_cast_after_clamp(name, tdt, maxfinite):
    decode = getattr(enc, name + "_decode")
    encode = getattr(enc, name + "_encode")
    pts = _fp8_midpoint_grid(decode, maxfinite)
    clamped = np.clip(pts, -maxfinite, maxfinite)
    want = torch.from_numpy(clamped).to(tdt).view(torch.uint8).numpy()
    got = encode(pts.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (pts[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_e4m3fn_hand_points():
    e = enc.fp8_e4m3fn_encode
    assert e(1.0) == 0x38
    assert e(448.0) == 0x7E
    assert e(464.0) == 0x7E          # past the largest finite value: saturates
    assert e(1e9) == 0x7E
    assert e(-1e9) == 0xFE
    assert e(2.0**-9) == 0x01        # smallest subnormal
    assert e(2.0**-10) == 0x00       # tie with zero -> even
    assert e(2.0**-6) == 0x08        # smallest normal
    assert e(0.875) == 0x36
    assert e(1.0625) == 0x38         # tie between 1.0 (even) and 1.125
    assert e(1.1875) == 0x3A         # tie between 1.125 and 1.25 (even)
    assert enc.fp8_e4m3fn_decode(0x7E) == 448.0


def test_e5m2_hand_points():
    e = enc.fp8_e5m2_encode
    assert e(1.0) == 0x3C
    assert e(57344.0) == 0x7B
    assert e(1e9) == 0x7B            # saturates instead of overflowing to inf
    assert e(2.0**-16) == 0x01
    assert e(2.0**-14) == 0x04


def test_int8_hand_points():
    q = lambda v: enc.int8_decode(enc.int8_encode(v))
    assert q(2.5) == 2 and q(3.5) == 4 and q(-2.5) == -2 and q(-3.5) == -4
    assert q(200.0) == 127 and q(-200.0) == -128 and q(127.5) == 127
    assert q(0.49) == 0 and q(-0.51) == -1


def test_code_ordinal_is_monotone_in_value():
    for name in ("fp8_e4m3fn", "fp8_e5m2", "int8"):
        codes = np.arange(256, dtype=np.uint8)
        vals = enc.decode(codes, name)
        fin = np.isfinite(vals)
        order = np.argsort(vals[fin], kind="stable")
        ords = enc.code_ordinal(codes[fin], name)[order]
        assert np.all(np.diff(ords) >= 0)
    codes = np.arange(2**16, dtype=np.uint32).astype(np.uint16)
    vals = enc.bf16_decode(codes)
    fin = np.isfinite(vals)
    order = np.argsort(vals[fin], kind="stable")
    assert np.all(np.diff(enc.code_ordinal(codes[fin], "bf16")[order]) >= 0)
