"""Pins for the DynamicQuant oracle: hand-worked rows (tests/golden), the
closed forms and invariants the formula fixes, and a brute force in exact
rational arithmetic (fractions.Fraction), which shares nothing with the
oracle's float64 evaluation."""
from fractions import Fraction

import numpy as np
import pytest

from oracle.dynamic_quant import dynamic_quant_quotients, ref_dynamic_quant
from helpers import ev, golden


def test_hand_worked_rows():
    g = golden("dynamic_quant_toy.json")
    for row, sc, want in zip(g["rows"], g["scales"], g["codes"]):
        codes, scale = ref_dynamic_quant(np.array([row], dtype=np.float64))
        assert list(codes[0]) == want
        assert scale[0] == np.float32(ev(sc))


def _rows(seed, n=200, h=512, bits=8):
    """Rows of values with `bits` significant bits (8: bfloat16, 11: float16)."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, h)) * rng.uniform(0.01, 100, (n, 1))
    m, e = np.frexp(q)
    return np.ldexp(np.rint(m * 2.0 ** bits) / 2.0 ** bits, e)


def test_row_extreme_maps_to_127_and_signs_are_kept():
    q = _rows(1)
    codes, scale = ref_dynamic_quant(q)
    assert np.all(np.abs(codes).max(axis=1) == 127)
    v, _ = dynamic_quant_quotients(q)
    assert np.all(np.sign(codes) == np.where(np.abs(v) <= 0.5, 0, np.sign(q)))
    # the scale is the float32 division of two float32 values (IEEE: correctly rounded)
    np.testing.assert_array_equal(scale, (np.abs(q).max(axis=1).astype(np.float32) / np.float32(127)))


def test_dequantised_error_is_at_most_half_a_step():
    q = _rows(2)
    codes, _ = ref_dynamic_quant(q)
    step = np.abs(q).max(axis=1, keepdims=True) / 127
    err = np.abs(codes * step - q)
    assert np.all(err <= step * (0.5 + 1e-12))


def test_odd_symmetry_and_power_of_two_scaling():
    q = _rows(3)
    c1, s1 = ref_dynamic_quant(q)
    c2, s2 = ref_dynamic_quant(-q)
    np.testing.assert_array_equal(c2, -c1)
    np.testing.assert_array_equal(s2, s1)
    c3, s3 = ref_dynamic_quant(q * 8.0)
    np.testing.assert_array_equal(c3, c1)
    np.testing.assert_array_equal(s3, s1 * np.float32(8))


def test_zero_row():
    codes, scale = ref_dynamic_quant(np.zeros((2, 16)))
    assert np.all(codes == 0) and np.all(scale == 0)


def _round_half_even(fr):
    f = fr.numerator // fr.denominator          # floor
    rem = fr - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f


def _nearest_f32(fr):
    """The float32 nearest to the rational fr > 0, ties to an even significand."""
    c = np.float32(float(fr))
    cands = [np.nextafter(c, np.float32(0)), c, np.nextafter(c, np.float32(np.inf))]
    best = min(abs(Fraction(float(x)) - fr) for x in cands)
    near = [x for x in cands if abs(Fraction(float(x)) - fr) == best]
    if len(near) == 1:
        return near[0]
    return [x for x in near if int(x.view(np.uint32)) % 2 == 0][0]


@pytest.mark.parametrize("bits", [8, 11])
def test_exact_rational_brute_force(bits):
    """Each code is round-half-even of the exact rational q * 127 / RowMax and
    each scale the float32 nearest to RowMax / 127, computed with Fractions."""
    q = _rows(4 + bits, n=6, h=40, bits=bits)
    # plant exact ties: an element whose quotient is k + 1/2 (RowMax = 127 * 2**-3)
    q[0, 0] = 127 * 2.0 ** -3
    q[0, 1:6] = np.array([0.5, 2.5, -3.5, 64.5, -100.5]) * 2.0 ** -3
    q[0, 6:] = np.clip(q[0, 6:], -1, 1) * 2.0 ** -4
    codes, scale = ref_dynamic_quant(q)
    for r in range(q.shape[0]):
        m = max(Fraction(abs(float(x))) for x in q[r])
        assert scale[r] == _nearest_f32(m / 127)
        for j, x in enumerate(q[r]):
            want = max(-127, min(127, _round_half_even(Fraction(float(x)) * 127 / m)))
            assert int(codes[r, j]) == want, (r, j, float(x))
    assert list(codes[0, 1:6]) == [0, 2, -4, 64, -100]


def test_exact_half_integers_survive_the_float64_division():
    """Quotients that are exact half-integers come out of the float64
    division exactly (they are representable and the division is correctly
    rounded), so ties are decided on the true value."""
    rng = np.random.default_rng(7)
    k = rng.integers(-127, 127, 4000)
    e = rng.integers(-30, 30, 4000)
    rows = np.stack([127.0 * np.ldexp(1.0, e), (k + 0.5) * np.ldexp(1.0, e)], axis=1)   # RowMax first
    v, _ = dynamic_quant_quotients(rows)
    np.testing.assert_array_equal(v[:, 1], k + 0.5)
    codes, _ = ref_dynamic_quant(rows)
    np.testing.assert_array_equal(codes[:, 1], np.where(k % 2 == 0, k, k + 1))


def _planted(q, kind):
    m = np.max(np.abs(q))
    if kind == "half-away-from-zero":
        v = q / (m / 127)
        return list(np.sign(v) * np.floor(np.abs(v) + 0.5))
    if kind == "scale times 127":
        return list(np.rint(q / (m * 127)))
    if kind == "row sum instead of row max":
        return list(np.clip(np.rint(q / (np.sum(np.abs(q)) / 127)), -127, 127))
    if kind == "scale rounded to float32 before the division":
        s = np.float64(np.float32(m / 127))
        return list(np.clip(np.rint(q / s), -127, 127))
    raise ValueError(kind)


@pytest.mark.parametrize("planted", ["half-away-from-zero", "scale times 127", "row sum instead of row max"])
def test_pins_reject_planted_slips(planted):
    g = golden("dynamic_quant_toy.json")
    assert any(_planted(np.array(row, dtype=np.float64), planted) != want
               for row, want in zip(g["rows"], g["codes"]))


def test_pins_reject_a_float32_scale_in_the_quotient():
    """Dividing by the float32-rounded scale is a plausible slip: on bfloat16
    rows the exact quotient is often a half-integer, which the slip moves off
    the tie, so the codes differ somewhere (checked against the rational
    brute force above on the same kind of rows)."""
    q = _rows(12, n=2000, h=512)
    codes, _ = ref_dynamic_quant(q)
    bad = np.array([_planted(row, "scale rounded to float32 before the division") for row in q])
    assert not np.array_equal(codes, bad.astype(np.int8))
