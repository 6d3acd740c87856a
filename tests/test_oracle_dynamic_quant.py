"""Pins for the DynamicQuant oracle: a hand-worked row (tests/golden), the
closed forms and invariants the formula fixes, and a scalar brute force."""
import math

import numpy as np
import pytest

from oracle.dynamic_quant import ref_dynamic_quant
from helpers import ev, golden


def test_hand_worked_rows():
    g = golden("dynamic_quant_toy.json")
    for row, sc, want in zip(g["rows"], g["scales"], g["codes"]):
        codes, scale = ref_dynamic_quant(np.array([row], dtype=np.float64))
        assert list(codes[0]) == want
        assert scale[0] == np.float32(ev(sc))


def _rows(seed, n=200, h=512):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, h)) * rng.uniform(0.01, 100, (n, 1))
    return q.astype(np.float32).astype(np.float64)   # float32-exact inputs


def test_row_extreme_maps_to_127_and_signs_are_kept():
    q = _rows(1)
    codes, scale = ref_dynamic_quant(q)
    assert np.all(np.abs(codes).max(axis=1) == 127)
    assert np.all(np.sign(codes) == np.where(np.abs(q / scale[:, None].astype(np.float64)) < 0.5, 0, np.sign(q)))
    np.testing.assert_array_equal(scale, (np.abs(q).max(axis=1).astype(np.float32) / np.float32(127)))


def test_dequantised_error_is_at_most_half_a_step():
    q = _rows(2)
    codes, scale = ref_dynamic_quant(q)
    err = np.abs(codes * scale[:, None].astype(np.float64) - q)
    assert np.all(err <= scale[:, None] * (0.5 + 1e-5))


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


def test_scalar_brute_force():
    """Each code from a plain loop in float32 arithmetic (numpy scalars)."""
    q = _rows(4, n=6, h=40)
    codes, scale = ref_dynamic_quant(q)
    for r in range(q.shape[0]):
        m = np.float32(0)
        for v in q[r]:
            m = max(m, np.float32(abs(v)))
        s = np.float32(m / np.float32(127))
        assert s == scale[r]
        for j, v in enumerate(q[r]):
            x = np.float32(np.float32(v) / s)
            want = int(np.rint(x))
            assert codes[r, j] == max(-127, min(127, want))


def _planted(q, kind):
    m = np.max(np.abs(q))
    if kind == "half-away-from-zero":
        v = q / (m / 127)
        return list(np.sign(v) * np.floor(np.abs(v) + 0.5))
    if kind == "scale times 127":
        return list(np.rint(q / (m * 127)))
    if kind == "row sum instead of row max":
        return list(np.clip(np.rint(q / (np.sum(np.abs(q)) / 127)), -127, 127))
    raise ValueError(kind)


@pytest.mark.parametrize("planted", ["half-away-from-zero", "scale times 127", "row sum instead of row max"])
def test_pins_reject_planted_slips(planted):
    g = golden("dynamic_quant_toy.json")
    assert any(_planted(np.array(row, dtype=np.float64), planted) != want
               for row, want in zip(g["rows"], g["codes"]))
