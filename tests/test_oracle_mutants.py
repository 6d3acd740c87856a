"""The pins must catch plausible slips: each mutant below plants one mistake
in a copy of an oracle step (on the CPU) and at least one pin has to reject it."""
import numpy as np
import pytest

import oracle
from helpers import evs, golden


def _rope_pins(rope):
    """True if `rope` passes the hand toys and the closed forms."""
    ok = True
    for name in ("kv_toy_dk2.json", "kv_toy_dk4.json"):
        g = golden(name)
        kv = np.array(g["kv"], dtype=np.float64)
        r = rope(kv[g["Dv"]:], np.array(g["cos"]), np.array(g["sin"]))
        ok &= np.allclose(r, evs(g["y_rope"]), rtol=1e-14, atol=1e-15)
    x = np.random.default_rng(1).standard_normal((3, 16))
    ok &= np.array_equal(rope(x, np.ones(16), np.zeros(16)), np.concatenate([x[:, 0::2], x[:, 1::2]], -1))
    ok &= np.array_equal(rope(x, np.zeros(16), np.ones(16)), np.concatenate([-x[:, 1::2], x[:, 0::2]], -1))
    return bool(ok)


def _norm_pins(norm):
    ok = True
    for name in ("kv_toy_dk2.json", "kv_toy_dk4.json"):
        g = golden(name)
        kv = np.array(g["kv"], dtype=np.float64)
        y = norm(kv[:g["Dv"]], np.array(g["gamma"], dtype=np.float64), g["eps"])
        ok &= np.allclose(y, evs(g["y_norm"]), rtol=1e-14, atol=1e-15)
    x = np.array([2.0, 0.0, 0.0, 0.0])
    ok &= np.allclose(norm(x, np.array([3.0, 1, 1, 1]), 3.0), [3.0, 0, 0, 0])
    return bool(ok)


def _cat(a, b):
    return np.concatenate((a, b), axis=-1)


ROPE_MUTANTS = {
    "sign on the wrong half": lambda x, c, s: _cat(x[..., 0::2], x[..., 1::2]) * c + _cat(x[..., 1::2], -x[..., 0::2]) * s,
    "halves swapped": lambda x, c, s: _cat(x[..., 1::2], x[..., 0::2]) * c + _cat(x[..., 0::2], -x[..., 1::2]) * s,
    "rotate-half instead of interleave": lambda x, c, s: x * c + _cat(-x[..., x.shape[-1] // 2:], x[..., :x.shape[-1] // 2]) * s,
    "cos/sin swapped": lambda x, c, s: _cat(x[..., 0::2], x[..., 1::2]) * s + _cat(-x[..., 1::2], x[..., 0::2]) * c,
    "cos of the neighbouring lane": lambda x, c, s: oracle.interleave_rope(x, np.roll(c, 1, -1), s),
}

NORM_MUTANTS = {
    "eps outside the sqrt": lambda x, g, e: x / (np.sqrt((x * x).mean(-1, keepdims=True)) + e) * g,
    "sum instead of mean": lambda x, g, e: x / np.sqrt((x * x).sum(-1, keepdims=True) + e) * g,
    "gamma dropped": lambda x, g, e: x / np.sqrt((x * x).mean(-1, keepdims=True) + e),
    "mean of |x| instead of x^2": lambda x, g, e: x / np.sqrt(np.abs(x).mean(-1, keepdims=True) + e) * g,
}


def _half_rope_pins(rope):
    """True if `rope` (rotate-half form) passes the complex-rotation closed form
    with a distinct angle per pair, and the identity and quarter-turn cases."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 16))
    th = rng.uniform(-np.pi, np.pi, (3, 8))
    c = np.concatenate((np.cos(th), np.cos(th)), -1)
    s = np.concatenate((np.sin(th), np.sin(th)), -1)
    y = rope(x, c, s)
    ok = np.allclose(y[:, :8] + 1j * y[:, 8:], (x[:, :8] + 1j * x[:, 8:]) * np.exp(1j * th), rtol=1e-13, atol=1e-14)
    ok &= np.array_equal(rope(x, np.ones(16), np.zeros(16)), x)
    ok &= np.array_equal(rope(x, np.zeros(16), np.ones(16)), np.concatenate([-x[:, 8:], x[:, :8]], -1))
    return bool(ok)


HALF_ROPE_MUTANTS = {
    "interleave instead of rotate-half": oracle.interleave_rope,
    "sign on the wrong half": lambda x, c, s: x * c + _cat(x[..., x.shape[-1] // 2:], -x[..., :x.shape[-1] // 2]) * s,
    "cos of the neighbouring lane": lambda x, c, s: oracle.rotate_half_rope(x, np.roll(c, 1, -1), s),
    "halves not swapped in the sin term": lambda x, c, s: x * c + x * s,
}


def test_true_oracle_passes_the_pins():
    assert _rope_pins(oracle.interleave_rope)
    assert _half_rope_pins(oracle.rotate_half_rope)
    assert _norm_pins(oracle.rms_norm)


@pytest.mark.parametrize("name", sorted(HALF_ROPE_MUTANTS))
def test_half_rope_mutant_is_caught(name):
    assert not _half_rope_pins(HALF_ROPE_MUTANTS[name])


@pytest.mark.parametrize("name", sorted(ROPE_MUTANTS))
def test_rope_mutant_is_caught(name):
    assert not _rope_pins(ROPE_MUTANTS[name])


@pytest.mark.parametrize("name", sorted(NORM_MUTANTS))
def test_norm_mutant_is_caught(name):
    assert not _norm_pins(NORM_MUTANTS[name])
