"""Pins for the QSA block-key oracle: hand-worked toys (tests/golden), the
no-norm/no-rope case against numpy's mean, chunking, constant keys, and the
rule that unused carry rows are never read."""
import numpy as np
import pytest
import torch

import oracle
from oracle import encoders as enc
from helpers import evs, golden, oracle_qsa_inputs, run_oracle_qsa
from attention_prologue_kv_gb300 import workloads as wl


def _golden_call(g, carry=False):
    raw = np.array(g["raw"], dtype=np.float64)
    N, L, Di = raw.shape
    kbs = g["kbs"]
    Dr = len(g["rope_cos"][0][0])
    bk = np.full((N, g["Bcap"], Di), wl.SENTINEL16, dtype=np.uint16)
    past_raw = np.array(g.get("past_raw", np.full((N, kbs - 1, Di), np.nan)), dtype=np.float64)
    past_rope = np.array(g.get("past_rope", np.full((N, 2 * Dr), np.nan)), dtype=np.float64)
    nr = np.full((N, kbs - 1, Di), np.nan) if carry else None
    npr = np.full((N, 2 * Dr), np.nan) if carry else None
    st = oracle.ref_qsa_prepare(raw, bk, np.array(g["key_length"]), np.array(g["rope_cos"], dtype=np.float64),
                                np.array(g["rope_sin"], dtype=np.float64),
                                np.array(g["k_norm_weight"], dtype=np.float64), past_raw, past_rope,
                                kbs, g["eps"], next_raw=nr, next_rope=npr)
    return bk, nr, npr, st


@pytest.mark.parametrize("name", ["qsa_two_block.json", "qsa_carry.json"])
def test_hand_worked_toys(name):
    g = golden(name)
    bk, nr, npr, st = _golden_call(g, carry=True)
    assert st == 0
    for j, exprs in g["expected_blocks"].items():
        want = evs(exprs)
        assert np.array_equal(bk[0, int(j)], enc.bf16_encode(want)), (j, enc.bf16_decode(bk[0, int(j)]), want)
    for j in g["untouched_blocks"]:
        assert np.all(bk[0, j] == wl.SENTINEL16)
    if "expected_next_raw" in g:
        rows = np.array(g["expected_next_raw"], dtype=object)
        n_rows = rows.shape[1]
        np.testing.assert_array_equal(nr[:, :n_rows], np.vectorize(float)(rows))
        np.testing.assert_allclose(npr, np.vectorize(float)(np.array(g["expected_next_rope"], dtype=object)))


def test_no_norm_no_rope_is_plain_block_mean():
    case = wl.make_qsa_case("t", 3, 48, Di=24, kbs=8, seed=1, past=[0, 0, 0], rope=False, norm=False)
    bk, _, _, st = run_oracle_qsa(case)
    assert st == 0
    raw = case.raw.to(torch.float64).numpy()
    want = raw.reshape(3, 6, 8, 24).mean(axis=2)
    assert np.array_equal(bk[:, :6], enc.bf16_encode(want))


def test_constant_keys_mean_is_the_key_and_unit_weight_gives_unit_rms():
    N, L, Di, kbs = 2, 16, 32, 4
    raw = np.tile(np.random.default_rng(0).standard_normal((N, 1, Di)), (1, L, 1))
    bk = np.full((N, 8, Di), wl.SENTINEL16, dtype=np.uint16)
    oracle.ref_qsa_prepare(raw, bk, np.array([L, L]), None, None, None,
                           np.full((N, kbs - 1, Di), np.nan), None, kbs)
    for j in range(4):
        assert np.array_equal(bk[:, j], enc.bf16_encode(raw[:, 0]))
    eps = float(np.float32(1e-6))
    bk2 = np.full((N, 8, Di), wl.SENTINEL16, dtype=np.uint16)
    # capture the float64 result through a float64 "encoder": decode is exact for the bf16 output,
    # so test the closed form on the float64 normalised vector directly
    m = raw[:, 0]
    u = oracle.rms_norm(m, np.ones(Di), eps)
    ms = (m * m).mean(-1)
    np.testing.assert_allclose(np.sqrt((u * u).mean(-1)), np.sqrt(ms / (ms + eps)), rtol=1e-13)
    oracle.ref_qsa_prepare(raw, bk2, np.array([L]), None, None, np.ones(Di),
                           np.full((N, kbs - 1, Di), np.nan), None, kbs)
    assert np.array_equal(bk2[:, 0], enc.bf16_encode(u))


def test_chunked_calls_equal_one_call():
    """One call over L tokens equals three chained calls over pieces of L,
    each feeding the next through the carry outputs."""
    N, L, Di, Dr, kbs = 4, 45, 16, 8, 6
    case = wl.make_qsa_case("t", N, L, Di=Di, Dr=Dr, kbs=kbs, seed=3, past=[0, 5, 13, 6], Bcap=12)
    whole, _, _, st = run_oracle_qsa(case)
    assert st == 0
    inp = oracle_qsa_inputs(case)
    P = np.array(case.meta["past"])
    pieces = [0, 7, 30, L]
    bk = np.full_like(whole, wl.SENTINEL16)
    past_raw, past_rope = inp["past_raw"], inp["past_rope"]
    for a, b in zip(pieces[:-1], pieces[1:]):
        nr = np.full((N, kbs - 1, Di), np.nan)
        npr = np.full((N, 2 * Dr), np.nan)
        st = oracle.ref_qsa_prepare(inp["raw"][:, a:b], bk, P + b, inp["rope_cos"][:, a:b],
                                    inp["rope_sin"][:, a:b], inp["k_norm_weight"], past_raw,
                                    past_rope, kbs, case.eps, next_raw=nr, next_rope=npr)
        assert st == 0
        # an unspecified carry rope (no incomplete block) stays NaN: it must never be read
        past_raw, past_rope = nr, npr
    assert np.array_equal(bk, whole)


def test_unused_carry_rows_are_never_read():
    case = wl.qsa_prepare_workload()
    bk, _, _, st = run_oracle_qsa(case)
    assert st == 0
    vals = enc.bf16_decode(bk[bk != wl.SENTINEL16])
    assert np.all(np.isfinite(vals))
    # 32 completed blocks per sequence (L = 2048 = 32 * 64)
    written = (bk != wl.SENTINEL16).all(-1)
    assert written.sum() == 32 * 32
    P = np.array(case.meta["past"])
    for n in range(case.N):
        assert np.array_equal(np.nonzero(written[n])[0], np.arange(P[n] // 64, P[n] // 64 + 32))


def test_shared_key_length_broadcasts():
    case = wl.make_qsa_case("t", 3, 20, Di=16, Dr=8, kbs=4, seed=5, shared_length=True)
    bk1, _, _, st = run_oracle_qsa(case)
    case.key_length = case.key_length.expand(3).clone()
    bk2, _, _, _ = run_oracle_qsa(case)
    assert st == 0 and np.array_equal(bk1, bk2)


def test_short_key_length_and_block_cap_raise_status():
    case = wl.make_qsa_case("t", 2, 16, Di=16, Dr=8, kbs=4, seed=6, past=[0, 3])
    case.key_length = torch.tensor([10, 19])   # sequence 0: key_length < L
    bk, _, _, st = run_oracle_qsa(case)
    assert st == oracle.STATUS_KEY_LENGTH
    assert np.all(bk[0] == wl.SENTINEL16)
    case = wl.make_qsa_case("t", 1, 16, Di=16, Dr=8, kbs=4, seed=6, past=[0], Bcap=2)
    bk, _, _, st = run_oracle_qsa(case)
    assert st == oracle.STATUS_BLOCK_CAP
    assert (bk[0] != wl.SENTINEL16).all(-1).sum() == 2


def test_rope_uses_first_token_of_block_on_last_dr_channels():
    """Rotating the tables of a block's non-first tokens changes nothing;
    rotating the first token's changes only the last Dr channels."""
    case = wl.make_qsa_case("t", 2, 32, Di=16, Dr=8, kbs=4, seed=8, past=[0, 2])
    bk, _, _, _ = run_oracle_qsa(case)
    c2 = wl.make_qsa_case("t", 2, 32, Di=16, Dr=8, kbs=4, seed=8, past=[0, 2])
    P = np.array([0, 2])
    for n in range(2):
        for t in range(32):
            if (P[n] + t) % 4 != 0:
                c2.rope_cos[n, t] = 7.0
                c2.rope_sin[n, t] = -3.0
    bk2, _, _, _ = run_oracle_qsa(c2)
    assert np.array_equal(bk, bk2)
    c3 = wl.make_qsa_case("t", 2, 32, Di=16, Dr=8, kbs=4, seed=8, past=[0, 2])
    c3.rope_cos[0, 4] = 0.0
    c3.rope_sin[0, 4] = 1.0
    bk3, _, _, _ = run_oracle_qsa(c3)
    assert np.array_equal(bk3[0, 1, :8], bk[0, 1, :8])
    assert not np.array_equal(bk3[0, 1, 8:], bk[0, 1, 8:])


# ---- RoPE layouts (which Dr channels rotate, and how pairs are formed) ----

def _no_rope(case):
    import dataclasses
    return dataclasses.replace(case, rope_cos=None, rope_sin=None, past_rope=None, Dr=0)


@pytest.mark.parametrize("layout", oracle.ROPE_LAYOUTS)
def test_rope_layout_rotates_only_its_channels(layout):
    """Against the same call with the rotation disabled: the Dr channels the
    layout names change, the others are bit-identical."""
    case = wl.make_qsa_case("t", 3, 40, Di=24, Dr=8, kbs=4, seed=21, past=[0, 3, 9])
    bk, _, _, st = run_oracle_qsa(case, rope_layout=layout)
    plain, _, _, _ = run_oracle_qsa(_no_rope(case))
    assert st == 0
    rot = slice(0, 8) if layout.endswith("first") else slice(16, 24)
    keep = slice(8, 24) if layout.endswith("first") else slice(0, 16)
    written = ~np.all(plain == wl.SENTINEL16, axis=-1)
    assert written.sum() == case.completed_blocks()
    assert np.array_equal(bk[..., keep], plain[..., keep])
    assert not np.array_equal(bk[written][:, rot], plain[written][:, rot])


@pytest.mark.parametrize("layout", oracle.ROPE_LAYOUTS)
def test_rope_layout_identity_and_quarter_turn(layout):
    """cos = 1, sin = 0 on every table: the rotate-half layouts leave the key
    unchanged, the interleaved ones de-interleave the rotated channels.
    cos = 0, sin = 1: pair (a, b) becomes (-b, a) in both, pairs taken by
    each layout's own rule."""
    case = wl.make_qsa_case("t", 2, 24, Di=16, Dr=8, kbs=4, seed=22, past=[0, 2], norm=False)
    plain, _, _, _ = run_oracle_qsa(_no_rope(case))
    v = enc.bf16_decode(plain)
    rot = slice(0, 8) if layout.endswith("first") else slice(8, 16)
    x = v[..., rot]
    if layout.startswith("half"):
        x1, x2 = x[..., :4], x[..., 4:]
    else:
        x1, x2 = x[..., 0::2], x[..., 1::2]
    for cv, sv, want in ((1.0, 0.0, np.concatenate((x1, x2), -1)), (0.0, 1.0, np.concatenate((-x2, x1), -1))):
        for t in (case.rope_cos, case.rope_sin, case.past_rope):
            t.fill_(0)
        case.rope_cos.fill_(cv)
        case.rope_sin.fill_(sv)
        case.past_rope[:, :8] = cv
        case.past_rope[:, 8:] = sv
        bk, _, _, _ = run_oracle_qsa(case, rope_layout=layout)
        got = enc.bf16_decode(bk)
        written = ~np.all(plain == wl.SENTINEL16, axis=-1)
        np.testing.assert_array_equal(got[written][:, rot], want[written])


def test_rotate_half_is_interleave_of_the_paired_lanes():
    """The two pairings differ only by which lanes form a pair: rotate-half on
    x equals the interleaved RoPE on x with its halves interleaved."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal((5, 12))
    c, s = rng.standard_normal((2, 5, 12))
    xi = np.empty_like(x)
    xi[:, 0::2], xi[:, 1::2] = x[:, :6], x[:, 6:]
    np.testing.assert_allclose(oracle.rotate_half_rope(x, c, s), oracle.interleave_rope(xi, c, s),
                               rtol=0, atol=0)


# ---- concat-output form (past_block_index_keys as a separate input) ----

def _past_codes(case, Bp, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, 0x7F00, (case.N, Bp, case.Di), dtype=np.uint16)


def test_concat_form_is_past_prefix_then_new_blocks():
    """Fresh output: rows j < floor(P/kbs) are the past keys bit for bit, the
    new blocks equal the in-place call's, rows of the past buffer at or
    beyond floor(P/kbs) are not copied, and everything else stays untouched."""
    case = wl.make_qsa_case("t", 3, 30, Di=16, Dr=8, kbs=4, seed=24, past=[0, 9, 17], Bcap=14)
    past = _past_codes(case, 6, 1)
    bk, _, _, st = run_oracle_qsa(case, past_block_keys=past)
    inplace, _, _, _ = run_oracle_qsa(case)
    assert st == 0
    for n, P in enumerate(case.meta["past"]):
        j0 = P // case.kbs
        assert np.array_equal(bk[n, :j0], past[n, :j0])
        assert np.array_equal(bk[n, j0:], inplace[n, j0:])


def test_concat_form_short_past_buffer_raises_status():
    case = wl.make_qsa_case("t", 2, 12, Di=16, Dr=8, kbs=4, seed=25, past=[4, 20], Bcap=10)
    past = _past_codes(case, 3, 2)       # sequence 1 has floor(20/4) = 5 past blocks
    bk, _, _, st = run_oracle_qsa(case, past_block_keys=past)
    assert st == oracle.STATUS_PAST_BLOCKS
    assert np.array_equal(bk[1, :3], past[1])
    assert np.all(bk[1, 3:5] == wl.SENTINEL16)
    assert np.array_equal(bk[0, :1], past[0, :1]) and np.all(bk[0, 1] != wl.SENTINEL16)


def test_concat_form_past_beyond_capacity_raises_block_cap():
    case = wl.make_qsa_case("t", 1, 4, Di=16, Dr=8, kbs=4, seed=26, past=[16], Bcap=3)
    past = _past_codes(case, 4, 3)
    bk, _, _, st = run_oracle_qsa(case, past_block_keys=past)
    assert st == oracle.STATUS_BLOCK_CAP
    assert np.array_equal(bk[0], past[0, :3])


@pytest.mark.parametrize("layout", ["interleave_last", "half_first"])
def test_robust_check_accepts_float32_and_rejects_truncation(layout):
    """The block-key exactness check used by the GPU parity tests: the same
    steps evaluated in float32 and rounded like the oracle pass (with most
    elements checked); truncating the float64 keys toward zero fails,
    although it stays within one ulp."""
    from attention_prologue_kv_gb300 import workloads as wl
    from helpers import check_robust_qsa, oracle_qsa_inputs
    from oracle import encoders as enc
    case = wl.make_qsa_case("rb", 3, 300, Di=64, Dr=32, kbs=32, seed=77, past_max=200)
    values = {}
    bk64 = np.full((case.N, case.Bcap, case.Di), 0x7FBF, dtype=np.uint16)
    oracle.ref_qsa_prepare(block_keys=bk64, values_out=values, rope_layout=layout, **oracle_qsa_inputs(case))
    assert len(values) > 10
    inp = {k: (v.astype(np.float32) if isinstance(v, np.ndarray) and v.dtype == np.float64 else v)
           for k, v in oracle_qsa_inputs(case).items()}
    bk32 = np.full_like(bk64, 0x7FBF)
    oracle.ref_qsa_prepare(block_keys=bk32, rope_layout=layout, **inp)
    assert check_robust_qsa(bk32, values, "bf16") > 0.85
    bad = bk64.copy()
    for (n, j), (u, _) in values.items():
        c = enc.bf16_encode(u)
        over = np.abs(enc.bf16_decode(c)) > np.abs(u)
        bad[n, j] = np.where(over, c - 1, c)          # one step toward zero in magnitude
    with pytest.raises(AssertionError, match="away from any rounding boundary"):
        check_robust_qsa(bad, values, "bf16")


def test_values_out_matches_the_written_keys():
    """values_out records, for each key written, the float64 value that
    encodes to it and a magnitude bound that dominates it."""
    from attention_prologue_kv_gb300 import workloads as wl
    from helpers import oracle_qsa_inputs
    from oracle import encoders as enc
    case = wl.make_qsa_case("vo", 2, 200, Di=32, Dr=16, kbs=16, seed=78, past_max=100)
    values = {}
    bk = np.full((case.N, case.Bcap, case.Di), 0x7FBF, dtype=np.uint16)
    oracle.ref_qsa_prepare(block_keys=bk, values_out=values, **oracle_qsa_inputs(case))
    written = {(n, j) for n in range(case.N) for j in range(case.Bcap) if not np.all(bk[n, j] == 0x7FBF)}
    assert set(values) == written and written
    for (n, j), (u, b) in values.items():
        assert np.array_equal(enc.bf16_encode(u), bk[n, j])
        assert np.all(b >= np.abs(u) * (1 - 1e-12))
