"""Pins for the KV-prologue oracle: closed forms, invariants, hand-worked toys
(tests/golden), placement rules and a brute-force scalar cross-check.

Each pin is chosen so that a plausible slip in the oracle fails it: a wrong
sign in cat(-x2, x1), swapped halves or lanes, cos/sin of the wrong lane,
eps outside the sqrt, a missing gamma, the mean replaced by a sum, a wrong
slot mapping, a skipped -1 row that writes anyway."""
import numpy as np
import pytest
import torch

import oracle
from oracle import encoders as enc
from helpers import evs, golden, run_oracle_kv
from attention_prologue_kv_gb300 import workloads as wl


@pytest.mark.parametrize("name", ["kv_toy_dk2.json", "kv_toy_dk4.json"])
def test_hand_worked_toys(name):
    g = golden(name)
    kv = np.array(g["kv"], dtype=np.float64)
    Dv = g["Dv"]
    y = oracle.rms_norm(kv[:Dv], np.array(g["gamma"], dtype=np.float64), g["eps"])
    r = oracle.interleave_rope(kv[Dv:], np.array(g["cos"]), np.array(g["sin"]))
    np.testing.assert_allclose(y, evs(g["y_norm"]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r, evs(g["y_rope"]), rtol=1e-14, atol=1e-15)


def test_quant_toy_codes():
    g = golden("kv_quant_toy.json")
    kv = np.array(g["kv"], dtype=np.float64)
    Dv = g["Dv"]
    y = oracle.rms_norm(kv[:Dv], np.array(g["gamma"], dtype=np.float64), g["eps"])
    for dt, want in g["codes"].items():
        got = oracle.quantise(y, dt, np.array(g["scale"], dtype=np.float32))
        assert list(got.astype(int)) == [w if w >= 0 else w + 256 for w in want], dt


def test_quantise_rounds_the_float64_product_once():
    """An 8-bit code is one rounding of the float64 product y * scale: values
    just past a rounding midpoint by less than float32 can resolve still round
    away from the midpoint (a float32 intermediate would land on the midpoint
    and tie to even instead)."""
    eps = 2.0 ** -40
    one = np.array([1.0])
    # int8: 2.5 + eps -> 3 (via float32: 2.5 -> 2)
    assert oracle.quantise(np.array([2.5 + eps]), "int8", one)[0] == 3
    assert oracle.quantise(np.array([-2.5 - eps]), "int8", one)[0] == np.uint8(256 - 3)
    # E4M3FN: midpoint of 1.0 (0x38) and 1.125 (0x39) is 1.0625
    assert oracle.quantise(np.array([1.0625 + eps]), "fp8_e4m3fn", one)[0] == 0x39
    assert oracle.quantise(np.array([1.0625]), "fp8_e4m3fn", one)[0] == 0x38
    # E5M2: midpoint of 1.0 (0x3C) and 1.25 (0x3D) is 1.125
    assert oracle.quantise(np.array([1.125 + eps]), "fp8_e5m2", one)[0] == 0x3D
    # the product itself is not rounded first: y = 1 + 2**-30, scale = 2.5 -> 2.5 + 2.5 * 2**-30 -> 3
    assert oracle.quantise(np.array([1.0 + 2.0 ** -30]), "int8", np.array([2.5]))[0] == 3


def test_rope_identity_angle_is_deinterleave():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 64))
    r = oracle.interleave_rope(x, np.ones(64), np.zeros(64))
    assert np.array_equal(r, np.concatenate([x[:, 0::2], x[:, 1::2]], axis=-1))


def test_rope_quarter_turn():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 64))
    r = oracle.interleave_rope(x, np.zeros(64), np.ones(64))
    assert np.array_equal(r, np.concatenate([-x[:, 1::2], x[:, 0::2]], axis=-1))


def _tables(theta, width):
    h = width // 2
    ang = np.concatenate([theta[..., :h], theta[..., :h]], axis=-1)
    return np.cos(ang), np.sin(ang)


def test_rope_preserves_pair_norm():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 64))
    cos, sin = _tables(rng.uniform(-10, 10, (50, 64)), 64)
    r = oracle.interleave_rope(x, cos, sin)
    n_in = np.hypot(x[:, 0::2], x[:, 1::2])
    n_out = np.hypot(r[:, :32], r[:, 32:])
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)


def test_rope_composes_angles():
    """rotate(t1) then re-interleave then rotate(t2) equals rotate(t1 + t2)."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((20, 16))
    t1 = rng.uniform(-3, 3, (20, 16))
    t2 = rng.uniform(-3, 3, (20, 16))
    c1, s1 = _tables(t1, 16)
    c2, s2 = _tables(t2, 16)
    c12, s12 = _tables(t1 + t2, 16)
    y = oracle.interleave_rope(x, c1, s1)
    y_inter = np.empty_like(y)
    y_inter[:, 0::2] = y[:, :8]
    y_inter[:, 1::2] = y[:, 8:]
    np.testing.assert_allclose(oracle.interleave_rope(y_inter, c2, s2),
                               oracle.interleave_rope(x, c12, s12), rtol=1e-10, atol=1e-12)


def test_rope_pair_lane_mapping_by_distinct_angles():
    """Output lane i and lane i + Dk/2 come from input pair (2i, 2i+1) only:
    rotating one pair by a quarter turn moves exactly those two outputs."""
    x = np.arange(1.0, 9.0)          # 8 lanes, 4 pairs
    cos = np.ones(8)
    sin = np.zeros(8)
    cos[[2, 6]] = 0.0
    sin[[2, 6]] = 1.0
    r = oracle.interleave_rope(x, cos, sin)
    # identity on pairs 0, 1, 3; pair 2 = (x4, x5) = (5, 6) -> (-6, 5)
    assert list(r) == [1, 3, -6, 7, 2, 4, 5, 8]


def test_rmsnorm_unit_gamma_has_closed_form_rms():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((40, 512)) * rng.uniform(0.01, 10, (40, 1))
    eps = float(np.float32(1e-6))
    y = oracle.rms_norm(x, np.ones(512), eps)
    ms = (x * x).mean(-1)
    rms_y = np.sqrt((y * y).mean(-1))
    np.testing.assert_allclose(rms_y, np.sqrt(ms / (ms + eps)), rtol=1e-13)
    assert np.all(np.abs(rms_y - 1) <= eps / (2 * ms) * 1.0001 + 1e-15)


def test_rmsnorm_scale_invariant_without_eps():
    rng = np.random.default_rng(6)
    x = rng.standard_normal((10, 512))
    g = rng.uniform(0.5, 1.5, 512)
    np.testing.assert_allclose(oracle.rms_norm(37.5 * x, g, 0.0), oracle.rms_norm(x, g, 0.0), rtol=1e-13)


def test_rmsnorm_eps_inside_sqrt_and_gamma_per_channel():
    x = np.array([2.0, 0.0, 0.0, 0.0])       # mean square 1
    y = oracle.rms_norm(x, np.array([3.0, 1, 1, 1]), 3.0)
    np.testing.assert_allclose(y, [2.0 / 2.0 * 3.0, 0, 0, 0])   # sqrt(1 + 3) = 2


def test_norm_mode_placement_hand():
    """Norm: batch b writes cache batch b at row index[b, s]; -1 skips."""
    case = wl.make_kv_case("t", 2, 2, Dv=8, Dk=8, mode="Norm", d0=2, d1=3, seed=9)
    case.index[:] = torch.tensor([[2, -1], [0, 1]])
    ckv, k, st = run_oracle_kv(case)
    assert st == 0
    written = {(b, r) for b in range(2) for r in range(3) if not np.all(ckv[b, r] == wl.SENTINEL16)}
    assert written == {(0, 2), (1, 0), (1, 1)}
    assert np.all(k[0, 0] == wl.SENTINEL16) and np.all(k[0, 1] == wl.SENTINEL16)
    # the row written at (0, 2) is token (0, 0) wherever that token lands
    case2 = wl.make_kv_case("t", 2, 2, Dv=8, Dk=8, mode="Norm", d0=2, d1=3, seed=9)
    case2.index[:] = torch.tensor([[0, 1], [2, 0]])
    ckv2, _, _ = run_oracle_kv(case2)
    assert np.array_equal(ckv[0, 2], ckv2[0, 0])
    assert np.array_equal(ckv[1, 0], ckv2[1, 2])
    assert np.array_equal(ckv[1, 1], ckv2[1, 0])


def test_pa_mode_placement_hand():
    """PA_BSND: slot v -> (v // BlockSize, v % BlockSize)."""
    case = wl.make_kv_case("t", 1, 3, Dv=8, Dk=8, mode="PA_BSND", d0=4, d1=2, seed=10)
    case.index[:] = torch.tensor([5, -1, 0])
    ckv, k, st = run_oracle_kv(case)
    assert st == 0
    written = {(a, b) for a in range(4) for b in range(2) if not np.all(ckv[a, b] == wl.SENTINEL16)}
    assert written == {(2, 1), (0, 0)}
    assert {(a, b) for a in range(4) for b in range(2) if not np.all(k[a, b] == wl.SENTINEL16)} == written


def test_pa_blk_mode_placement_hand():
    """PA_BLK_BSND: one index entry per BlockSize tokens; token s goes to entry + s % BlockSize."""
    case = wl.make_kv_case("t", 2, 3, Dv=8, Dk=8, mode="PA_BLK_BSND", d0=5, d1=2, seed=11)
    # Bkv=2, Skv=3, BlockSize=2 -> 2 entries per sequence
    case.index[:] = torch.tensor([6, 0, -1, 2])
    ckv, k, st = run_oracle_kv(case)
    assert st == 0
    written = {(a, b) for a in range(5) for b in range(2) if not np.all(ckv[a, b] == wl.SENTINEL16)}
    # seq 0: s=0,1 -> slots 6,7 = (3,0),(3,1); s=2 -> slot 0 = (0,0); seq 1: s=0,1 skipped; s=2 -> slot 2 = (1,0)
    assert written == {(3, 0), (3, 1), (0, 0), (1, 0)}


@pytest.mark.parametrize("mode,bad", [("Norm", 32), ("Norm", -2), ("PA_BSND", 4096 * 128),
                                      ("PA_BSND", -7)])
def test_out_of_range_index_sets_status_and_writes_nothing(mode, bad):
    if mode == "Norm":
        case = wl.make_kv_case("t", 2, 4, Dv=16, Dk=8, mode="Norm", d0=2, d1=32, seed=12)
        case.index[1, 2] = bad
    else:
        case = wl.make_kv_case("t", 4, 1, Dv=16, Dk=8, mode="PA_BSND", d0=4096, d1=128, seed=12)
        case.index[2] = bad
    ckv, k, st = run_oracle_kv(case)
    assert st == oracle.STATUS_INDEX
    n_written = int(np.sum(~np.all(ckv.reshape(-1, 16) == wl.SENTINEL16, axis=-1)))
    assert n_written == 7 if mode == "Norm" else n_written == 3


def test_blk_entry_that_would_leave_its_block_is_rejected():
    case = wl.make_kv_case("t", 1, 2, Dv=8, Dk=8, mode="PA_BLK_BSND", d0=4, d1=2, seed=13)
    case.index[:] = torch.tensor([3])      # token 1 would land in slot 4 (next block)
    ckv, k, st = run_oracle_kv(case)
    assert st == oracle.STATUS_INDEX
    written = {(a, b) for a in range(4) for b in range(2) if not np.all(ckv[a, b] == wl.SENTINEL16)}
    assert written == {(1, 1)}


@pytest.mark.parametrize("ckv_dtype,k_dtype,mode", [
    ("bf16", "bf16", "Norm"), ("bf16", "bf16", "PA_BSND"), ("fp8_e4m3fn", "bf16", "PA_BSND"),
    ("int8", "bf16", "PA_BSND"), ("fp8_e5m2", "fp8_e4m3fn", "PA_BLK_BSND"), ("bf16", "int8", "PA_BSND"),
    ("f16", "f16", "Norm"),
])
def test_scalar_loop_matches_vectorised(ckv_dtype, k_dtype, mode):
    if mode == "Norm":
        kw = dict(mode="Norm", d0=3, d1=9)
    elif mode == "PA_BLK_BSND":
        kw = dict(mode="PA_BLK_BSND", d0=8, d1=4)
    else:
        kw = dict(mode="PA_BSND", d0=6, d1=4)
    indt = "f16" if ckv_dtype == "f16" else "bf16"
    case = wl.make_kv_case("t", 3, 7, Dv=24, Dk=16, ckv_dtype=ckv_dtype, k_dtype=k_dtype,
                           seed=14, skip=2, kc_scale=0.75, in_dtype=indt, **kw)
    a_ckv, a_k, a_st = run_oracle_kv(case)
    b_ckv, b_k, b_st = run_oracle_kv(case, loop=True)
    assert a_st == b_st == 0
    assert np.array_equal(a_ckv, b_ckv)
    assert np.array_equal(a_k, b_k)


def test_kc_scale_multiplies_normalised_part_only():
    c1 = wl.make_kv_case("t", 2, 3, Dv=16, Dk=8, mode="PA_BSND", d0=2, d1=4, seed=15)
    c2 = wl.make_kv_case("t", 2, 3, Dv=16, Dk=8, mode="PA_BSND", d0=2, d1=4, seed=15, kc_scale=2.0)
    a_ckv, a_k, _ = run_oracle_kv(c1)
    b_ckv, b_k, _ = run_oracle_kv(c2)
    assert np.array_equal(a_k, b_k)
    w = ~np.all(a_ckv == wl.SENTINEL16, axis=-1)
    # times 2 is exact in bf16: the exponent field moves up by one
    np.testing.assert_array_equal(enc.bf16_decode(b_ckv[w]), 2 * enc.bf16_decode(a_ckv[w]))


def test_untouched_slots_keep_any_prior_contents():
    case = wl.decode_paged()
    ckv = np.random.default_rng(0).integers(0, 2**16, (case.d0, case.d1, case.Dv), dtype=np.uint16)
    k = np.random.default_rng(1).integers(0, 2**16, (case.d0, case.d1, case.Dk), dtype=np.uint16)
    ckv0, k0 = ckv.copy(), k.copy()
    run_oracle_kv(case, ckv, k)
    idx = case.index.numpy()
    live = idx[idx >= 0]
    mask = np.ones(case.d0 * case.d1, bool)
    mask[live] = False
    assert np.array_equal(ckv.reshape(-1, case.Dv)[mask], ckv0.reshape(-1, case.Dv)[mask])
    assert np.array_equal(k.reshape(-1, case.Dk)[mask], k0.reshape(-1, case.Dk)[mask])
    assert not np.array_equal(ckv.reshape(-1, case.Dv)[live], ckv0.reshape(-1, case.Dv)[live])
    assert (idx == -1).sum() == 5


def _robust_case(ckv_dtype, k_dtype):
    from attention_prologue_kv_gb300 import workloads as wl
    return wl.make_kv_case("rb", 3, 40, Dv=64, Dk=16, mode="PA_BSND", d0=4, d1=64, seed=91, skip=4,
                           ckv_dtype=ckv_dtype, k_dtype=k_dtype, kv_std=3.0)


def _encode_like_gpu(case, enc_fn):
    """Caches holding enc_fn(float32 evaluation of the oracle's values), at
    the oracle's rows: a stand-in for a GPU result, built on the CPU."""
    import oracle
    from helpers import f32_arg, kv_token_rows, oracle_kv_inputs, sentinel_caches_np
    kv, gamma, cos, sin, _ = oracle_kv_inputs(case)
    f32 = lambda a: None if a is None else np.asarray(a, dtype=np.float32)
    vy, vr, _ = oracle.kv_values(f32(kv), f32(gamma), f32(cos), f32(sin), Dv=case.Dv, eps=np.float32(f32_arg(case.eps)),
                                 ckv_scale=None if case.ckv_scale is None else case.ckv_scale.numpy(),
                                 k_scale=None if case.k_scale is None else case.k_scale.numpy())
    ckv, k = sentinel_caches_np(case)
    rows, bs, ss = kv_token_rows(case)
    ckv.reshape(-1, case.Dv)[rows] = enc_fn(vy[bs, ss].astype(np.float64), case.ckv_dtype)
    k.reshape(-1, case.Dk)[rows] = enc_fn(vr[bs, ss].astype(np.float64), case.k_dtype)
    return ckv, k


@pytest.mark.parametrize("dtypes", [("bf16", "bf16"), ("fp8_e4m3fn", "int8"), ("int8", "fp8_e5m2")])
def test_robust_check_accepts_float32_and_rejects_truncation(dtypes):
    """The exactness check used by the GPU parity tests: a float32 evaluation
    of the method, rounded like the oracle, passes (and most elements are
    checked); the same values encoded by truncation toward zero fail it,
    although they stay within one ulp / one code of the oracle."""
    from oracle import encoders as enc
    from helpers import check_robust_kv
    case = _robust_case(*dtypes)
    good_ckv, good_k = _encode_like_gpu(case, enc.encode)
    assert check_robust_kv(case, good_ckv, good_k) > 0.95

    def trunc(v, dt):
        if dt == "int8":
            return enc.encode(np.trunc(v), dt)
        # step toward zero: the largest code magnitude not above |v|
        c = enc.encode(v, dt)
        back = enc.decode(c, dt)
        over = np.abs(back) > np.abs(v)
        ordn = enc.code_ordinal(c, dt)
        ordn = np.where(over, ordn - np.sign(ordn), ordn)
        mag = np.abs(ordn)
        width = 16 if dt in enc.DTYPES_16 else 8
        signbit = np.where(ordn < 0, 1 << (width - 1), 0)
        return (mag | signbit).astype(enc.code_dtype(dt))
    bad_ckv, bad_k = _encode_like_gpu(case, trunc)
    with pytest.raises(AssertionError, match="away from any rounding boundary"):
        check_robust_kv(case, bad_ckv, bad_k)


@pytest.mark.parametrize("dtypes", [("bf16", "bf16"), ("fp8_e4m3fn", "int8"), ("f16", "fp8_e5m2")])
def test_kv_values_encode_to_the_oracle_caches(dtypes):
    """kv_values (the float64 value each element encodes) agrees with the
    oracle: encoding it gives the written rows code for code, and the RoPE
    magnitude bound dominates the value."""
    from oracle import encoders as enc
    from helpers import f32_arg, kv_token_rows, oracle_kv_inputs, run_oracle_kv
    from attention_prologue_kv_gb300 import workloads as wl
    in_dtype = "f16" if dtypes[0] == "f16" else "bf16"
    case = wl.make_kv_case("kvv", 3, 30, Dv=48, Dk=24, mode="PA_BSND", d0=4, d1=32, seed=93, skip=5,
                           ckv_dtype=dtypes[0], k_dtype=dtypes[1], in_dtype=in_dtype, kc_scale=0.8)
    ref_ckv, ref_k, _ = run_oracle_kv(case)
    kv, gamma, cos, sin, _ = oracle_kv_inputs(case)
    vy, vr, mr = oracle.kv_values(kv, gamma, cos, sin, Dv=case.Dv, eps=f32_arg(case.eps),
                                  ckv_scale=None if case.ckv_scale is None else case.ckv_scale.numpy(),
                                  k_scale=None if case.k_scale is None else case.k_scale.numpy(),
                                  kc_scale=f32_arg(case.kc_scale))
    rows, bs, ss = kv_token_rows(case)
    assert len(rows) == case.active_tokens()
    assert np.array_equal(enc.encode(vy[bs, ss], case.ckv_dtype), ref_ckv.reshape(-1, case.Dv)[rows])
    assert np.array_equal(enc.encode(vr[bs, ss], case.k_dtype), ref_k.reshape(-1, case.Dk)[rows])
    assert np.all(mr >= np.abs(vr) * (1 - 1e-15))
