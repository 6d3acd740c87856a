"""Seeded random configurations of every entry point against the oracle:
shapes, cache modes, code types, scales, strides, skip counts, RoPE layouts,
the concat form, carry outputs and params_ready drawn from a fixed seed per
case, so that combinations the targeted tests do not list are covered too.
Same acceptance as the targeted tests: untouched bytes and copies
bit-exact, 16-bit results within 2**-7*|ref| + 1e-6, 8-bit codes within one
code, DynamicQuant scales equal and codes within one code of the exact
quotient's (equal away from ties, everywhere in exact mode), status bits
equal."""
import numpy as np
import pytest
import torch

from attention_prologue_kv_gb300 import workloads as wl
from helpers import (check_robust_kv, check_robust_qsa, compare_cache, compare_dynamic_quant, run_gpu_kv,
                     run_gpu_qsa, run_oracle_kv, run_oracle_qsa)

pytestmark = pytest.mark.gpu

CODES8 = ["int8", "fp8_e4m3fn", "fp8_e5m2"]


def kv_config(i):
    r = np.random.default_rng(5000 + i)
    in_dtype = str(r.choice(["bf16", "f16"]))
    Dv = int(r.choice([1, 7, 8, 20, 24, 64, 128, 256, 512, 520, 1024, 1032]))
    Dk = int(r.choice([2, 4, 6, 8, 16, 64, 72, 128, 256, 258]))
    Bkv, Skv = int(r.integers(1, 7)), int(r.integers(1, 60))
    mode = str(r.choice(["Norm", "PA_BSND", "PA_BLK_BSND"]))
    d1 = int(r.integers(1, 70))
    if mode == "Norm":
        d1 = max(d1, Skv)
        d0 = Bkv + int(r.integers(0, 3))
    elif mode == "PA_BSND":
        d0 = -(-Bkv * Skv // d1) + int(r.integers(0, 4))
    else:
        d0 = Bkv * -(-Skv // d1) + int(r.integers(0, 4))
    ckv = str(r.choice([in_dtype] + CODES8))
    k = str(r.choice([in_dtype] + CODES8))
    return dict(Bkv=Bkv, Skv=Skv, Dv=Dv, Dk=Dk, mode=mode, d0=d0, d1=d1, ckv_dtype=ckv, k_dtype=k,
                in_dtype=in_dtype, seed=6000 + i, kv_std=float(r.choice([0.5, 1.0, 3.0])),
                skip=int(r.integers(0, 1 + Bkv * Skv // 4)) if mode != "PA_BLK_BSND" else 0,
                scale_len=1 if r.random() < 0.3 else None, k_scale_len=1 if r.random() < 0.3 else None,
                kc_scale=float(r.choice([1.0, 0.7, 1.9])), row_pad=int(r.choice([0, 0, 8, 3]))), \
        bool(r.random() < 0.5)


@pytest.mark.parametrize("i", range(40))
def test_kv_random_configurations(i):
    cfg, params_ready = kv_config(i)
    case = wl.make_kv_case("fuzz", **cfg)
    ref_ckv, ref_k, ref_st = run_oracle_kv(case)
    g_ckv, g_k, g_st = run_gpu_kv(case, params_ready=params_ready)
    assert g_st == ref_st, cfg
    n1, _ = compare_cache(g_ckv, ref_ckv, case.ckv_dtype, case.Dv)
    n2, _ = compare_cache(g_k, ref_k, case.k_dtype, case.Dk)
    assert n1 == n2 == case.active_tokens(), cfg
    if n1:
        check_robust_kv(case, g_ckv, g_k)


def qsa_config(i):
    r = np.random.default_rng(7000 + i)
    Di = int(r.choice([8, 16, 24, 32, 64, 128, 256]))
    rope = bool(r.random() < 0.8)
    Dr = int(r.choice([d for d in (2, 4, 6, 8, 16, 32, 64) if d <= Di])) if rope else 0
    kbs = int(r.choice([2, 3, 5, 8, 16, 33, 64]))
    N, L = int(r.integers(1, 7)), int(r.integers(0, 150))
    return dict(N=N, L=L, Di=Di, Dr=Dr, kbs=kbs, seed=8000 + i, past_max=int(r.integers(1, 400)),
                rope=rope, norm=bool(r.random() < 0.8), shared_length=bool(r.random() < 0.2),
                in_dtype=str(r.choice(["bf16", "f16"]))), \
        dict(carry=bool(r.random() < 0.7),
             rope_layout=str(r.choice(["interleave_last", "interleave_first", "half_last", "half_first"])),
             concat=bool(r.random() < 0.4), bp_extra=int(r.integers(-2, 3)),
             params_ready=bool(r.random() < 0.5))


@pytest.mark.parametrize("i", range(30))
def test_qsa_random_configurations(i):
    cfg, opt = qsa_config(i)
    case = wl.make_qsa_case("fuzz", **cfg)
    past_bk = None
    if opt["concat"]:
        K = case.key_length.expand(case.N) if case.key_length.numel() == 1 else case.key_length
        j0max = int(((K - case.L) // case.kbs).max())
        Bp = max(0, j0max + opt["bp_extra"])
        past_bk = np.random.default_rng(i).integers(0, 0x7C00, (case.N, Bp, case.Di), dtype=np.uint16)
    kw = dict(carry=opt["carry"], rope_layout=opt["rope_layout"], past_block_keys=past_bk)
    values = {}
    r_bk, r_nr, r_npr, r_st = run_oracle_qsa(case, values_out=values, **kw)
    g_bk, g_nr, g_npr, g_st = run_gpu_qsa(case, params_ready=opt["params_ready"], **kw)
    assert g_st == r_st, (cfg, opt)
    compare_cache(g_bk, r_bk, "bf16" if cfg["in_dtype"] == "bf16" else "f16", case.Di)
    check_robust_qsa(g_bk, values, "bf16" if cfg["in_dtype"] == "bf16" else "f16")
    if opt["carry"]:
        assert np.array_equal(g_nr, r_nr, equal_nan=True)
        if case.Dr:
            assert np.array_equal(g_npr, r_npr, equal_nan=True)


@pytest.mark.parametrize("i", range(16))
def test_dynamic_quant_random_configurations(i):
    import attention_prologue_kv_gb300 as kvr
    r = np.random.default_rng(9000 + i)
    H = int(r.choice([1, 3, 8, 24, 100, 256, 512, 1000, 1024, 1032, 2048]))
    q = wl.dynamic_quant_decode(seed=9100 + i, T=int(r.integers(1, 20)), heads=int(r.integers(1, 9)), Hckv=H,
                                dtype=str(r.choice(["bf16", "f16"])))
    q = q * float(r.choice([1e-3, 1.0, 50.0]))
    out = torch.full(q.shape, 99, dtype=torch.int8, device="cuda")
    scale = torch.full(q.shape[:-1] + (1,), -1.0, dtype=torch.float32, device="cuda")
    exact = bool(i % 2)
    kvr.dynamic_quant(q.cuda(), out, scale, exact=exact)
    torch.cuda.synchronize()
    compare_dynamic_quant(out.cpu().numpy(), scale.cpu().numpy(), q.reshape(-1, H).to(torch.float64).numpy(),
                          exact)


@pytest.mark.parametrize("i", range(20))
def test_kv_random_configurations_compiled_split(i):
    """The same draws with the row split the kernels compile as constants
    (Dv = 512, Dk = 64): modes, code types, scales, strides, skips, f16 and
    params_ready still vary."""
    cfg, params_ready = kv_config(100 + i)
    cfg.update(Dv=512, Dk=64)
    case = wl.make_kv_case("fuzz", **cfg)
    ref_ckv, ref_k, ref_st = run_oracle_kv(case)
    g_ckv, g_k, g_st = run_gpu_kv(case, params_ready=params_ready)
    assert g_st == ref_st, cfg
    n1, _ = compare_cache(g_ckv, ref_ckv, case.ckv_dtype, case.Dv)
    n2, _ = compare_cache(g_k, ref_k, case.k_dtype, case.Dk)
    assert n1 == n2 == case.active_tokens(), cfg
    if n1:
        check_robust_kv(case, g_ckv, g_k)


@pytest.mark.parametrize("i", range(20))
def test_qsa_random_configurations_compiled_shapes(i):
    """QSA draws with (Di, kbs) from the compiled set."""
    cfg, opt = qsa_config(100 + i)
    r = np.random.default_rng(7500 + i)
    cfg.update(Di=int(r.choice([64, 128, 256])), kbs=int(r.choice([32, 64, 128])), L=int(r.integers(0, 400)))
    cfg["Dr"] = min(cfg["Dr"], cfg["Di"]) if cfg["rope"] else 0
    case = wl.make_qsa_case("fuzz", **cfg)
    past_bk = None
    if opt["concat"]:
        K = case.key_length.expand(case.N) if case.key_length.numel() == 1 else case.key_length
        Bp = max(0, int(((K - case.L) // case.kbs).max()) + opt["bp_extra"])
        past_bk = np.random.default_rng(i).integers(0, 0x7C00, (case.N, Bp, case.Di), dtype=np.uint16)
    kw = dict(carry=opt["carry"], rope_layout=opt["rope_layout"], past_block_keys=past_bk)
    values = {}
    r_bk, r_nr, r_npr, r_st = run_oracle_qsa(case, values_out=values, **kw)
    g_bk, g_nr, g_npr, g_st = run_gpu_qsa(case, params_ready=opt["params_ready"], **kw)
    assert g_st == r_st, (cfg, opt)
    compare_cache(g_bk, r_bk, "bf16" if cfg["in_dtype"] == "bf16" else "f16", case.Di)
    check_robust_qsa(g_bk, values, "bf16" if cfg["in_dtype"] == "bf16" else "f16")
    if opt["carry"]:
        assert np.array_equal(g_nr, r_nr, equal_nan=True)
        if case.Dr:
            assert np.array_equal(g_npr, r_npr, equal_nan=True)
