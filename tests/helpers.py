"""Shared test plumbing: golden-fixture loading and torch <-> oracle marshalling.
Holds no arithmetic of the method."""
import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def ev(expr):
    """Evaluate a hand-derived closed form such as '3/sqrt(12.5)'."""
    return float(eval(str(expr), {"__builtins__": {}}, {"sqrt": math.sqrt}))


def evs(exprs):
    return np.array([ev(e) for e in exprs], dtype=np.float64)


def f64(t):
    """torch tensor (bf16/f16/f32) -> float64 numpy array (exact widening)."""
    if t is None:
        return None
    return t.detach().cpu().to(torch.float64).numpy()


def codes_of(t):
    """torch cache tensor -> numpy array of its bit patterns (uint16 / uint8)."""
    t = t.detach().cpu()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.uint8).numpy()


def oracle_kv_inputs(case):
    """KVCase -> the oracle's float64 view: kv [Bkv, Skv, D], cos/sin [Bkv, Skv, Dk]."""
    D = case.Dv + case.Dk
    kv = f64(case.kv).reshape(case.Bkv, case.Skv, D)
    cos = f64(case.cos).reshape(case.Bkv, case.Skv, case.Dk)
    sin = f64(case.sin).reshape(case.Bkv, case.Skv, case.Dk)
    return kv, f64(case.gamma), cos, sin, case.index.numpy()


def sentinel_caches_np(case):
    from attention_prologue_kv_gb300.workloads import sentinel
    from oracle.encoders import code_dtype
    ckv = np.full((case.d0, case.d1, case.Dv), sentinel(case.ckv_dtype), dtype=code_dtype(case.ckv_dtype))
    k = np.full((case.d0, case.d1, case.Dk), sentinel(case.k_dtype), dtype=code_dtype(case.k_dtype))
    return ckv, k


def run_oracle_kv(case, ckv=None, k=None, loop=False):
    import oracle
    if ckv is None:
        ckv, k = sentinel_caches_np(case)
    kv, gamma, cos, sin, index = oracle_kv_inputs(case)
    fn = oracle.ref_kv_rmsnorm_rope_cache_loop if loop else oracle.ref_kv_rmsnorm_rope_cache
    st = fn(kv, gamma, cos, sin, index, ckv, k, Dv=case.Dv, mode=case.mode, eps=case.eps,
            ckv_dtype=case.ckv_dtype, k_dtype=case.k_dtype,
            ckv_scale=None if case.ckv_scale is None else case.ckv_scale.numpy(),
            k_scale=None if case.k_scale is None else case.k_scale.numpy(),
            kc_scale=case.kc_scale)
    return ckv, k, st


def oracle_qsa_inputs(case):
    return dict(raw=f64(case.raw), key_length=case.key_length.numpy(),
                rope_cos=f64(case.rope_cos), rope_sin=f64(case.rope_sin),
                k_norm_weight=f64(case.k_norm_weight), past_raw=f64(case.past_raw),
                past_rope=f64(case.past_rope), key_block_size=case.kbs, eps=case.eps)


def run_oracle_qsa(case, block_keys=None, carry=False):
    import oracle
    from attention_prologue_kv_gb300.workloads import SENTINEL16
    if block_keys is None:
        block_keys = np.full((case.N, case.Bcap, case.Di), SENTINEL16, dtype=np.uint16)
    nr = npr = None
    if carry:
        nr = np.full((case.N, case.kbs - 1, case.Di), np.nan)
        npr = np.full((case.N, 2 * case.Dr), np.nan) if case.Dr else None
    st = oracle.ref_qsa_prepare(block_keys=block_keys, next_raw=nr, next_rope=npr,
                                **oracle_qsa_inputs(case))
    return block_keys, nr, npr, st
