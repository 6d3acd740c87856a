"""Debug validation of kv_rmsnorm_rope_cache's index (kvr_set_debug_validate,
or KVR_DEBUG_VALIDATE=1): an entry out of range, or two tokens naming the same
cache row (which the index restrictions of "aclnnKvRmsNormRopeCache" forbid),
is refused on the host with KVR_ERR_INDEX before anything is launched; valid
calls run unchanged; a call under CUDA-graph capture is not checked."""
import numpy as np
import pytest
import torch

import attention_prologue_kv_gb300 as kvr
from attention_prologue_kv_gb300 import workloads as wl
from helpers import codes_of, compare_cache, kv_to_device, run_gpu_kv, run_oracle_kv, sentinel_cache

pytestmark = pytest.mark.gpu

KVR_ERR_INDEX = 7


@pytest.fixture
def debug_on():
    kvr.set_debug_validate(True)
    try:
        yield
    finally:
        kvr.set_debug_validate(False)


def _call(case, staged=False):
    """One call on sentinel caches; returns (error code or 0, ckv codes, k codes)."""
    sh_ckv, sh_k = case.cache_shapes()
    ckv = sentinel_cache(sh_ckv, case.ckv_dtype)
    k = sentinel_cache(sh_k, case.k_dtype)
    args = (kv_to_device(case), case.gamma.cuda(), case.cos.cuda(), case.sin.cuda(), case.index.cuda(), ckv, k)
    code = 0
    try:
        if staged:
            # the staged form: the index is checked after the copy (here an
            # unrelated 16-byte copy; the bound inputs are already on the device)
            step = kvr.prepare_kv_rmsnorm_rope_cache(*args, cache_mode=case.mode, eps=case.eps)
            host = torch.zeros(16, dtype=torch.uint8).pin_memory()
            dev = torch.zeros(16, dtype=torch.uint8, device="cuda")
            step.staged(host, dev, 16)
        else:
            kvr.kv_rmsnorm_rope_cache(*args, cache_mode=case.mode, eps=case.eps)
    except kvr.KvrError as e:
        code = e.code
    torch.cuda.synchronize()
    return code, codes_of(ckv), codes_of(k)


def _untouched(case, ckv, k):
    return bool(np.all(ckv == wl.sentinel(case.ckv_dtype)) and np.all(k == wl.sentinel(case.k_dtype)))


@pytest.mark.parametrize("mode", ["Norm", "PA_BSND", "PA_BLK_BSND"])
def test_valid_calls_run_unchanged(debug_on, mode):
    case = wl.make_kv_case("dv", 3, 40, mode=mode, d0=64 if mode != "Norm" else 3, d1=16 if mode != "Norm" else 64,
                           seed=301, skip=4 if mode != "PA_BLK_BSND" else 1)
    r_ckv, r_k, r_st = run_oracle_kv(case)
    g_ckv, g_k, g_st = run_gpu_kv(case)
    assert g_st == r_st == 0
    compare_cache(g_ckv, r_ckv, case.ckv_dtype, case.Dv)
    compare_cache(g_k, r_k, case.k_dtype, case.Dk)


def test_repeated_paged_slot_is_refused(debug_on):
    case = wl.make_kv_case("dr", 2, 20, mode="PA_BSND", d0=32, d1=16, seed=302)
    case.index[7] = case.index[3]
    code, ckv, k = _call(case)
    assert code == KVR_ERR_INDEX and _untouched(case, ckv, k)
    code, ckv, k = _call(case, staged=True)
    assert code == KVR_ERR_INDEX


def test_norm_repeat_within_a_batch_refused_across_batches_allowed(debug_on):
    case = wl.make_kv_case("dn", 2, 8, mode="Norm", d0=2, d1=16, seed=303)
    case.index[1, :] = case.index[0, :]          # same slots, different cache batches: allowed
    assert _call(case)[0] == 0
    case.index[1, 5] = case.index[1, 2]          # repeated within batch 1
    code, ckv, k = _call(case)
    assert code == KVR_ERR_INDEX and _untouched(case, ckv, k)


def test_out_of_range_entry_is_refused(debug_on):
    case = wl.make_kv_case("do", 2, 10, mode="PA_BSND", d0=8, d1=16, seed=304)
    case.index[4] = 8 * 16
    assert _call(case)[0] == KVR_ERR_INDEX
    case.index[4] = -2
    assert _call(case)[0] == KVR_ERR_INDEX


def test_block_entries_repeated_or_overflowing_are_refused(debug_on):
    case = wl.make_kv_case("db", 2, 40, mode="PA_BLK_BSND", d0=32, d1=16, seed=305)
    base = case.index.clone()
    case.index[4] = case.index[1]                # two entries name one block
    assert _call(case)[0] == KVR_ERR_INDEX
    case.index.copy_(base)
    case.index[2] = case.index[2] + 9            # last block of sequence 0 holds 8 tokens: 9 + 8 > 16
    assert _call(case)[0] == KVR_ERR_INDEX
    case.index.copy_(base)
    case.index[2] = case.index[2] + 8            # 8 + 8 = 16 still fits its block
    assert _call(case)[0] == 0


def test_off_by_default_and_not_checked_under_capture():
    case = wl.make_kv_case("dc", 1, 16, mode="PA_BSND", d0=8, d1=16, seed=306)
    case.index[5] = case.index[2]
    assert _call(case)[0] == 0                   # off: the repeat only leaves an unspecified winner
    kvr.set_debug_validate(True)
    try:
        sh_ckv, sh_k = case.cache_shapes()
        ckv, k = sentinel_cache(sh_ckv, case.ckv_dtype), sentinel_cache(sh_k, case.k_dtype)
        args = (kv_to_device(case), case.gamma.cuda(), case.cos.cuda(), case.sin.cuda(), case.index.cuda(),
                ckv, k)
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            kvr.kv_rmsnorm_rope_cache(*args, cache_mode=case.mode, eps=case.eps)
        g.replay()
        torch.cuda.synchronize()
    finally:
        kvr.set_debug_validate(False)


def test_environment_variable_turns_it_on():
    """KVR_DEBUG_VALIDATE=1 in the environment: on from the first call."""
    import os
    import subprocess
    import sys
    code = (
        "import sys; sys.path[:0] = [%r, %r]\n"
        "import torch, attention_prologue_kv_gb300 as kvr\n"
        "from attention_prologue_kv_gb300 import workloads as wl\n"
        "from helpers import run_gpu_kv\n"
        "case = wl.make_kv_case('de', 1, 16, mode='PA_BSND', d0=8, d1=16, seed=307)\n"
        "case.index[5] = case.index[2]\n"
        "try:\n"
        "    run_gpu_kv(case); print('ran')\n"
        "except kvr.KvrError as e:\n"
        "    print('refused', e.code)\n") % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                           os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, KVR_DEBUG_VALIDATE="1")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
    assert out.stdout.strip().splitlines()[-1] == "refused %d" % KVR_ERR_INDEX, out.stderr[-2000:]
