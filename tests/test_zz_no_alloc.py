"""The host-staged KV call that allocates nothing
(kv_rmsnorm_rope_cache_staged_static) against the host-staged call that
copies into a device buffer the caller allocated (kv_rmsnorm_rope_cache_staged)
and against the float64 oracle.

Callers that cannot allocate device memory (code running inside an
allocator's own callbacks, plugins of a framework that owns all device
memory, processes whose memory budget is spent) cannot provide that buffer;
the new entry point stages into a static device array of the library instead.
Both entry points are called here through the C ABI, twice in a row on two
different batches, and after each call the caches and the status word the
new one leaves must match the existing one's, and the oracle's, within the
parity tests' tolerance. Requests that do not fit the array are refused before anything
runs. This file is collected last, so a run that stops at the first failure
has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

from attention_prologue_kv_gb300 import _native as N
from attention_prologue_kv_gb300 import workloads as wl
from helpers import check_robust_kv, codes_of, compare_cache, run_oracle_kv, sentinel_cache

pytestmark = pytest.mark.gpu

STAGE_BYTES = 8 * 1024 * 1024   # KVR_STATIC_STAGE_BYTES of include/kvr.h


def _packed(case):
    """The case's kv, cos, sin and index back to back in pinned host memory,
    and their byte offsets (the last entry is the total)."""
    parts = [case.kv.reshape(-1).view(torch.uint8), case.cos.reshape(-1).view(torch.uint8),
             case.sin.reshape(-1).view(torch.uint8), case.index.reshape(-1).view(torch.uint8)]
    offs = [0]
    for p in parts:
        offs.append(offs[-1] + p.numel())
    return torch.cat(parts).pin_memory(), offs


def _args(case, gamma, ckv, k, status, kv=None, cos=None, sin=None, index=None):
    ptr = lambda t: None if t is None else t.data_ptr()
    return N.KvArgs(kv=ptr(kv), in_dtype=N.KVR_BF16, Bkv=case.Bkv, Skv=case.Skv, Dv=case.Dv, Dk=case.Dk,
                    kv_row_stride=0, gamma=ptr(gamma), cos=ptr(cos), sin=ptr(sin), index=ptr(index),
                    mode=1, cache_d0=case.d0, cache_d1=case.d1, ckv_cache=ptr(ckv), ckv_dtype=N.KVR_BF16,
                    ckv_scale=None, ckv_scale_len=0, k_cache=ptr(k), k_dtype=N.KVR_BF16, k_scale=None,
                    k_scale_len=0, eps=case.eps, kc_scale=1.0, dev_status=ptr(status), params_ready=0)


def test_static_staging_matches_the_staged_call_twice_in_a_row():
    lib = N.lib()
    stream = torch.cuda.current_stream().cuda_stream
    a = wl.make_kv_case("na", 256, 1, mode="PA_BSND", d0=64, d1=128, seed=801, skip=5)
    b = wl.make_kv_case("nb", 256, 1, mode="PA_BSND", d0=64, d1=128, seed=802, skip=3)
    b.index[17] = 64 * 128 + 5          # out of range: skipped, KVR_DEVERR_INDEX in the status word
    b.gamma = a.gamma                   # one set of weights for both batches
    gamma = a.gamma.cuda()
    valid = lambda c: {int(x) for x in c.index.tolist() if 0 <= x < 64 * 128}
    rows_after = [len(valid(a)), len(valid(a) | valid(b))]
    batches = [_packed(a), _packed(b)]
    offs = batches[0][1]
    nbytes = offs[4]
    assert nbytes <= STAGE_BYTES and batches[1][1] == offs

    # the existing entry point: the caller's device buffer, inputs bound into it
    stage = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    views = (stage[offs[0]:offs[1]].view(torch.bfloat16), stage[offs[1]:offs[2]].view(torch.bfloat16),
             stage[offs[2]:offs[3]].view(torch.bfloat16), stage[offs[3]:offs[4]].view(torch.int64))
    ckv_ref, k_ref = sentinel_cache((64, 128, 1, 512), "bf16"), sentinel_cache((64, 128, 1, 64), "bf16")
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
    args_ref = _args(a, gamma, ckv_ref, k_ref, st_ref, *views)
    # the new entry point: kv, cos, sin and index come from the static area
    ckv, k = sentinel_cache((64, 128, 1, 512), "bf16"), sentinel_cache((64, 128, 1, 64), "bf16")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    args_new = _args(a, gamma, ckv, k, st)
    hs_ref = torch.full((2,), -1, dtype=torch.int32).pin_memory()
    hs = torch.full((2,), -1, dtype=torch.int32).pin_memory()
    r_ckv = r_k = None                  # the oracle's caches, carried across the two calls

    for i, (host, _) in enumerate(batches):
        r = lib.kv_rmsnorm_rope_cache_staged(ctypes.byref(args_ref), host.data_ptr(), stage.data_ptr(), nbytes,
                                             hs_ref[i:].data_ptr(), stream)
        assert r == N.KVR_OK
        r = lib.kv_rmsnorm_rope_cache_staged_static(ctypes.byref(args_new), host.data_ptr(), nbytes, offs[0],
                                                    offs[1], offs[2], offs[3], hs[i:].data_ptr(), stream)
        assert r == N.KVR_OK
        torch.cuda.synchronize()
        assert int(hs[i]) == int(hs_ref[i]) == (0 if i == 0 else N.KVR_DEVERR_INDEX)
        n1, _ = compare_cache(codes_of(ckv), codes_of(ckv_ref), "bf16", 512)
        n2, _ = compare_cache(codes_of(k), codes_of(k_ref), "bf16", 64)
        assert n1 == n2 == rows_after[i]
        r_ckv, r_k, r_st = run_oracle_kv((a, b)[i], r_ckv, r_k)
        assert r_st == (0 if i == 0 else N.KVR_DEVERR_INDEX)
        n1, _ = compare_cache(codes_of(ckv), r_ckv, "bf16", 512)
        n2, _ = compare_cache(codes_of(k), r_k, "bf16", 64)
        assert n1 == n2 == rows_after[i]
        check_robust_kv((a, b)[i], codes_of(ckv), codes_of(k))   # this call's rows, exact away from ties
    assert int(st.item()) == int(st_ref.item()) == N.KVR_DEVERR_INDEX


def test_static_staging_refuses_what_does_not_fit():
    """Too many bytes, or an input outside the copied bytes: refused on the
    host, nothing enqueued, the caches untouched."""
    lib = N.lib()
    stream = torch.cuda.current_stream().cuda_stream
    a = wl.make_kv_case("nc", 4, 8, mode="PA_BSND", d0=8, d1=16, seed=803)
    host, offs = _packed(a)
    ckv, k = sentinel_cache((8, 16, 1, 512), "bf16"), sentinel_cache((8, 16, 1, 64), "bf16")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gamma = a.gamma.cuda()
    args = _args(a, gamma, ckv, k, st)
    call = lambda nbytes, o: lib.kv_rmsnorm_rope_cache_staged_static(
        ctypes.byref(args), host.data_ptr(), nbytes, o[0], o[1], o[2], o[3], None, stream)
    assert call(STAGE_BYTES + 16, offs) == N.KVR_ERR_SHAPE
    assert call(offs[4] - 8, offs) == N.KVR_ERR_SHAPE                          # index past the copied bytes
    assert call(offs[4], [offs[0], offs[1] + 1, offs[2], offs[3]]) == N.KVR_ERR_SHAPE   # misaligned cos
    torch.cuda.synchronize()
    assert np.all(codes_of(ckv) == wl.SENTINEL16) and np.all(codes_of(k) == wl.SENTINEL16)
    assert call(offs[4], offs) == N.KVR_OK
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and not np.all(codes_of(k) == wl.SENTINEL16)
