"""Failure detection without a GPU fault: a kernel's wait for copies that
never land gives up at its time limit (or when its abort flag is raised),
reports KVR_DEVERR_TIMEOUT through the status word the host reads, and the
context stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import attention_prologue_kv_gb300 as kvr
from attention_prologue_kv_gb300 import workloads as wl
from helpers import compare_cache, run_gpu_kv, run_oracle_kv

pytestmark = pytest.mark.gpu


def test_wait_gives_up_at_its_time_limit_and_the_context_stays_usable():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvr.check_bounded_wait(st, limit_us=20000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == 0x8
    assert 0.015 < dt < 2.0
    case = wl.make_kv_case("after", 2, 16, mode="PA_BSND", d0=4, d1=16, seed=70)
    ref_ckv, ref_k, ref_st = run_oracle_kv(case)
    g_ckv, g_k, g_st = run_gpu_kv(case)
    assert g_st == ref_st == 0
    compare_cache(g_ckv, ref_ckv, "bf16", case.Dv)


def test_abort_flag_ends_the_wait_early():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    kvr.check_bounded_wait(st, limit_us=900000, abort_after_us=2000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(st.item()) == 0x8
    assert dt < 0.5   # far below the 0.9 s limit


def test_status_bits_accumulate_with_the_other_bits():
    st = torch.full((1,), 0x2, dtype=torch.int32, device="cuda")
    kvr.check_bounded_wait(st, limit_us=1000)
    torch.cuda.synchronize()
    assert int(st.item()) == 0x2 | 0x8
