"""The C ABI without a GPU: libkvr.so builds, loads, exports every function
include/kvr.h declares, its structure layouts match the ctypes binding
(checked against offsetof() from a C compiler), and host-side validation
returns its status before any CUDA call."""
import ctypes
import os
import re
import shutil
import subprocess

import pytest

from attention_prologue_kv_gb300 import _native as N
from attention_prologue_kv_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvr.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return N.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\([^;]*\)\s*;", text, flags=re.M))


def test_header_declares_the_entry_points():
    assert _declared_functions() == set(N.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert lib.kvr_abi_version() == N.ABI_VERSION == 10


def test_status_strings(lib):
    for code in range(8):
        assert N.status_string(code) != "unknown status"
    assert N.status_string(99) == "unknown status"


PROBE = r"""
#include <stdio.h>
#include <stddef.h>
#include "kvr.h"
#define F(T, m) printf("%s.%s %zu\n", #T, #m, offsetof(T, m));
int main(void) {
    printf("kvr_kv_args %zu\n", sizeof(kvr_kv_args));
    printf("kvr_qsa_args %zu\n", sizeof(kvr_qsa_args));
    printf("kvr_dq_args %zu\n", sizeof(kvr_dq_args));
    %FIELDS%
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="no C compiler")
def test_struct_layout_matches_c(tmp_path):
    fields = []
    for T, cls in (("kvr_kv_args", N.KvArgs), ("kvr_qsa_args", N.QsaArgs), ("kvr_dq_args", N.DqArgs)):
        for name, _ in cls._fields_:
            fields.append("F(%s, %s)" % (T, name))
    src = tmp_path / "probe.c"
    src.write_text(PROBE.replace("%FIELDS%", "\n    ".join(fields)))
    exe = tmp_path / "probe"
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = dict(line.split() for line in out if line.strip())
    assert int(got["kvr_kv_args"]) == ctypes.sizeof(N.KvArgs)
    assert int(got["kvr_qsa_args"]) == ctypes.sizeof(N.QsaArgs)
    assert int(got["kvr_dq_args"]) == ctypes.sizeof(N.DqArgs)
    for T, cls in (("kvr_kv_args", N.KvArgs), ("kvr_qsa_args", N.QsaArgs), ("kvr_dq_args", N.DqArgs)):
        for name, _ in cls._fields_:
            assert int(got["%s.%s" % (T, name)]) == getattr(cls, name).offset, (T, name)


def _kv_args(**kw):
    fake = 1 << 20   # host-side validation never dereferences pointers
    a = dict(kv=fake, in_dtype=N.KVR_BF16, Bkv=2, Skv=3, Dv=512, Dk=64, kv_row_stride=0,
             gamma=fake * 2, cos=fake * 3, sin=fake * 4, index=fake * 5, mode=1, cache_d0=8,
             cache_d1=16, ckv_cache=fake * 64, ckv_dtype=N.KVR_BF16, ckv_scale=None,
             ckv_scale_len=0, k_cache=fake * 128, k_dtype=N.KVR_BF16, k_scale=None,
             k_scale_len=0, eps=1e-6, kc_scale=1.0, dev_status=None)
    a.update(kw)
    return N.KvArgs(**a)


@pytest.mark.parametrize("kw,want", [
    (dict(Dk=63), N.KVR_ERR_SHAPE),
    (dict(Dk=0), N.KVR_ERR_SHAPE),
    (dict(Dv=0), N.KVR_ERR_SHAPE),
    (dict(Bkv=-1), N.KVR_ERR_SHAPE),
    (dict(cache_d1=0), N.KVR_ERR_SHAPE),
    (dict(kv_row_stride=100), N.KVR_ERR_SHAPE),
    (dict(mode=7), N.KVR_ERR_MODE),
    (dict(in_dtype=N.KVR_INT8), N.KVR_ERR_DTYPE),
    (dict(ckv_dtype=N.KVR_F16), N.KVR_ERR_DTYPE),
    (dict(kv=None), N.KVR_ERR_NULL),
    (dict(index=None), N.KVR_ERR_NULL),
    (dict(k_cache=None), N.KVR_ERR_NULL),
    (dict(ckv_dtype=N.KVR_FP8_E4M3FN), N.KVR_ERR_NULL),                    # 8-bit cache without scale
    (dict(ckv_scale=1 << 30, ckv_scale_len=512), N.KVR_ERR_NULL),            # 16-bit cache with scale
    (dict(ckv_dtype=N.KVR_INT8, ckv_scale=1 << 30, ckv_scale_len=7), N.KVR_ERR_SHAPE),
    (dict(mode=0, cache_d0=1), N.KVR_ERR_SHAPE),                              # Norm: Bcache < Bkv
    (dict(eps=-1.0), N.KVR_ERR_SHAPE),
    (dict(kc_scale=float("nan")), N.KVR_ERR_SHAPE),
    (dict(index=(1 << 20) * 5 + 4), N.KVR_ERR_SHAPE),                         # misaligned int64
    (dict(ckv_cache=(1 << 20) + 64), N.KVR_ERR_ALIAS),                        # cache over kv
    (dict(k_cache=(1 << 20) * 64 + 1024), N.KVR_ERR_ALIAS),                   # caches overlap
    (dict(Bkv=1 << 31, Skv=1 << 31), N.KVR_ERR_SHAPE),                        # kv offsets would overflow
    (dict(cache_d0=1 << 40, cache_d1=1 << 20), N.KVR_ERR_SHAPE),              # cache offsets would overflow
])
def test_kv_host_validation(lib, kw, want):
    a = _kv_args(**kw)
    assert lib.kv_rmsnorm_rope_cache(ctypes.byref(a), None) == want


@pytest.mark.parametrize("kw,call,want", [
    (dict(), dict(bytes=-1), N.KVR_ERR_SHAPE),
    (dict(), dict(host_src=None), N.KVR_ERR_NULL),
    (dict(), dict(dev_dst=None), N.KVR_ERR_NULL),
    (dict(), dict(host_status=1 << 40), N.KVR_ERR_NULL),          # status copy without dev_status
    (dict(Dk=63), dict(), N.KVR_ERR_SHAPE),                        # the call's own validation first
    (dict(ckv_cache=(1 << 20) + 64), dict(), N.KVR_ERR_ALIAS),
    (dict(Bkv=0, kv=None), dict(bytes=0, host_src=None, dev_dst=None), N.KVR_OK),   # nothing to enqueue
])
def test_kv_staged_host_validation(lib, kw, call, want):
    """The host-staged entry point validates everything before it enqueues a copy."""
    a = _kv_args(**kw)
    c = dict(host_src=1 << 41, dev_dst=1 << 20, bytes=4096, host_status=None)
    c.update(call)
    assert lib.kv_rmsnorm_rope_cache_staged(ctypes.byref(a), c["host_src"], c["dev_dst"], c["bytes"],
                                            c["host_status"], None) == want


def test_debug_validation_switch_keeps_host_validation_first(lib):
    """With the debug index check on, host validation still decides first
    (no index copy is attempted for an invalid call), and an empty problem is
    still OK without touching the device; the switch can be turned off again."""
    lib.kvr_set_debug_validate(1)
    try:
        assert lib.kv_rmsnorm_rope_cache(ctypes.byref(_kv_args(kv=None)), None) == N.KVR_ERR_NULL
        assert lib.kv_rmsnorm_rope_cache(ctypes.byref(_kv_args(Dk=63)), None) == N.KVR_ERR_SHAPE
        assert lib.kv_rmsnorm_rope_cache(ctypes.byref(_kv_args(Bkv=0, kv=None, index=None)), None) == N.KVR_OK
    finally:
        lib.kvr_set_debug_validate(0)


def test_kv_empty_problem_is_ok_without_launch(lib):
    a = _kv_args(Bkv=0, kv=None, index=None)
    assert lib.kv_rmsnorm_rope_cache(ctypes.byref(a), None) == N.KVR_OK
    a = _kv_args(Skv=0)
    assert lib.kv_rmsnorm_rope_cache(ctypes.byref(a), None) == N.KVR_OK
    assert lib.kv_rmsnorm_rope_cache(None, None) == N.KVR_ERR_NULL


def _qsa_args(**kw):
    fake = 1 << 20
    a = dict(raw_index_keys=fake, in_dtype=N.KVR_BF16, N=4, L=64, Di=128, block_keys=fake * 8,
             Bcap=16, key_length=fake * 16, key_length_len=4, rope_cos=fake * 24,
             rope_sin=fake * 32, Dr=64, k_norm_weight=fake * 40, past_incomplete_raw_keys=fake * 48,
             past_incomplete_rope=fake * 56, key_block_size=16, eps=1e-6,
             next_incomplete_raw_keys=None, next_incomplete_rope=None, dev_status=None)
    a.update(kw)
    return N.QsaArgs(**a)


@pytest.mark.parametrize("kw,want", [
    (dict(key_block_size=1), N.KVR_ERR_SHAPE),
    (dict(Di=0), N.KVR_ERR_SHAPE),
    (dict(Di=8192), N.KVR_ERR_SHAPE),
    (dict(Dr=63), N.KVR_ERR_SHAPE),
    (dict(Dr=256), N.KVR_ERR_SHAPE),
    (dict(key_length_len=3), N.KVR_ERR_SHAPE),
    (dict(Bcap=0), N.KVR_ERR_SHAPE),
    (dict(in_dtype=N.KVR_FP8_E4M3FN), N.KVR_ERR_DTYPE),
    (dict(raw_index_keys=None), N.KVR_ERR_NULL),
    (dict(past_incomplete_raw_keys=None), N.KVR_ERR_NULL),
    (dict(rope_sin=None), N.KVR_ERR_NULL),                    # half a rope pair
    (dict(past_incomplete_rope=None), N.KVR_ERR_NULL),        # rope without its carry
    (dict(rope_cos=None, rope_sin=None), N.KVR_ERR_NULL),     # carry rope without rope
    (dict(next_incomplete_raw_keys=(1 << 20) * 48), N.KVR_ERR_ALIAS),
    (dict(next_incomplete_rope=(1 << 20) * 56 + 2), N.KVR_ERR_ALIAS),
    (dict(block_keys=(1 << 20) + 64), N.KVR_ERR_ALIAS),
    (dict(rope_layout=4), N.KVR_ERR_MODE),
    (dict(rope_layout=-1), N.KVR_ERR_MODE),
    (dict(Bp=-1), N.KVR_ERR_SHAPE),
    (dict(N=1 << 31, L=1 << 30), N.KVR_ERR_SHAPE),                 # key offsets would overflow
    (dict(Bcap=1 << 60), N.KVR_ERR_SHAPE),
    (dict(past_block_index_keys=(1 << 20) * 8 + 256, Bp=4), N.KVR_ERR_ALIAS),     # overlaps block_keys
    (dict(past_block_index_keys=(1 << 20) * 64, Bp=4,
          next_incomplete_raw_keys=(1 << 20) * 64 + 32), N.KVR_ERR_ALIAS),       # carry out over it
    (dict(past_block_index_keys=(1 << 20) * 64 + 1, Bp=4), N.KVR_ERR_SHAPE),     # misaligned
])
def test_qsa_host_validation(lib, kw, want):
    a = _qsa_args(**kw)
    assert lib.qsa_prepare(ctypes.byref(a), None) == want


def test_qsa_empty_problem_is_ok(lib):
    """No new tokens and nothing else to write: OK without a launch (the
    token tables may then be NULL). With carry outputs or a separate past
    buffer an L = 0 call still has work, so it is not returned early."""
    assert lib.qsa_prepare(ctypes.byref(_qsa_args(L=0)), None) == N.KVR_OK
    assert lib.qsa_prepare(ctypes.byref(_qsa_args(L=0, raw_index_keys=None, rope_cos=None,
                                                  rope_sin=None)), None) == N.KVR_OK
    assert lib.qsa_prepare(ctypes.byref(_qsa_args(N=0, key_length_len=0)), None) in (N.KVR_OK, N.KVR_ERR_SHAPE)


@pytest.mark.parametrize("kw,want", [
    (dict(in_dtype=N.KVR_INT8), N.KVR_ERR_DTYPE),
    (dict(Hckv=0), N.KVR_ERR_SHAPE),
    (dict(rows=-1), N.KVR_ERR_SHAPE),
    (dict(rows=1 << 60), N.KVR_ERR_SHAPE),                        # row offsets would overflow
    (dict(q_row_stride=100), N.KVR_ERR_SHAPE),
    (dict(q_nope=None), N.KVR_ERR_NULL),
    (dict(dequant_scale=None), N.KVR_ERR_NULL),
    (dict(q_out=(1 << 20) + 512), N.KVR_ERR_ALIAS),
    (dict(dequant_scale=(1 << 20) * 4 + 1000), N.KVR_ERR_ALIAS),
    (dict(rows=0, q_nope=None), N.KVR_OK),
])
def test_dynamic_quant_host_validation(lib, kw, want):
    a = dict(q_nope=1 << 20, in_dtype=N.KVR_BF16, rows=64, Hckv=512, q_row_stride=0,
             q_out=(1 << 20) * 4, dequant_scale=(1 << 20) * 8)
    a.update(kw)
    assert lib.dynamic_quant(ctypes.byref(N.DqArgs(**a)), None) == want


def test_device_copy_validation(lib):
    assert lib.kvr_device_copy(None, None, 0, None) == N.KVR_OK
    assert lib.kvr_device_copy(None, 16, 16, None) == N.KVR_ERR_NULL
    assert lib.kvr_device_copy(32, 64, 15, None) == N.KVR_ERR_SHAPE
    assert lib.kvr_device_copy(32, 48, 32, None) == N.KVR_ERR_ALIAS


def test_python_binding_rejects_cpu_tensors():
    import torch
    import attention_prologue_kv_gb300 as kvr
    x = torch.zeros(2, 1, 3, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        kvr.kv_rmsnorm_rope_cache(x, x[0, 0, 0, :512], x, x, torch.zeros(6, dtype=torch.int64),
                                  x, x)


def test_store_after_delay_validation(lib):
    d, s = 1 << 20, 1 << 21
    assert lib.kvr_store_after_delay(None, s, 4, 1000, None) == N.KVR_ERR_NULL
    assert lib.kvr_store_after_delay(d, None, 4, 1000, None) == N.KVR_ERR_NULL
    assert lib.kvr_store_after_delay(d + 4, s, 4, 1000, None) == N.KVR_ERR_SHAPE       # not 8-byte aligned
    assert lib.kvr_store_after_delay(d, s, -1, 1000, None) == N.KVR_ERR_SHAPE
    assert lib.kvr_store_after_delay(d, s, (1 << 20) + 1, 1000, None) == N.KVR_ERR_SHAPE
    assert lib.kvr_store_after_delay(d, s, 4, -1, None) == N.KVR_ERR_SHAPE
    assert lib.kvr_store_after_delay(d, s, 4, 10**8 + 1, None) == N.KVR_ERR_SHAPE      # above 0.1 s
    assert lib.kvr_store_after_delay(d, d + 8, 4, 1000, None) == N.KVR_ERR_ALIAS       # overlapping
    assert lib.kvr_store_after_delay(None, None, 0, 1000, None) == N.KVR_OK             # nothing to copy


def test_bounded_wait_check_validation(lib):
    assert lib.kvr_check_bounded_wait(None, 100000, 0, None) == N.KVR_ERR_NULL
    assert lib.kvr_check_bounded_wait(1 << 20, 10, 0, None) == N.KVR_ERR_SHAPE            # limit below 1 us
    assert lib.kvr_check_bounded_wait(1 << 20, 2 * 10**9, 0, None) == N.KVR_ERR_SHAPE      # above 1 s
    assert lib.kvr_check_bounded_wait(1 << 20, 100000, 200000, None) == N.KVR_ERR_SHAPE    # abort after the limit


def test_static_staging_host_validation(lib):
    """The no-allocation staged call refuses, before any device work, a
    request larger than its static area (8 MiB) or inputs outside the copied
    bytes; an empty problem is OK and copies nothing."""
    big = 8 * 1024 * 1024
    call = lambda a, nbytes, offs: lib.kv_rmsnorm_rope_cache_staged_static(
        ctypes.byref(a), 1 << 41, nbytes, offs[0], offs[1], offs[2], offs[3], None, None)
    a = _kv_args(kv=None, cos=None, sin=None, index=None)          # the four inputs come from the area
    T = 2 * 3
    offs = [0, T * 576 * 2, T * 576 * 2 + T * 128, T * 576 * 2 + T * 256]
    total = offs[3] + T * 8
    assert call(a, big + 16, offs) == N.KVR_ERR_SHAPE
    assert call(a, -1, offs) == N.KVR_ERR_SHAPE
    assert call(a, total - 8, offs) == N.KVR_ERR_SHAPE                        # index past the copied bytes
    assert call(a, total, [0, offs[1] + 1, offs[2], offs[3]]) == N.KVR_ERR_SHAPE   # misaligned cos
    # misaligned index: 8 more bytes copied, so that the index still lies inside them
    # and the 8-byte alignment rule alone refuses the call
    assert call(a, total + 8, [0, offs[1], offs[2], offs[3] + 4]) == N.KVR_ERR_SHAPE
    assert call(_kv_args(Bkv=0, kv=None, cos=None, sin=None, index=None), total, offs) == N.KVR_OK
